// BF16 sink/recent decode, q rotation and the online-softmax merge.
//
// Method (OSCAR author write-up, m.th-motor.com, serving paragraph): the BF16 kernel covers the
// sink and recent tokens with the raw query, the INT2 kernel the rotated history, and an
// online-softmax merge combines the two. Values of INT2 tokens live in the rotated basis;
// unless the value rotation is absorbed into the projection weights ("oscar-2bit-kv-cache",
// arddev.tech, section "Аналитика"), the merged INT2 output is brought back by R_V^T.
#include "device_common.cuh"

namespace oscar {
namespace {

constexpr int kBfWarps = kBf16WarpsPerPage;
constexpr int kBfSlotsPerPair = kBf16SlotsPerPair;

// Token slot `tau` of BF16 page `pg` (0 = sink page, 1..4 = recent ring pages) holds a live
// token of a sequence with length L and demote frontier F.
__device__ __forceinline__ bool bf16_slot_live(int pg, int tau, int L, int F) {
  if (pg == 0) return tau < min(kSink, L);
  const int slot = (pg - 1) * kPage + tau;
  const int base = L - kRecent;
  const int pos = base + ((slot - base) % kRecent + kRecent) % kRecent;
  return pos >= F && pos < L && pos >= 0;
}

// One CTA per (sequence, KV head): the live pages among the sink page and the 4 recent-ring
// pages stream through two shared-memory stages (K and V page of 16 KB each, 1-D bulk copies,
// bounded waits); warp w takes tokens 16w .. 16w+15 of every page with an online softmax across
// the pages, and the CTA combines its 4 warps into one partial for the pair.
constexpr int kBfStages = 2;
constexpr int kBfPageBytes = kPage * kHeadDim * 2;
constexpr int kBfSmem = kBfStages * 2 * kBfPageBytes + kBfStages * 8;

template <int HG>
__global__ void __launch_bounds__(kBfWarps * 32)
    k_decode_bf16(DevPool P, StepDims S, int layer, const __nv_bfloat16* __restrict__ q,
                  float* __restrict__ part) {
  constexpr int NT = HG / 4;
  constexpr int SLOT = HG * (2 + kHeadDim);
  static_assert(kBfWarps * HG * kHeadDim * 4 <= kBfStages * 2 * kBfPageBytes, "reduction buffer");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBfStages * 2 * kBfPageBytes);
  __shared__ float red_m[kBfWarps][HG], red_l[kBfWarps][HG];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int pair = blockIdx.x;
  const int bi = pair / P.Hkv, h = pair - bi * P.Hkv;
  const StepSeq st = P.step[bi];
  const int L = st.L_new, F = st.F_new;
  float* slot = part + (size_t)pair * SLOT;

  // live pages (CTA-uniform): bit pg set when page pg holds a live token
  uint32_t live = 0;
#pragma unroll
  for (int pg = 0; pg < kBf16PagesPerPair; ++pg)
    if (__syncthreads_or(bf16_slot_live(pg, threadIdx.x & (kPage - 1), L, F))) live |= 1u << pg;
  if ((live & 1u) && (st.sink_page < 0 || st.sink_page >= P.max_sink_pages)) {
    if (threadIdx.x == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
    live &= ~1u;
  }
  const int n_live = __popc(live);
  if (n_live == 0) {  // an empty segment
    for (int k = threadIdx.x; k < SLOT; k += blockDim.x) slot[k] = (k < 2 * HG && (k & 1) == 0) ? -INFINITY : 0.f;
    return;
  }
  auto nth_page = [&](int i) {  // page index of the i-th live page
    uint32_t m = live;
    for (int k = 0; k < i; ++k) m &= m - 1;
    return __ffs(m) - 1;
  };
  auto issue = [&](int i, int stg) {  // thread 0: bulk copies of live page i into stage stg
    const int pg = nth_page(i);
    const __nv_bfloat16 *srcK, *srcV;
    if (pg == 0) {
      const size_t off = (size_t)layer * P.sink_layer_stride + ((size_t)st.sink_page * P.Hkv + h) * kPage * kHeadDim;
      srcK = P.sink_k + off;
      srcV = P.sink_v + off;
    } else {
      const size_t off = (size_t)layer * P.ring_layer_stride +
                         (((size_t)st.seq_id * P.Hkv + h) * kRecent + (pg - 1) * kPage) * kHeadDim;
      srcK = P.ring_k + off;
      srcV = P.ring_v + off;
    }
    uint8_t* dst = smem + stg * 2 * kBfPageBytes;
    mbar_expect_tx(&bar[stg], 2 * kBfPageBytes);
    const uint64_t pol = policy_evict_first();
    bulk_g2s(dst, srcK, kBfPageBytes, &bar[stg], pol);
    bulk_g2s(dst + kBfPageBytes, srcV, kBfPageBytes, &bar[stg], pol);
  };
  if (threadIdx.x == 0) {
    for (int k = 0; k < kBfStages; ++k) mbar_init(&bar[k], 1);
    fence_mbar_init();
    for (int k = 0; k < kBfStages && k < n_live; ++k) issue(k, k);
  }
  __syncthreads();

  // query fragments: column 2h' holds head h' of the n-tile, column 2h'+1 is zero
  uint32_t qf[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(
        q + ((size_t)bi * P.Hq + (size_t)h * HG + nt * 4 + (g >> 1)) * kHeadDim);
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
      qf[nt][k8][0] = (g & 1) ? 0u : qh[(16 * k8 + 2 * tq) >> 1];
      qf[nt][k8][1] = (g & 1) ? 0u : qh[(16 * k8 + 2 * tq + 8) >> 1];
    }
  }
  float acc[NT][8][4], mrow[NT], lrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mrow[nt] = -INFINITY;
    lrow[nt] = 0.f;
#pragma unroll
    for (int m8 = 0; m8 < 8; ++m8)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][m8][e] = 0.f;
  }
  const int t0 = warp * 16, mi = lane >> 3, r = lane & 7;
  int stg = 0;
  uint32_t par = 0;
  int i = 0;
  for (; i < n_live; ++i) {
    if (!__syncthreads_and(mbar_wait(&bar[stg], par, P.err))) break;  // CTA-uniform give-up
    const int pg = nth_page(i);
    const uint32_t sK = smem_u32(smem + stg * 2 * kBfPageBytes), sV = sK + kBfPageBytes;
    const bool v0 = bf16_slot_live(pg, t0 + g, L, F), v1 = bf16_slot_live(pg, t0 + g + 8, L, F);
    if (__any_sync(0xffffffffu, v0 || v1)) {
      float d[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[nt][e] = 0.f;
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {
        uint32_t a[4];
        ldmatrix_x4(a, sK + bf16_chunk_offset(t0 + r + 8 * (mi & 1), 2 * k8 + (mi >> 1)));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(d[nt], a[0], a[1], a[2], a[3], qf[nt][k8][0], qf[nt][k8][1]);
      }
      uint32_t bT[NT], bB[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float sc0 = v0 ? (d[nt][0] + d[nt][1]) * kScoreLog2 : -INFINITY;
        const float sc1 = v1 ? (d[nt][2] + d[nt][3]) * kScoreLog2 : -INFINITY;
        float mt = fmaxf(sc0, sc1);
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        const float mn = fmaxf(mrow[nt], mt);
        if (mn > mrow[nt]) {  // uniform over the 8 lanes of this head
          const float alpha = fast_exp2(mrow[nt] - mn);
          lrow[nt] *= alpha;
#pragma unroll
          for (int m8 = 0; m8 < 8; ++m8)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][m8][e] *= alpha;
          mrow[nt] = mn;
        }
        const float p0 = fast_exp2(sc0 - mrow[nt]), p1 = fast_exp2(sc1 - mrow[nt]);
        lrow[nt] += p0 + p1;
        bT[nt] = movmatrix_trans(split_bf16(p0));
        bB[nt] = movmatrix_trans(split_bf16(p1));
      }
#pragma unroll
      for (int m8 = 0; m8 < 8; ++m8) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, sV + bf16_chunk_offset(t0 + r + 8 * (mi >> 1), 2 * m8 + (mi & 1)));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt][m8], a[0], a[1], a[2], a[3], bT[nt], bB[nt]);
      }
    }
    __syncthreads();  // every warp is done with this stage
    if (threadIdx.x == 0 && i + kBfStages < n_live) {
      fence_proxy_async();
      issue(i + kBfStages, stg);
    }
    if (++stg == kBfStages) {
      stg = 0;
      par ^= 1u;
    }
  }
  if (i < n_live) {
    // gave up at live page i: bounded waits for the copies issued for pages i .. i+kBfStages-1,
    // then an empty partial (the timeout bit is set)
    if (threadIdx.x == 0) {
      int sj = stg;
      uint32_t pj = par;
      for (int j = 0; j < kBfStages && i + j < n_live; ++j) {
        mbar_wait(&bar[sj], pj, P.err);
        if (++sj == kBfStages) {
          sj = 0;
          pj ^= 1u;
        }
      }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < SLOT; k += blockDim.x) slot[k] = (k < 2 * HG && (k & 1) == 0) ? -INFINITY : 0.f;
    return;
  }
  // lane sums of l over the 8 lanes of each head, then combine the 4 warps in shared memory
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int o = 4; o <= 16; o <<= 1) lrow[nt] += __shfl_xor_sync(0xffffffffu, lrow[nt], o);
  float* red = reinterpret_cast<float*>(smem);  // the stages are free: every copy was consumed
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = nt * 4 + tq;
    float* o = red + (warp * HG + head) * kHeadDim;
#pragma unroll
    for (int m8 = 0; m8 < 8; ++m8) {
      o[16 * m8 + g] = acc[nt][m8][0] + acc[nt][m8][1];
      o[16 * m8 + g + 8] = acc[nt][m8][2] + acc[nt][m8][3];
    }
    if (g == 0) {
      red_m[warp][head] = mrow[nt];
      red_l[warp][head] = lrow[nt];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < HG * kHeadDim; idx += blockDim.x) {
    const int head = idx / kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kBfWarps; ++w) M = fmaxf(M, red_m[w][head]);
    float o = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBfWarps; ++w)
        if (red_m[w][head] > -INFINITY) o += fast_exp2(red_m[w][head] - M) * red[(w * HG) * kHeadDim + idx];
    }
    slot[2 * HG + idx] = o;
  }
  if (threadIdx.x < HG) {
    const int head = threadIdx.x;
    float M = -INFINITY, Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kBfWarps; ++w) M = fmaxf(M, red_m[w][head]);
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBfWarps; ++w)
        if (red_m[w][head] > -INFINITY) Ls += fast_exp2(red_m[w][head] - M) * red_l[w][head];
    }
    slot[2 * head] = M;
    slot[2 * head + 1] = Ls;
  }
}

// Rows (query heads) per CTA of the rotation kernels: ceil(16 / group) sequences x group heads;
// the CTA stages its KV head's 128x128 fp32 matrix (64 KB) in shared memory with one bulk copy.
constexpr int kRowWarps = 8;
constexpr int kRowsPerCta = 8;
constexpr int kRowsPerWarp = kRowsPerCta / kRowWarps;
constexpr int kUBytes = kHeadDim * kHeadDim * 4;

__device__ __forceinline__ void stage_u(float* sU, uint64_t* bar, const float* Ug) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_expect_tx(bar, kUBytes);
    bulk_g2s(sU, Ug, kUBytes, bar, policy_evict_last());
  }
}

// q_rot[i, h, :] = q[i, h, :] . R_K[layer, kv head] = ((q . U) H) P.
template <int HG>
__global__ void __launch_bounds__(kRowWarps * 32)
    k_rotate_q(DevPool P, StepDims S, int layer, const __nv_bfloat16* __restrict__ q, float* __restrict__ q_rot) {
  constexpr int SG = kRowsPerCta / HG;
  extern __shared__ __align__(128) uint8_t smem[];
  float* sU = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kUBytes);
  const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  stage_u(sU, bar, P.Uk + ((size_t)layer * P.Hkv + h) * kHeadDim * kHeadDim);
  float x[kRowsPerWarp][4], t[kRowsPerWarp][4];
  size_t row[kRowsPerWarp];
  bool ok[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int idx = warp * kRowsPerWarp + r;
    const int bi = blockIdx.x * SG + idx / HG;
    ok[r] = bi < S.n_seqs;
    row[r] = ((size_t)bi * P.Hq + (size_t)h * HG + idx % HG);
    x[r][0] = x[r][1] = x[r][2] = x[r][3] = 0.f;
    if (ok[r]) {
      const uint2 w = *reinterpret_cast<const uint2*>(q + row[r] * kHeadDim + 4 * lane);
      const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
      x[r][0] = __low2float(a);
      x[r][1] = __high2float(a);
      x[r][2] = __low2float(b);
      x[r][3] = __high2float(b);
    }
  }
  __syncthreads();
  if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, P.err))) return;
  matvec_u<kRowsPerWarp>(x, sU, t, lane);
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    fwht128(t[r], lane);
    if (!ok[r]) continue;
    float* o = q_rot + row[r] * kHeadDim;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[rot_pos(lane, e)] = t[r][e];
  }
}

// Softmax-combine n partial slots of one (row, head) in a warp: every lane loads one slot's
// (max, sum) so the loads overlap; a warp max gives the common reference; the output vectors are
// then summed with their weights (lane l holds dims 4l..4l+3). slot(k) returns the slot's base
// pointer or nullptr for an empty one. Result: M (log2 max), Ls (sum), a (unnormalised).
template <int HG, typename SlotFn>
__device__ __forceinline__ void combine_slots(int n, SlotFn slot, int hh, int lane, float& M, float& Ls,
                                              float (&a)[4]) {
  M = -INFINITY;
  Ls = 0.f;
  a[0] = a[1] = a[2] = a[3] = 0.f;
  for (int base = 0; base < n; base += 32) {
    const int k = base + lane;
    const float* sl = k < n ? slot(k) : nullptr;
    float m = -INFINITY, l = 0.f;
    if (sl) {
      m = sl[hh * 2];
      l = sl[hh * 2 + 1];
    }
    float cm = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float nm = fmaxf(M, cm);
    if (nm == -INFINITY) continue;
    const float sa = (M == -INFINITY) ? 0.f : fast_exp2(M - nm);
    const float wk = (m == -INFINITY || !(l > 0.f)) ? 0.f : fast_exp2(m - nm);
    float lk = wk * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lk += __shfl_xor_sync(0xffffffffu, lk, o);
    Ls = Ls * sa + lk;
#pragma unroll
    for (int e = 0; e < 4; ++e) a[e] *= sa;
    const int cnt = min(32, n - base);
    // 16 slots per block, all loads issued before their sums (a block past cnt re-reads the last
    // slot with weight 0, so every load is of a slot that exists)
    for (int jb = 0; jb < cnt; jb += 16) {
      float4 o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        o[j] = *reinterpret_cast<const float4*>(slot(base + min(jb + j, cnt - 1)) + 2 * HG + hh * kHeadDim + 4 * lane);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float wj = __shfl_sync(0xffffffffu, wk, (jb + j) & 31);
        const float w = jb + j < cnt ? wj : 0.f;
        a[0] = fmaf(w, o[j].x, a[0]);
        a[1] = fmaf(w, o[j].y, a[1]);
        a[2] = fmaf(w, o[j].z, a[2]);
        a[3] = fmaf(w, o[j].w, a[3]);
      }
    }
    M = nm;
  }
}

// One CTA per (group of rows, KV head), a row being one (sequence, query head): WPR warps per row
// (kRowWarps / WPR rows per CTA). The warps of a row each softmax-combine every WPR-th INT2 split
// (rotated basis) and the first one joins their results through shared memory; then the
// un-rotation by U_V^T staged in shared memory, and the merge with the BF16 partial. Two warps
// per row serve steps with many splits per row (few sequences), one warp the others.
template <int HG, int WPR>
__global__ void __launch_bounds__(kRowWarps * 32)
    k_merge(DevPool P, StepDims S, int layer, const float* __restrict__ pint2, const float* __restrict__ pbf16,
            float* __restrict__ out) {
  static_assert(kRowsPerWarp == 1, "one row per warp");
  constexpr int RPC = kRowWarps / WPR;  // rows per CTA
  constexpr int SLOT = HG * (2 + kHeadDim);
  extern __shared__ __align__(128) uint8_t smem[];
  float* sU = reinterpret_cast<float*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kUBytes);
  const int h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* buf = reinterpret_cast<float*>(smem + kUBytes + 16) + warp * kHeadDim;
  // exchange area of the warps of a row: [warp][max, sum, 128 outputs]
  float* xch = reinterpret_cast<float*>(smem + kUBytes + 16) + kRowWarps * kHeadDim + warp * (2 + kHeadDim);
  if (!P.absorbed) stage_u(sU, bar, P.Utv + ((size_t)layer * P.Hkv + h) * kHeadDim * kHeadDim);
  const int part = warp % WPR;
  const int rg = blockIdx.x * RPC + warp / WPR;  // this warp's row
  const int bi = rg / HG, hh = rg % HG;
  const bool ok = bi < S.n_seqs;
  const int pair = bi * P.Hkv + h;
  float oi[1][4], Mi, Li, ai[4];
  {
    int n_int2 = 0;
    int64_t wf = 0;
    const int64_t U = P.dims->total_units, NW = P.dims->nw;
    if (ok) {
      const StepSeq& st = P.step[bi];
      if (st.n_pages > 0 && U > 0) {
        const int64_t ua = (int64_t)st.unit_offset + (int64_t)h * st.n_pages, ub = ua + st.n_pages - 1;
        wf = ((ua + 1) * NW - 1) / U;
        n_int2 = (int)(((ub + 1) * NW - 1) / U - wf + 1);
      }
    }
    // every worker owns at least one unit (workers <= units), so workers wf .. wf+n_int2-1 each
    // wrote a partial for this pair; this warp takes every WPR-th of them
    const int mine = n_int2 > part ? (n_int2 - part + WPR - 1) / WPR : 0;
    combine_slots<HG>(mine, [&](int k) -> const float* {
      return pint2 + (size_t)(wf + part + (int64_t)k * WPR + pair) * SLOT;
    }, hh, lane, Mi, Li, ai);
  }
  if constexpr (WPR > 1) {
    if (lane == 0) {
      xch[0] = Mi;
      xch[1] = Li;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) xch[2 + 4 * lane + e] = ai[e];
    __syncthreads();
    if (part == 0) {
      float M = Mi;
#pragma unroll
      for (int j = 1; j < WPR; ++j) M = fmaxf(M, xch[j * (2 + kHeadDim)]);
      float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (M > -INFINITY) {
#pragma unroll
        for (int j = 0; j < WPR; ++j) {
          const float* x = xch + j * (2 + kHeadDim);
          const float mj = x[0];
          if (mj == -INFINITY) continue;
          const float sj = fast_exp2(mj - M);
          L += sj * x[1];
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] = fmaf(sj, x[2 + 4 * lane + e], acc[e]);
        }
      }
      Mi = M;
      Li = L;
#pragma unroll
      for (int e = 0; e < 4; ++e) ai[e] = acc[e];
    }
  }
  {
    const float inv = Li > 0.f ? 1.f / Li : 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) oi[0][e] = ai[e] * inv;
  }
  if (!P.absorbed) {
    // o . R_V^T = ((o P) H) U^T : permute, Walsh-Hadamard, then the basis back-rotation
    float t[1][4], y[1][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) buf[4 * lane + e] = oi[0][e];
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e) t[0][e] = buf[bitrev7(4 * lane + e)];
    fwht128(t[0], lane);
    __syncthreads();
    if (!__all_sync(0xffffffffu, mbar_wait(bar, 0, P.err))) return;
    matvec_u<1>(t, sU, y, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) oi[0][e] = y[0][e];
  }
  if (!ok || part != 0) return;
  float Mb, Lb, ab[4];
  combine_slots<HG>(kBfSlotsPerPair, [&](int k) -> const float* {
    return pbf16 + ((size_t)pair * kBfSlotsPerPair + k) * SLOT;
  }, hh, lane, Mb, Lb, ab);
  float res[4] = {0.f, 0.f, 0.f, 0.f};
  const float Mx = fmaxf(Mi, Mb);
  if (Mx > -INFINITY) {
    const float wi = (Li > 0.f) ? Li * fast_exp2(Mi - Mx) : 0.f;
    const float eb = (Lb > 0.f) ? fast_exp2(Mb - Mx) : 0.f;
    const float den = wi + Lb * eb;
#pragma unroll
    for (int e = 0; e < 4; ++e) res[e] = (wi * oi[0][e] + eb * ab[e]) / den;
  }
  float4* dst = reinterpret_cast<float4*>(out + ((size_t)bi * P.Hq + (size_t)h * HG + hh) * kHeadDim + 4 * lane);
  *dst = make_float4(res[0], res[1], res[2], res[3]);
}

// Warps per merged row: two when the step has on average 16 or more INT2 splits per (sequence,
// KV head) pair (nw_max bounds the step's worker count), else one.
inline int merge_wpr(const StepDims& S) { return S.nw_max >= 16 * S.n_pairs ? 2 : 1; }

}  // namespace

cudaError_t preload_decode_bf16_merge(int hg) {
  cudaFuncAttributes a;
  cudaError_t e = hg == 4 ? cudaFuncGetAttributes(&a, k_decode_bf16<4>) : cudaFuncGetAttributes(&a, k_decode_bf16<8>);
  if (e == cudaSuccess) e = hg == 4 ? cudaFuncGetAttributes(&a, k_merge<4, 1>) : cudaFuncGetAttributes(&a, k_merge<8, 1>);
  if (e == cudaSuccess) e = hg == 4 ? cudaFuncGetAttributes(&a, k_merge<4, 2>) : cudaFuncGetAttributes(&a, k_merge<8, 2>);
  return e;
}

cudaError_t launch_decode_bf16(const DevPool& P, const StepDims& S, int layer, const void* q,
                               float* partials, cudaStream_t s) {
  if (S.n_pairs <= 0) return cudaSuccess;
  const dim3 grid(S.n_pairs);
  if (P.hg == 4) {
    cudaFuncSetAttribute(k_decode_bf16<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBfSmem);
    k_decode_bf16<4><<<grid, kBfWarps * 32, kBfSmem, s>>>(P, S, layer, (const __nv_bfloat16*)q, partials);
  } else {
    cudaFuncSetAttribute(k_decode_bf16<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBfSmem);
    k_decode_bf16<8><<<grid, kBfWarps * 32, kBfSmem, s>>>(P, S, layer, (const __nv_bfloat16*)q, partials);
  }
  return cudaGetLastError();
}

cudaError_t launch_rotate_q(const DevPool& P, const StepDims& S, int layer, const void* q,
                            float* q_rot, cudaStream_t s) {
  if (S.n_seqs <= 0) return cudaSuccess;
  const int sg = kRowsPerCta / P.hg;
  dim3 grid((S.n_seqs + sg - 1) / sg, P.Hkv);
  const int smem = kUBytes + 16;
  if (P.hg == 4) {
    cudaFuncSetAttribute(k_rotate_q<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k_rotate_q<4><<<grid, kRowWarps * 32, smem, s>>>(P, S, layer, (const __nv_bfloat16*)q, q_rot);
  } else {
    cudaFuncSetAttribute(k_rotate_q<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k_rotate_q<8><<<grid, kRowWarps * 32, smem, s>>>(P, S, layer, (const __nv_bfloat16*)q, q_rot);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const DevPool& P, const StepDims& S, int layer, const float* partials_int2,
                         const float* partials_bf16, float* out, cudaStream_t s) {
  if (S.n_pairs <= 0) return cudaSuccess;
  const int wpr = merge_wpr(S), rpc = kRowWarps / wpr;
  dim3 grid((S.n_seqs * P.hg + rpc - 1) / rpc, P.Hkv);
  const int smem = kUBytes + 16 + kRowWarps * kHeadDim * 4 + (wpr > 1 ? kRowWarps * (2 + kHeadDim) * 4 : 0);
  auto go = [&](auto kernel) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kernel<<<grid, kRowWarps * 32, smem, s>>>(P, S, layer, partials_int2, partials_bf16, out);
  };
  if (P.hg == 4) {
    if (wpr > 1) go(k_merge<4, 2>);
    else go(k_merge<4, 1>);
  } else {
    if (wpr > 1) go(k_merge<8, 2>);
    else go(k_merge<8, 1>);
  }
  return cudaGetLastError();
}

}  // namespace oscar
