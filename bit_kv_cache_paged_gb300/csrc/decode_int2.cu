// Split-K paged INT2 decode for GQA on sm_103a.
//
// Method (OSCAR author write-up, m.th-motor.com, serving paragraph): the INT2 kernel unpacks
// the 2-bit codes, restores scale and zero point and accumulates in floating point; keys are
// compared in the rotated basis, so scores use q_rot = q.R_K.
//
// Arithmetic per history token t and query head h of the KV group (G = group size):
//   score[h,t] = sum_groups s_K[t,g] * (q_rot[h,g] . c_K[t,g]) + z_K[t,g] * sum(q_rot[h,g])
//   acc[h,:]  += p[h,t] * (s_V[t,g] * c_V[t,:] + z_V[t,g])
// The two code contractions run on tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate):
//  * codes are exact small integers; one AND of a packed 32-bit word (or of its copy shifted by
//    4 or 6 bits) drops two of them into the mantissas of an f16x2 pair as subnormals
//    c * 2^-20, c * 2^-18 or c * 2^-16 (see slot_op), so unpacking costs about 1.25 ALU
//    instructions per two codes;
//  * those power-of-two factors are undone exactly: folded into the fp16 hi/lo split of q_rot for
//    the scores (per dim), and applied per output dim in the epilogue for the values;
//  * the query side and the softmax weights are split into fp16 hi + lo halves (N = 8 columns =
//    4 heads x {hi, lo}), which keeps ~22 bits of precision (the query's lo half is stored times
//    2^11 and its column scaled back in fp32).
// Work split: every warp is an independent worker with a contiguous range of (pair, page)
// units (pair = (sequence, KV head)); it streams its INT2 pages through a private ring of
// shared-memory stages with 1-D bulk copies (TMA engine) and mbarriers, keeps an online softmax
// per head, and writes one partial (max, sum, unnormalised output) per pair segment it covers.
#include <type_traits>

#include "device_common.cuh"

namespace oscar {
namespace {

constexpr int kWarps = 4;   // workers per CTA
constexpr int kStages = 3;  // INT2 pages in flight per worker (4 CTAs = 16 workers fit per SM)
constexpr int kMinCtas = 4;

template <int NG>
struct Int2Geom {
  static constexpr int BLOCK = int2_block_bytes(kHeadDim / NG);
  static constexpr int SMEM = kWarps * kStages * BLOCK + kWarps * kStages * 8;
};

// Code operands. Within every 16-bit half of a packed 32-bit code word, 2-bit slot k sits at bits
// 2k..2k+1. Three copies of the word (w << 4, w, w >> 6) move every slot to mantissa bits 4-5,
// 6-7 or 8-9, and one AND per operand leaves an f16x2 pair whose halves are the subnormals
// c * 2^(slot_exp(k) - 20):
//   slot k     0     1     2     3     4     5     6     7
//   copy       <<4   <<4   w     w     w     >>6   >>6   >>6
//   bits       4-5   6-7   4-5   6-7   8-9   4-5   6-7   8-9
//   slot_exp   0     2     0     2     4     0     2     4
// Operands this far up the subnormal range multiply at full precision on the tensor core; the
// lowest subnormal slots (c * 2^-24, c * 2^-22, bits 0-3) do not.
constexpr uint32_t kMask4 = 0x00300030u;
constexpr uint32_t kMask6 = 0x00C000C0u;
constexpr uint32_t kMask8 = 0x03000300u;

__host__ __device__ constexpr int slot_exp(int k) { return k < 2 ? 2 * k : k < 5 ? 2 * (k - 2) : 2 * (k - 5); }

__device__ __forceinline__ uint32_t slot_op(uint32_t w, int k) {
  switch (k) {
    case 0: return (w << 4) & kMask4;
    case 1: return (w << 4) & kMask6;
    case 2: return w & kMask4;
    case 3: return w & kMask6;
    case 4: return w & kMask8;
    case 5: return (w >> 6) & kMask4;
    case 6: return (w >> 6) & kMask6;
    default: return (w >> 6) & kMask8;
  }
}

// High bit of slot k alone (Lloyd-Max codebook pass): the operand is 2 * h * 2^(slot_exp(k) - 20),
// h the code's high bit.
constexpr uint32_t kHi4 = 0x00200020u;
constexpr uint32_t kHi6 = 0x00800080u;
constexpr uint32_t kHi8 = 0x02000200u;

__device__ __forceinline__ uint32_t slot_op_hi(uint32_t w, int k) {
  switch (k) {
    case 0: return (w << 4) & kHi4;
    case 1: return (w << 4) & kHi6;
    case 2: return w & kHi4;
    case 3: return w & kHi6;
    case 4: return w & kHi8;
    case 5: return (w >> 6) & kHi4;
    case 6: return (w >> 6) & kHi6;
    default: return (w >> 6) & kHi8;
  }
}

// split2_f16_scaled_lo with the lo residuals formed in one packed f32x2 subtract and multiply.
__device__ __forceinline__ void split2_f16_scaled_lo_x2(float a, float b, uint32_t& ra, uint32_t& rb) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const float2 lo = __fmul2_rn(__fadd2_rn(make_float2(a, b), make_float2(-hf.x, -hf.y)),
                               make_float2(kLoScale, kLoScale));
  const __half2 pa = __floats2half2_rn(a, lo.x);
  const __half2 pb = __floats2half2_rn(b, lo.y);
  ra = *reinterpret_cast<const uint32_t*>(&pa);
  rb = *reinterpret_cast<const uint32_t*>(&pb);
}

// Cursor over (batch index i, KV head h, page p) in unit order, with the sequence's page-table
// row and demote frontier cached while it stays on one sequence.
struct UnitIt {
  int i, h, p, np, F;
  const int32_t* pt;
};

__device__ __forceinline__ void it_load_seq(const DevPool& P, UnitIt& it) {
  const StepSeq& st = P.step[it.i];
  it.np = st.n_pages;
  it.F = st.F_new;
  it.pt = P.page_table + (size_t)st.seq_id * P.maxp;
}

__device__ __forceinline__ void it_seek(const DevPool& P, int n_seqs, int u, UnitIt& it) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {  // largest i with unit_offset_i <= u
    const int mid = (lo + hi + 1) >> 1;
    if (P.step[mid].unit_offset <= u) lo = mid; else hi = mid - 1;
  }
  it.i = lo;
  it_load_seq(P, it);
  const int local = u - P.step[lo].unit_offset;
  it.h = local / it.np;
  it.p = local - it.h * it.np;
}

__device__ __forceinline__ void it_next(const DevPool& P, int n_seqs, UnitIt& it) {
  if (++it.p < it.np) return;
  it.p = 0;
  if (++it.h < P.Hkv) return;
  it.h = 0;
  do {
    ++it.i;
    it.np = it.i < n_seqs ? P.step[it.i].n_pages : 1;
  } while (it.np == 0);
  if (it.i < n_seqs) it_load_seq(P, it);
}

// LM: Lloyd-Max codebook pools. A code c = l + 2h (bits l, h) stands for the level
// (0, a, 3 - a, 3)[c] = a * (c + 2 kappa h), kappa = 1.5 (1 - a) / a: every contraction adds a
// second mma over the high-bit operands with the other factor scaled by kappa, into the same
// accumulators, and the factor a joins the score / output scale.
template <int HG, int NG, bool LM>
__global__ void __launch_bounds__(kWarps * 32, (HG == 4 && NG == 1) ? kMinCtas : (HG == 8 && NG == 1 && !LM) ? 3 : 1)
    k_decode_int2(DevPool P, StepDims S, int layer, const float* __restrict__ q_rot,
                  float* __restrict__ part) {
  constexpr int NT = HG / 4;
  // 16-token tiles per softmax pass (bounded by registers: the pass keeps its own accumulators)
  constexpr int TB = LM ? ((NT == 1 && NG == 1) ? 4 : 1) : (NT == 1 && NG == 1) ? 4 : (NT == 2 && NG == 4) ? 1 : 2;
  constexpr int NTL = LM ? NT : 1;  // n-tiles of the scaled query fragments (LM only)
  constexpr int BLOCK = Int2Geom<NG>::BLOCK;
  constexpr int SLOT = HG * (2 + kHeadDim);
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int w = blockIdx.x * kWarps + warp;
  // this step's worker and unit counts (device copy; the launch covers nw_max workers)
  const int nw = P.dims->nw;
  if (w >= nw) return;
  const int64_t U = P.dims->total_units;
  const int u0 = (int)(((int64_t)w * U) / nw), u1 = (int)(((int64_t)(w + 1) * U) / nw);
  const int n_units = u1 - u0;
  if (n_units <= 0) return;

  uint8_t* stg = smem + (size_t)warp * kStages * BLOCK;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * BLOCK) + warp * kStages;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();
  const uint8_t* layer_base = P.int2 + (size_t)layer * P.int2_layer_stride;

  UnitIt pit;
  it_seek(P, S.n_seqs, u0, pit);
  UnitIt cit = pit;
  int issued = 0;

  // An out-of-range page id is replaced by page 0 (in bounds) so the barrier completes; the
  // error bit fails the call, whose output is then not used.
  auto issue = [&](int s) {
    uint32_t pid = (uint32_t)pit.pt[pit.p];
    if (lane == 0) {
      if (pid >= (uint32_t)P.max_int2_pages) {
        set_err(P.err, OSCAR_DEVERR_PAGE);
        pid = 0;
      }
      const uint8_t* src = layer_base + ((size_t)pid * P.Hkv + pit.h) * BLOCK;
      mbar_expect_tx(&bar[s], BLOCK);
      bulk_g2s(stg + s * BLOCK, src, BLOCK, &bar[s], pol);
    }
    ++issued;
    if (issued < n_units) it_next(P, S.n_seqs, pit);
  };

#pragma unroll 1
  for (int s = 0; s < kStages && s < n_units; ++s) issue(s);

  // ---- segment state
  float m[NT], acc[NT][8][4];
  float2 l2[NT], zacc2[NT][NG];  // two partial sums per thread (tokens g and g + 8)
  uint32_t qf[NT][8][2], qf2[NTL][8][2];
  float dsc[NT], qs[NT][NG];
  float kappa_v = 0.f, a_v = 1.f;

  auto begin_segment = [&](const UnitIt& it) {
    const float* qb = q_rot + ((size_t)it.i * P.Hq + (size_t)it.h * HG) * kHeadDim;
    float a_k = 1.f, kappa_k = 0.f;
    if constexpr (LM) {
      const float* cb = P.cb_a + ((size_t)layer * P.Hkv + it.h) * 2;
      a_k = cb[0];
      a_v = cb[1];
      kappa_k = 1.5f * (1.f - a_k) / a_k;
      kappa_v = 1.5f * (1.f - a_v) / a_v;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float* qh = qb + (nt * 4 + (g >> 1)) * kHeadDim;
      float v[8][4];
      float mx = 0.f, qsum[NG];
#pragma unroll
      for (int k = 0; k < NG; ++k) qsum[k] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float2 a = *reinterpret_cast<const float2*>(qh + 16 * s + 2 * tq);
        const float2 b = *reinterpret_cast<const float2*>(qh + 16 * s + 2 * tq + 8);
        v[s][0] = a.x * kScoreLog2;
        v[s][1] = a.y * kScoreLog2;
        v[s][2] = b.x * kScoreLog2;
        v[s][3] = b.y * kScoreLog2;
        const int gr = NG == 1 ? 0 : (s >> 1);
        qsum[gr] += (v[s][0] + v[s][1]) + (v[s][2] + v[s][3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(v[s][e]));
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
        for (int k = 0; k < NG; ++k) qsum[k] += __shfl_xor_sync(0xffffffffu, qsum[k], o);
      }
      int eh = 14 - (mx > 0.f ? ilogbf(mx) : 0);
      eh = max(-100, min(100, eh));
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        // dims 16s+2tq+{0,1} are slot 2(s&3) of their code word, dims 16s+2tq+{8,9} slot 2(s&3)+1
        const float f0 = ldexpf(1.f, eh - slot_exp(2 * (s & 3)));
        const float f1 = ldexpf(1.f, eh - slot_exp(2 * (s & 3) + 1));
        float x[4] = {v[s][0] * f0, v[s][1] * f0, v[s][2] * f1, v[s][3] * f1};
        uint16_t hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half hh = __float2half_rn(x[e]);
          const __half ll = __float2half_rn((x[e] - __half2float(hh)) * kLoScale);
          hv[e] = __half_as_ushort((g & 1) ? ll : hh);
        }
        qf[nt][s][0] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
        qf[nt][s][1] = (uint32_t)hv[2] | ((uint32_t)hv[3] << 16);
        if constexpr (LM) {  // the same split of kappa * q for the high-bit pass
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float y = x[e] * kappa_k;
            const __half hh = __float2half_rn(y);
            const __half ll = __float2half_rn((y - __half2float(hh)) * kLoScale);
            hv[e] = __half_as_ushort((g & 1) ? ll : hh);
          }
          qf2[nt][s][0] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
          qf2[nt][s][1] = (uint32_t)hv[2] | ((uint32_t)hv[3] << 16);
        }
      }
      // constants of the head whose D columns this thread holds (head tq of this n-tile)
      const float my_dsc = ldexpf(1.f, 20 - eh) * a_k;
      dsc[nt] = __shfl_sync(0xffffffffu, my_dsc, (2 * tq) * 4);
#pragma unroll
      for (int k = 0; k < NG; ++k) qs[nt][k] = __shfl_sync(0xffffffffu, qsum[k], (2 * tq) * 4);
      m[nt] = -INFINITY;
      l2[nt] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < NG; ++k) zacc2[nt][k] = make_float2(0.f, 0.f);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
    }
  };

  auto finalize = [&](int bi, int bh) {
    const int pair = bi * P.Hkv + bh;
    float* slot = part + (size_t)(w + pair) * SLOT;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float lt = l2[nt].x + l2[nt].y, zt[NG];
#pragma unroll
      for (int k = 0; k < NG; ++k) zt[k] = zacc2[nt][k].x + zacc2[nt][k].y;
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) {
        lt += __shfl_xor_sync(0xffffffffu, lt, o);
#pragma unroll
        for (int k = 0; k < NG; ++k) zt[k] += __shfl_xor_sync(0xffffffffu, zt[k], o);
      }
      const int head = nt * 4 + tq;
      if (g == 0) {
        slot[head * 2] = m[nt];
        slot[head * 2 + 1] = lt;
      }
      float* o = slot + 2 * HG + head * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const int dim = 16 * mt + g + 8 * v;
          // dim 16mt+g+8v: slot 2(mt&3)+v; a_v = 1 unless the pool has a Lloyd-Max codebook
          const float unscale = (float)(1 << (20 - slot_exp(2 * (mt & 3) + v))) * a_v;
          const int gr = NG == 1 ? 0 : (mt >> 1);
          o[dim] = fmaf(acc[nt][mt][2 * v + 1], kLoUnscale, acc[nt][mt][2 * v]) * unscale + zt[gr];
        }
    }
  };

  begin_segment(cit);
  // stage s of page k is k mod kStages; its barrier phase parity flips on every wrap
  int s = 0;
  uint32_t par = 0;

#pragma unroll 1
  for (int k = 0; k < n_units; ++k) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[s], par, P.err));
    if (!ok) {
      // give up: wait (bounded) for this worker's other copies in flight, then leave
      int sj = s;
      uint32_t pj = par;
      for (int j = k + 1; j < issued; ++j) {
        if (++sj == kStages) {
          sj = 0;
          pj ^= 1u;
        }
        mbar_wait(&bar[sj], pj, P.err);
      }
      return;
    }
    const int valid = (cit.p == cit.np - 1) ? (cit.F - kSink) - kPage * cit.p : kPage;
    {
      const uint8_t* blk = stg + s * BLOCK;
      const uint8_t* kc = blk;
      const uint8_t* vc = blk + kPage * kCodeBytes;
      const uint32_t* kz = reinterpret_cast<const uint32_t*>(blk + 2 * kPage * kCodeBytes);
      const uint32_t* vz = kz + kPage * NG;
      // TB 16-token tiles per pass: independent mma chains and one softmax reduction per pass.
      // Full pages (all but a pair's last) take the path without masking.
      auto page_pass = [&](auto full_tag, int tb) {
        constexpr bool kFull = decltype(full_tag)::value;
        uint2 k0[TB], k1[TB];
        bool vv[TB][2];
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          const int t0 = (tb + t) * 16;
          k0[t] = *reinterpret_cast<const uint2*>(kc + (t0 + g) * kCodeBytes + tq * 8);
          k1[t] = *reinterpret_cast<const uint2*>(kc + (t0 + g + 8) * kCodeBytes + tq * 8);
          vv[t][0] = kFull || (t0 + g < valid);
          vv[t][1] = kFull || (t0 + g + 8 < valid);
        }
        float d[TB][NT][NG][4];
#pragma unroll
        for (int t = 0; t < TB; ++t)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
              for (int e = 0; e < 4; ++e) d[t][nt][gr][e] = 0.f;
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          const int gr = NG == 1 ? 0 : (s8 >> 1);
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            // slice s8: word s8 >> 2 of the chunk; dims +0/+1 in slot 2(s8&3), dims +8/+9 in the next
            const uint32_t xa = (s8 < 4) ? k0[t].x : k0[t].y;
            const uint32_t xb = (s8 < 4) ? k1[t].x : k1[t].y;
            const int k = 2 * (s8 & 3);
            const uint32_t a0 = slot_op(xa, k), a1 = slot_op(xb, k), a2 = slot_op(xa, k + 1), a3 = slot_op(xb, k + 1);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16(d[t][nt][gr], a0, a1, a2, a3, qf[nt][s8][0], qf[nt][s8][1]);
            if constexpr (LM) {
              const uint32_t h0 = slot_op_hi(xa, k), h1 = slot_op_hi(xb, k), h2 = slot_op_hi(xa, k + 1),
                             h3 = slot_op_hi(xb, k + 1);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_f16(d[t][nt][gr], h0, h1, h2, h3, qf2[nt][s8][0], qf2[nt][s8][1]);
            }
          }
        }
        // scores of tokens (tb+t)*16 + g + 8u, online softmax once per pass; the two tokens
        // (u = 0, 1) of a thread go through packed f32x2 arithmetic
        float2 p[TB][NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float2 sc[TB];
          float mt = -INFINITY;
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            const int tok = (tb + t) * 16 + g;
            float2 acc_s = make_float2(0.f, 0.f);
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
              const uint2 szw = *reinterpret_cast<const uint2*>(kz + sz_index(tok, gr, NG));
              const float2 sz0 = half2_to_float2(szw.x);
              const float2 sz1 = half2_to_float2(szw.y);
              const float2 x = make_float2(fmaf(d[t][nt][gr][1], kLoUnscale, d[t][nt][gr][0]),
                                           fmaf(d[t][nt][gr][3], kLoUnscale, d[t][nt][gr][2]));
              const float2 dot = __fmul2_rn(x, make_float2(dsc[nt], dsc[nt]));
              acc_s = __ffma2_rn(make_float2(sz0.x, sz1.x), dot,
                                 __ffma2_rn(make_float2(sz0.y, sz1.y), make_float2(qs[nt][gr], qs[nt][gr]), acc_s));
            }
            sc[t].x = vv[t][0] ? acc_s.x : -INFINITY;
            sc[t].y = vv[t][1] ? acc_s.y : -INFINITY;
            mt = fmaxf(mt, fmaxf(sc[t].x, sc[t].y));
          }
          // the head's running max only moves if some lane's own max exceeds it; otherwise the
          // 8-lane reduction would return m unchanged and is skipped
          if (__any_sync(0xffffffffu, mt > m[nt])) {
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float mn = fmaxf(m[nt], mt);
            const float alpha = (mn > m[nt]) ? fast_exp2(m[nt] - mn) : 1.f;
            const float2 alpha2 = make_float2(alpha, alpha);
            l2[nt] = __fmul2_rn(l2[nt], alpha2);
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) zacc2[nt][gr] = __fmul2_rn(zacc2[nt][gr], alpha2);
#pragma unroll
            for (int mi = 0; mi < 8; ++mi)
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const float2 v = __fmul2_rn(make_float2(acc[nt][mi][e], acc[nt][mi][e + 1]), alpha2);
                acc[nt][mi][e] = v.x;
                acc[nt][mi][e + 1] = v.y;
              }
            m[nt] = mn;
          }
          const float nref = (m[nt] == -INFINITY) ? 0.f : -m[nt];
#pragma unroll
          for (int t = 0; t < TB; ++t) {
            const float2 e = __fadd2_rn(sc[t], make_float2(nref, nref));
            p[t][nt] = make_float2(fast_exp2(e.x), fast_exp2(e.y));
            l2[nt] = __fadd2_rn(l2[nt], p[t][nt]);
          }
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          const int t0 = (tb + t) * 16;
          const uint4 vw = *reinterpret_cast<const uint4*>(vc + t0 * kCodeBytes + lane * 16);
          const uint32_t W[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
          for (int gr = 0; gr < NG; ++gr) {
            const uint2 szw = *reinterpret_cast<const uint2*>(vz + sz_index(t0 + g, gr, NG));
            const float2 sz0 = half2_to_float2(szw.x);
            const float2 sz1 = half2_to_float2(szw.y);
            const float sv0 = sz0.x, zv0 = sz0.y, sv1 = sz1.x, zv1 = sz1.y;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              // p is exactly 0 for masked tokens; the selects keep stale (s, z) bytes of a partial
              // page out of the sums
              const float2 pm = p[t][nt];
              const float2 sv = make_float2(vv[t][0] ? sv0 : 0.f, vv[t][1] ? sv1 : 0.f);
              const float2 zv = make_float2(vv[t][0] ? zv0 : 0.f, vv[t][1] ? zv1 : 0.f);
              const float2 wv = __fmul2_rn(pm, sv);
              zacc2[nt][gr] = __ffma2_rn(pm, zv, zacc2[nt][gr]);
              const float w0 = wv.x, w1 = wv.y;
              uint32_t r0, r1;
              split2_f16_scaled_lo_x2(w0, w1, r0, r1);
              const uint32_t bT = movmatrix_trans(r0);
              const uint32_t bB = movmatrix_trans(r1);
              [[maybe_unused]] uint32_t bT2 = 0, bB2 = 0;  // Lloyd-Max pools only
              if constexpr (LM) {
                split2_f16_scaled_lo(w0 * kappa_v, w1 * kappa_v, r0, r1);
                bT2 = movmatrix_trans(r0);
                bB2 = movmatrix_trans(r1);
              }
#pragma unroll
              for (int mi = (NG == 1 ? 0 : 2 * gr); mi < (NG == 1 ? 8 : 2 * gr + 2); ++mi) {
                // word (mi >> 2) holds tokens 2tq, 2tq+1 and word 2 + (mi >> 2) tokens 2tq+8, 2tq+9;
                // row dims 16mi+g and 16mi+g+8 are slots 2(mi&3) and 2(mi&3)+1 of both
                const uint32_t lo = W[mi >> 2], hi = W[2 + (mi >> 2)];
                const int k = 2 * (mi & 3);
                mma_f16(acc[nt][mi], slot_op(lo, k), slot_op(lo, k + 1), slot_op(hi, k), slot_op(hi, k + 1), bT, bB);
                if constexpr (LM)
                  mma_f16(acc[nt][mi], slot_op_hi(lo, k), slot_op_hi(lo, k + 1), slot_op_hi(hi, k),
                          slot_op_hi(hi, k + 1), bT2, bB2);
              }
            }
          }
        }
      };
      if (valid == kPage) {
#pragma unroll 1
        for (int tb = 0; tb < kPage / 16; tb += TB) page_pass(std::integral_constant<bool, true>(), tb);
      } else {
#pragma unroll 1
        for (int tb = 0; tb < kPage / 16 && tb * 16 < valid; tb += TB)
          page_pass(std::integral_constant<bool, false>(), tb);
      }
    }
    __syncwarp();
    if (issued < n_units) {
      fence_proxy_async();
      issue(s);
    }
    if (++s == kStages) {
      s = 0;
      par ^= 1u;
    }
    const bool last = (k == n_units - 1);
    const int bi = cit.i, bh = cit.h;
    if (!last) it_next(P, S.n_seqs, cit);
    if (last || cit.i != bi || cit.h != bh) {
      finalize(bi, bh);
      if (!last) begin_segment(cit);
    }
  }
}

template <int HG, int NG, bool LM>
void set_attr() {
  cudaFuncSetAttribute(k_decode_int2<HG, NG, LM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       Int2Geom<NG>::SMEM);
}

template <int HG, int NG, bool LM>
int max_workers_for(int num_sms) {
  set_attr<HG, NG, LM>();
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, k_decode_int2<HG, NG, LM>, kWarps * 32,
                                                    Int2Geom<NG>::SMEM) != cudaSuccess ||
      blocks < 1)
    blocks = 1;
  return blocks * kWarps * num_sms;
}

template <int HG, int NG, bool LM>
cudaError_t launch_t(const DevPool& P, const StepDims& S, int layer, const float* q_rot, float* part,
                     cudaStream_t s) {
  set_attr<HG, NG, LM>();
  const int grid = (S.nw_max + kWarps - 1) / kWarps;
  k_decode_int2<HG, NG, LM><<<grid, kWarps * 32, Int2Geom<NG>::SMEM, s>>>(P, S, layer, q_rot, part);
  return cudaGetLastError();
}

template <int HG, int NG, bool LM>
cudaError_t preload_t() {
  cudaFuncAttributes a;
  return cudaFuncGetAttributes(&a, k_decode_int2<HG, NG, LM>);
}

template <bool LM>
cudaError_t preload_lm(int hg, int ngroups) {
  if (hg == 4) return ngroups == 1 ? preload_t<4, 1, LM>() : preload_t<4, 4, LM>();
  return ngroups == 1 ? preload_t<8, 1, LM>() : preload_t<8, 4, LM>();
}

template <bool LM>
int max_workers_lm(int hg, int ngroups, int num_sms) {
  if (hg == 4) return ngroups == 1 ? max_workers_for<4, 1, LM>(num_sms) : max_workers_for<4, 4, LM>(num_sms);
  return ngroups == 1 ? max_workers_for<8, 1, LM>(num_sms) : max_workers_for<8, 4, LM>(num_sms);
}

template <bool LM>
cudaError_t launch_lm(const DevPool& P, const StepDims& S, int layer, const float* q_rot, float* partials,
                      cudaStream_t s) {
  if (P.hg == 4)
    return P.ngroups == 1 ? launch_t<4, 1, LM>(P, S, layer, q_rot, partials, s)
                          : launch_t<4, 4, LM>(P, S, layer, q_rot, partials, s);
  return P.ngroups == 1 ? launch_t<8, 1, LM>(P, S, layer, q_rot, partials, s)
                        : launch_t<8, 4, LM>(P, S, layer, q_rot, partials, s);
}

}  // namespace

cudaError_t preload_decode_int2(int hg, int ngroups, int lloyd) {
  return lloyd ? preload_lm<true>(hg, ngroups) : preload_lm<false>(hg, ngroups);
}

int decode_int2_max_workers(int hg, int ngroups, int lloyd, int num_sms) {
  return lloyd ? max_workers_lm<true>(hg, ngroups, num_sms) : max_workers_lm<false>(hg, ngroups, num_sms);
}

cudaError_t launch_decode_int2(const DevPool& P, const StepDims& S, int layer, const float* q_rot,
                               float* partials, cudaStream_t s) {
  if (S.total_units <= 0 || S.nw <= 0) return cudaSuccess;
  return P.lloyd ? launch_lm<true>(P, S, layer, q_rot, partials, s) : launch_lm<false>(P, S, layer, q_rot, partials, s);
}

}  // namespace oscar
