// Demote (rotate, clip, quantise, pack), append, and the parity/debug kernels of liboscar.
//
// Demote restates the OSCAR serving pipeline (OSCAR author write-up, m.th-motor.com, serving
// paragraph): the oldest recent token is rotated by R = U.H.P (rotation paragraph; the order
// alignment -> Walsh-Hadamard -> bit-reversal is the one in "oscar-2bit-kv-cache",
// arddev.tech, section "Аналитика"), clipped, quantised to 2 bits with an fp16 scale and zero
// point per group, packed 4 codes per byte and written to the INT2 history page.
//
// INT2 block layout (one page x layer x KV head; the decode kernel's operand order):
//   [0, 2048)      K codes, token-major, 32 B per token. Token bytes 8*tq .. 8*tq+7 (tq = 0..3)
//                  hold the 32 codes of dims {16s + 2tq + {0,1,8,9}}; dim j sits in 32-bit
//                  word j>>6 of that 8-B chunk at bit 16*(j&1) + 8*((j>>5)&1) + 2*((j>>3)&3).
//   [2048, 4096)   V codes in 4 slices of 16 tokens x 32 B. Slice byte
//                  16*(4g + tq) + 4*(2u + (w>>1)) + 2e + (w&1) holds the codes of dims
//                  {g + 8p + 32w : p = 0..3} (bits 2p) of token 2tq + e + 8u of the slice
//                  (g = 0..7, tq = 0..3, e = 0..1, u = 0..1, w = 0..3).
//   then           K (scale, zero) fp16 pairs [64][128/G], V pairs [64][128/G].
// Both code orders let the decode kernel turn one 32-bit word and two shifted copies of it into
// eight f16x2 mma operands with one AND each (codes land in fp16 subnormal mantissas; see
// decode_int2.cu).
#include "device_common.cuh"

namespace oscar {

namespace {

constexpr int kDemoteWarps = 8;
constexpr int kDemoteRowsPerWarp = 8;
constexpr int kDemoteNR = 4;  // rows rotated together (U reuse)
constexpr int kDemoteRowsPerCta = kDemoteWarps * kDemoteRowsPerWarp;

__device__ __forceinline__ int find_batch(const StepSeq* st, int n, int r, int field) {
  // largest i with offset_i <= r (offsets ascending); field 0: dem_offset, 1: app_offset
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int off = field == 0 ? st[mid].dem_offset : st[mid].app_offset;
    if (off <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&w.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w.y);
  x[0] = __low2float(a);
  x[1] = __high2float(a);
  x[2] = __low2float(b);
  x[3] = __high2float(b);
}

// Quantise one row held as v[e] = value at position rot_pos(lane, e) and write codes and
// (scale, zero) into the INT2 block. Every step is one IEEE fp32 operation (no contraction).
// lloyd_a > 0: codes index the Lloyd-Max levels (0, a, 3 - a, 3) of the same group frame (nearest
// level of u = (x - z)/s); lloyd_a == 0: the uniform levels (round half to even, clamped).
template <int NG>
__device__ void quantize_store(const float (&v)[4], float clip, float lloyd_a, uint8_t* blk, int kv, int tau,
                               uint8_t* code_buf, int lane, uint32_t* err) {
  float mn[4], mx[4];
  if (NG == 1) {
    float a = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
    float b = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      a = fminf(a, __shfl_xor_sync(0xffffffffu, a, m));
      b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, m));
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) { mn[e] = a; mx[e] = b; }
  } else {
    // group of element e = rot_pos(lane, e) >> 5 = 2*(e&1) + (e>>1): one element per lane
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a = v[e], b = v[e];
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        a = fminf(a, __shfl_xor_sync(0xffffffffu, a, m));
        b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, m));
      }
      mn[e] = a;
      mx[e] = b;
    }
  }
  uint32_t codes_here = 0;
  bool bad = false;
  uint32_t sz[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float lo = __fmul_rn(clip, mn[e]);
    const float hi = __fmul_rn(clip, mx[e]);
    const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    const __half s16 = __float2half_rn(s32);
    const __half z16 = __float2half_rn(lo);
    const float sf = __half2float(s16), zf = __half2float(z16);
    bad |= !isfinite(s32) || !isfinite(lo) || !isfinite(sf) || !isfinite(zf);
    int c = 0;
    if (sf != 0.f) {
      const float u = __fdiv_rn(__fsub_rn(v[e], zf), sf);
      if (lloyd_a > 0.f) {
        const float t0 = __fmul_rn(lloyd_a, 0.5f), t2 = __fsub_rn(3.0f, t0);
        c = (u > t0 ? 1 : 0) + (u >= 1.5f ? 1 : 0) + (u > t2 ? 1 : 0);
      } else {
        c = __float2int_rn(u);
        c = min(3, max(0, c));
      }
    }
    const int pos = rot_pos(lane, e);
    code_buf[pos] = (uint8_t)c;
    codes_here |= (uint32_t)c << (8 * e);
    sz[e] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
  }
  (void)codes_here;
  if (bad && lane == 0) set_err(err, OSCAR_DEVERR_SCALE);
  __syncwarp();
  // (scale, zero) pairs
  uint32_t* szp = reinterpret_cast<uint32_t*>(blk + 2 * kPage * kCodeBytes + kv * kPage * NG * 4) +
                  tau * NG;
  if (lane == 0) {
    if (NG == 1) {
      szp[0] = sz[0];
    } else {
      // group g holds element e with 2*(e&1) + (e>>1) == g
      szp[0] = sz[0];
      szp[1] = sz[2];
      szp[2] = sz[1];
      szp[3] = sz[3];
    }
  }
  // packed codes: lane k builds byte k of this token's 32 code bytes
  const int k = lane;
  uint32_t byte = 0;
  if (kv == 0) {
    const int tq = k >> 3, word = (k >> 2) & 1, b = k & 3, e = b >> 1, sh8 = b & 1;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int j = 64 * word + 32 * sh8 + 8 * p + 2 * tq + e;
      byte |= (uint32_t)code_buf[j] << (2 * p);
    }
    blk[tau * kCodeBytes + k] = (uint8_t)byte;
  } else {
    const int g = k >> 2, word = k & 3;
#pragma unroll
    for (int p = 0; p < 4; ++p) byte |= (uint32_t)code_buf[g + 8 * p + 32 * word] << (2 * p);
    const int slice = tau >> 4, ts = tau & 15;
    const int tq = (ts >> 1) & 3, e = ts & 1, u = ts >> 3;
    blk[kPage * kCodeBytes + slice * 512 + (g * 4 + tq) * 16 + 4 * (2 * u + (word >> 1)) + 2 * e + (word & 1)] =
        (uint8_t)byte;
  }
  __syncwarp();
}

template <int NG>
__global__ void __launch_bounds__(kDemoteWarps * 32)
    k_demote(DevPool P, StepDims S, int layer, const __nv_bfloat16* __restrict__ k_new,
             const __nv_bfloat16* __restrict__ v_new) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* sU = reinterpret_cast<float*>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* code_buf = smem + kHeadDim * kHeadDim * 4 + warp * kHeadDim;
  float* perm_buf = reinterpret_cast<float*>(smem + kHeadDim * kHeadDim * 4 + kDemoteWarps * kHeadDim) +
                    warp * kHeadDim;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kHeadDim * kHeadDim * 4 + kDemoteWarps * kHeadDim +
                                               kDemoteWarps * kHeadDim * 4);
  const int h = blockIdx.y, kv = blockIdx.z;
  const bool rotate = !(kv == 1 && P.absorbed);
  if (rotate && threadIdx.x == 0) {
    // stage this (layer, KV head, K|V) basis U (64 KB) with one bulk copy
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_expect_tx(bar, kHeadDim * kHeadDim * 4);
    bulk_g2s(sU, (kv == 0 ? P.Uk : P.Uv) + ((size_t)layer * P.Hkv + h) * kHeadDim * kHeadDim,
             kHeadDim * kHeadDim * 4, bar, policy_evict_last());
  }
  // row -> (sequence, position, source) for this CTA's rows, one thread per row; the searches
  // overlap with the U copy in flight
  __shared__ int4 s_row[kDemoteRowsPerCta];
  const float clip = (kv == 0 ? P.clip_k : P.clip_v)[layer * P.Hkv + h];
  const float lloyd_a = P.lloyd ? P.cb_a[(layer * P.Hkv + h) * 2 + kv] : 0.f;
  const __nv_bfloat16* src_new = kv == 0 ? k_new : v_new;
  const __nv_bfloat16* ring = (kv == 0 ? P.ring_k : P.ring_v) + (size_t)layer * P.ring_layer_stride;
  uint8_t* int2_layer = P.int2 + (size_t)layer * P.int2_layer_stride;
  bool u_ready = !rotate;

  for (int base = blockIdx.x * kDemoteRowsPerCta; base < S.total_dem;
       base += gridDim.x * kDemoteRowsPerCta) {
    if (threadIdx.x < kDemoteRowsPerCta) {
      const int row = base + threadIdx.x;
      int4 e = make_int4(-1, 0, 0, 0);  // seq id, position, source row of k_new/v_new or -1 (ring)
      if (row < S.total_dem) {
        const int i = find_batch(P.step, S.n_seqs, row, 0);
        const StepSeq& st = P.step[i];
        const int p = st.F_old + (row - st.dem_offset);
        e = make_int4(st.seq_id, p, p < st.L_old ? -1 : st.in_offset + p - st.L_old, 0);
      }
      s_row[threadIdx.x] = e;
    }
    __syncthreads();
    if (!u_ready) {
      const bool got = mbar_wait(bar, 0, P.err);
      if (__syncthreads_and(got) == 0) return;  // CTA-uniform give-up
      u_ready = true;
    }
#pragma unroll 1
    for (int rb = 0; rb < kDemoteRowsPerWarp; rb += kDemoteNR) {
      float x[kDemoteNR][4];
      int seq[kDemoteNR], pos[kDemoteNR];
      bool ok[kDemoteNR];
#pragma unroll
      for (int r = 0; r < kDemoteNR; ++r) {
        const int4 e = s_row[warp * kDemoteRowsPerWarp + rb + r];
        ok[r] = e.x >= 0;
        x[r][0] = x[r][1] = x[r][2] = x[r][3] = 0.f;
        seq[r] = e.x;
        pos[r] = e.y;
        if (ok[r]) {
          const int p = e.y;
          const __nv_bfloat16* src;
          if (e.z < 0) {
            const int slot = p & (kRecent - 1);
            src = ring + (((size_t)e.x * P.Hkv + h) * kRecent) * kHeadDim;
            src = reinterpret_cast<const __nv_bfloat16*>(
                reinterpret_cast<const uint8_t*>(src) + bf16_chunk_offset(slot, lane >> 1) + (lane & 1) * 8);
          } else {
            src = src_new + ((size_t)e.z * P.Hkv + h) * kHeadDim + 4 * lane;
          }
          load_bf16x4(src, x[r]);
          const bool fin = isfinite(x[r][0]) && isfinite(x[r][1]) && isfinite(x[r][2]) && isfinite(x[r][3]);
          if (!__all_sync(0xffffffffu, fin) && lane == 0) set_err(P.err, OSCAR_DEVERR_INPUT);
        }
      }
      float v[kDemoteNR][4];
      if (rotate) {
        matvec_u<kDemoteNR>(x, sU, v, lane);
#pragma unroll
        for (int r = 0; r < kDemoteNR; ++r) fwht128(v[r], lane);
      }
#pragma unroll
      for (int r = 0; r < kDemoteNR; ++r) {
        if (!ok[r]) continue;  // warp-uniform
        if (!rotate) {
          // already-rotated values: bring position rot_pos(lane, e) into element e
#pragma unroll
          for (int e = 0; e < 4; ++e) perm_buf[4 * lane + e] = x[r][e];
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 4; ++e) v[r][e] = perm_buf[rot_pos(lane, e)];
          __syncwarp();
        }
        const int pg = (pos[r] - kSink) >> 6, tau = (pos[r] - kSink) & (kPage - 1);
        const int pid = P.page_table[(size_t)seq[r] * P.maxp + pg];
        if (pid < 0 || pid >= P.max_int2_pages) {
          if (lane == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
          continue;
        }
        uint8_t* blk = int2_layer + ((size_t)pid * P.Hkv + h) * P.block_bytes;
        quantize_store<NG>(v[r], clip, lloyd_a, blk, kv, tau, code_buf, lane, P.err);
      }
    }
    __syncthreads();  // s_row is rewritten for the next chunk
  }
  if (!u_ready) mbar_wait(bar, 0, P.err);  // never leave with the U copy in flight
}

// Append: 32 threads per (row, kv head) copy 16 B chunks of K and V into the sink page or the
// recent ring (swizzled BF16 layout).
__global__ void __launch_bounds__(256) k_append(DevPool P, StepDims S, int layer,
                                                const __nv_bfloat16* __restrict__ k_new,
                                                const __nv_bfloat16* __restrict__ v_new) {
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int t = threadIdx.x & 31;
  if (item >= S.total_app * P.Hkv) return;
  const int row = item / P.Hkv, h = item - row * P.Hkv;
  const int i = find_batch(P.step, S.n_seqs, row, 1);
  const StepSeq st = P.step[i];
  const int a = row - st.app_offset;
  const int n_sink_new = max(0, min(kSink, st.L_new) - st.L_old);
  int pos;
  bool to_sink;
  if (a < n_sink_new) {
    pos = st.L_old + a;
    to_sink = true;
  } else {
    pos = max(st.F_new, st.L_old) + (a - n_sink_new);
    to_sink = false;
  }
  const int kv = t >> 4, c = t & 15;
  const __nv_bfloat16* src = (kv == 0 ? k_new : v_new) +
                             ((size_t)(st.in_offset + pos - st.L_old) * P.Hkv + h) * kHeadDim + 8 * c;
  const uint4 val = *reinterpret_cast<const uint4*>(src);
  uint8_t* dst;
  if (to_sink) {
    if (st.sink_page < 0 || st.sink_page >= P.max_sink_pages) {
      if (t == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
      return;
    }
    __nv_bfloat16* base = (kv == 0 ? P.sink_k : P.sink_v) + (size_t)layer * P.sink_layer_stride +
                          ((size_t)st.sink_page * P.Hkv + h) * kPage * kHeadDim;
    dst = reinterpret_cast<uint8_t*>(base) + bf16_chunk_offset(pos, c);
  } else {
    __nv_bfloat16* base = (kv == 0 ? P.ring_k : P.ring_v) + (size_t)layer * P.ring_layer_stride +
                          ((size_t)st.seq_id * P.Hkv + h) * kRecent * kHeadDim;
    dst = reinterpret_cast<uint8_t*>(base) + bf16_chunk_offset(pos & (kRecent - 1), c);
  }
  *reinterpret_cast<uint4*>(dst) = val;
}

// Debug: the demote path's rotation of plain bf16 rows, written in position order.
__global__ void k_debug_rotate(DevPool P, int layer, int head, int kv, const __nv_bfloat16* x_in,
                               int n, float* out) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= n) return;
  float x[1][4], v[1][4];
  load_bf16x4(x_in + (size_t)warp * kHeadDim + 4 * lane, x[0]);
  float* o = out + (size_t)warp * kHeadDim;
  if (kv == 1 && P.absorbed) {
#pragma unroll
    for (int e = 0; e < 4; ++e) o[4 * lane + e] = x[0][e];
    return;
  }
  const float* U = (kv == 0 ? P.Uk : P.Uv) + ((size_t)layer * P.Hkv + head) * kHeadDim * kHeadDim;
  matvec_u<1>(x, U, v, lane);
  fwht128(v[0], lane);
#pragma unroll
  for (int e = 0; e < 4; ++e) o[rot_pos(lane, e)] = v[0][e];
}

// Debug: INT2 tokens back to canonical layout. One warp per token; lane k writes code byte k.
__global__ void k_debug_read_int2(DevPool P, int seq, int layer, int head, int pos0, int n,
                                  uint8_t* ck, uint32_t* szk, uint8_t* cv, uint32_t* szv) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n) return;
  const int pos = pos0 + w;
  const int pg = (pos - kSink) >> 6, tau = (pos - kSink) & (kPage - 1);
  const int pid = P.page_table[(size_t)seq * P.maxp + pg];
  if (pid < 0 || pid >= P.max_int2_pages) {
    if (lane == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
    return;
  }
  const uint8_t* blk = P.int2 + (size_t)layer * P.int2_layer_stride + ((size_t)pid * P.Hkv + head) * P.block_bytes;
  uint32_t bk = 0, bv = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * lane + q;
    {  // K
      const int tq = (j & 7) >> 1, word = j >> 6, e = j & 1, sh8 = (j >> 5) & 1, p = (j >> 3) & 3;
      const uint8_t byte = blk[tau * kCodeBytes + tq * 8 + word * 4 + 2 * e + sh8];
      bk |= (uint32_t)((byte >> (2 * p)) & 3) << (2 * q);
    }
    {  // V
      const int g = j & 7, word = j >> 5, p = (j >> 3) & 3;
      const int slice = tau >> 4, ts = tau & 15, tq = (ts >> 1) & 3, e = ts & 1, u = ts >> 3;
      const uint8_t byte =
          blk[kPage * kCodeBytes + slice * 512 + (g * 4 + tq) * 16 + 4 * (2 * u + (word >> 1)) + 2 * e + (word & 1)];
      bv |= (uint32_t)((byte >> (2 * p)) & 3) << (2 * q);
    }
  }
  ck[(size_t)w * kCodeBytes + lane] = (uint8_t)bk;
  cv[(size_t)w * kCodeBytes + lane] = (uint8_t)bv;
  const int ng = kHeadDim / P.G;
  const uint32_t* sz = reinterpret_cast<const uint32_t*>(blk + 2 * kPage * kCodeBytes);
  if (lane < ng) {
    szk[(size_t)w * ng + lane] = sz[tau * ng + lane];
    szv[(size_t)w * ng + lane] = sz[kPage * ng + tau * ng + lane];
  }
}

// Diagnostic: raw INT2 key scores q_rot . k_hat (k_hat = code * s + z per group, fp32) of tokens
// [pos0, pos0+n) for the hg query heads of one KV head. One warp per token; lane l covers
// dims 4l..4l+3 of the canonical (rotated, bit-reversed) order.
__global__ void k_debug_int2_scores(DevPool P, int seq, int layer, int head, int pos0, int n,
                                    const float* __restrict__ q_rot, int hg, float* __restrict__ out) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (w >= n) return;
  const int pos = pos0 + w;
  const int pg = (pos - kSink) >> 6, tau = (pos - kSink) & (kPage - 1);
  const int pid = P.page_table[(size_t)seq * P.maxp + pg];
  if (pid < 0 || pid >= P.max_int2_pages) {
    if (lane == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
    return;
  }
  const uint8_t* blk = P.int2 + (size_t)layer * P.int2_layer_stride + ((size_t)pid * P.Hkv + head) * P.block_bytes;
  const int ng = kHeadDim / P.G;
  const uint32_t* sz = reinterpret_cast<const uint32_t*>(blk + 2 * kPage * kCodeBytes);
  const float la = P.cb_a[(layer * P.Hkv + head) * 2];  // K codebook level a (Lloyd-Max pools)
  float kh[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * lane + q;
    const int tq = (j & 7) >> 1, word = j >> 6, e = j & 1, sh8 = (j >> 5) & 1, p = (j >> 3) & 3;
    const uint8_t byte = blk[tau * kCodeBytes + tq * 8 + word * 4 + 2 * e + sh8];
    const uint32_t szw = sz[tau * ng + j / P.G];
    const int c = (byte >> (2 * p)) & 3;
    const float lv = P.lloyd ? (c == 0 ? 0.f : c == 3 ? 3.f : c == 1 ? la : 3.f - la) : (float)c;
    kh[q] = fmaf(lv, half_lo(szw), half_hi(szw));
  }
  for (int hh = 0; hh < hg; ++hh) {
    const float* qh = q_rot + (size_t)hh * kHeadDim + 4 * lane;
    float d = qh[0] * kh[0] + qh[1] * kh[1] + qh[2] * kh[2] + qh[3] * kh[3];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) out[(size_t)hh * n + w] = d;
  }
}

// Debug: BF16 tokens (sink or ring) back to plain [n][128] rows. 16 threads per token per K/V.
__global__ void k_debug_read_bf16(DevPool P, int seq, int sink_page, int layer, int head, int pos0,
                                  int n, __nv_bfloat16* k_out, __nv_bfloat16* v_out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int tok = idx >> 5, t = idx & 31;
  if (tok >= n) return;
  const int pos = pos0 + tok, kv = t >> 4, c = t & 15;
  const uint8_t* src;
  if (pos < kSink) {
    const __nv_bfloat16* base = (kv == 0 ? P.sink_k : P.sink_v) + (size_t)layer * P.sink_layer_stride +
                                ((size_t)sink_page * P.Hkv + head) * kPage * kHeadDim;
    src = reinterpret_cast<const uint8_t*>(base) + bf16_chunk_offset(pos, c);
  } else {
    const __nv_bfloat16* base = (kv == 0 ? P.ring_k : P.ring_v) + (size_t)layer * P.ring_layer_stride +
                                ((size_t)seq * P.Hkv + head) * kRecent * kHeadDim;
    src = reinterpret_cast<const uint8_t*>(base) + bf16_chunk_offset(pos & (kRecent - 1), c);
  }
  __nv_bfloat16* dst = (kv == 0 ? k_out : v_out) + (size_t)tok * kHeadDim + 8 * c;
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}

// Failure-detection self test: an mbarrier that expects 16 bytes nobody sends. The bounded wait
// runs out, records OSCAR_DEVERR_TIMEOUT and the kernel returns.
__global__ void k_debug_timeout(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_expect_tx(&bar, 16);
  }
  __syncthreads();
  mbar_wait(&bar, 0, err);
}

__global__ void k_scatter_i32(int32_t* dst, const int32_t* pairs, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[pairs[2 * i]] = pairs[2 * i + 1];
}

__global__ void k_transpose_u(const float* U, float* Ut, int n_mats) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_mats * kHeadDim * kHeadDim) return;
  const int m = idx / (kHeadDim * kHeadDim), r = idx % (kHeadDim * kHeadDim);
  const int a = r / kHeadDim, b = r % kHeadDim;
  Ut[(size_t)m * kHeadDim * kHeadDim + b * kHeadDim + a] = U[idx];
}

}  // namespace

cudaError_t launch_scatter_i32(int32_t* dst, const int32_t* pairs, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_scatter_i32<<<(n + 255) / 256, 256, 0, s>>>(dst, pairs, n);
  return cudaGetLastError();
}

cudaError_t launch_debug_timeout(uint32_t* err, cudaStream_t s) {
  k_debug_timeout<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_transpose_u(const float* U, float* Ut, int n_mats, cudaStream_t s) {
  const int total = n_mats * kHeadDim * kHeadDim;
  k_transpose_u<<<(total + 255) / 256, 256, 0, s>>>(U, Ut, n_mats);
  return cudaGetLastError();
}

static size_t demote_smem() {
  return (size_t)kHeadDim * kHeadDim * 4 + kDemoteWarps * kHeadDim + kDemoteWarps * kHeadDim * 4 + 16;
}

cudaError_t launch_demote(const DevPool& P, const StepDims& S, int layer, const void* k_new,
                          const void* v_new, cudaStream_t s) {
  if (S.total_dem <= 0) return cudaSuccess;
  const size_t smem = demote_smem();
  int want = (S.total_dem + kDemoteRowsPerCta - 1) / kDemoteRowsPerCta;
  const int cap = (2 * P.num_sms + 2 * P.Hkv - 1) / (2 * P.Hkv);
  const int gx = want < (cap > 0 ? cap : 1) ? want : (cap > 0 ? cap : 1);
  dim3 grid(gx, P.Hkv, 2);
  if (P.ngroups == 1) {
    cudaFuncSetAttribute(k_demote<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_demote<1><<<grid, kDemoteWarps * 32, smem, s>>>(P, S, layer, (const __nv_bfloat16*)k_new,
                                                      (const __nv_bfloat16*)v_new);
  } else {
    cudaFuncSetAttribute(k_demote<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k_demote<4><<<grid, kDemoteWarps * 32, smem, s>>>(P, S, layer, (const __nv_bfloat16*)k_new,
                                                      (const __nv_bfloat16*)v_new);
  }
  return cudaGetLastError();
}

cudaError_t launch_append(const DevPool& P, const StepDims& S, int layer, const void* k_new,
                          const void* v_new, cudaStream_t s) {
  if (S.total_app <= 0) return cudaSuccess;
  const int items = S.total_app * P.Hkv;
  k_append<<<(items + 7) / 8, 256, 0, s>>>(P, S, layer, (const __nv_bfloat16*)k_new,
                                            (const __nv_bfloat16*)v_new);
  return cudaGetLastError();
}

cudaError_t launch_debug_rotate(const DevPool& P, int layer, int head, int kv, const void* x, int n,
                                float* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_debug_rotate<<<(n + 3) / 4, 128, 0, s>>>(P, layer, head, kv, (const __nv_bfloat16*)x, n, out);
  return cudaGetLastError();
}

cudaError_t launch_debug_read_int2(const DevPool& P, int seq, int layer, int head, int pos0, int n,
                                   uint8_t* ck, void* szk, uint8_t* cv, void* szv, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_debug_read_int2<<<(n + 3) / 4, 128, 0, s>>>(P, seq, layer, head, pos0, n, ck, (uint32_t*)szk, cv,
                                                 (uint32_t*)szv);
  return cudaGetLastError();
}

cudaError_t launch_debug_int2_scores(const DevPool& P, int seq, int layer, int head, int pos0, int n,
                                     const float* q_rot, float* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_debug_int2_scores<<<(n + 3) / 4, 128, 0, s>>>(P, seq, layer, head, pos0, n, q_rot, P.hg, out);
  return cudaGetLastError();
}

cudaError_t launch_debug_read_bf16(const DevPool& P, int seq, int sink_page, int L, int F, int layer,
                                   int head, int pos0, int n, void* k, void* v, cudaStream_t s) {
  (void)L;
  (void)F;
  if (n <= 0) return cudaSuccess;
  k_debug_read_bf16<<<(n * 32 + 127) / 128, 128, 0, s>>>(P, seq, sink_page, layer, head, pos0, n,
                                                         (__nv_bfloat16*)k, (__nv_bfloat16*)v);
  return cudaGetLastError();
}

}  // namespace oscar
