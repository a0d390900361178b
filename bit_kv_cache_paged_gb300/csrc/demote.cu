// Append, the INT2 page layout, and the parity/debug kernels of liboscar. The demote itself
// (rotate by R = U.H.P, clip, quantise, pack; OSCAR author write-up, m.th-motor.com, serving
// paragraph) runs on the tensor cores in demote_tc.cu and writes the layout below.
//
// INT2 block layout (one page x layer x KV head; the decode kernel's operand order):
//   [0, 2048)      K codes, token-major, 32 B per token. Token bytes 8*tq .. 8*tq+7 (tq = 0..3)
//                  hold the 32 codes of dims {16s + 2tq + {0,1,8,9}}; dim j sits in 32-bit
//                  word j>>6 of that 8-B chunk at bit 16*(j&1) + 8*((j>>5)&1) + 2*((j>>3)&3).
//   [2048, 4096)   V codes in 4 slices of 16 tokens x 32 B. Slice byte
//                  16*(4g + tq) + 4*(2u + (w>>1)) + 2e + (w&1) holds the codes of dims
//                  {g + 8p + 32w : p = 0..3} (bits 2p) of token 2tq + e + 8u of the slice
//                  (g = 0..7, tq = 0..3, e = 0..1, u = 0..1, w = 0..3).
//   then           K (scale, zero) fp16 pairs, 64 tokens x 128/G groups, V pairs likewise; the
//                  pair of token tau, group gr at word sz_index(tau, gr, 128/G) (tokens g and
//                  g + 8 of a 16-token tile adjacent).
// Both code orders let the decode kernel turn one 32-bit word and two shifted copies of it into
// eight f16x2 mma operands with one AND each (codes land in fp16 subnormal mantissas; see
// decode_int2.cu).
#include "device_common.cuh"

namespace oscar {

namespace {

constexpr int kAppendStepCache = 256;  // step-plan rows held in shared memory

// Append: 32 threads per (row, kv head) copy 16 B chunks of K and V into the sink page or the
// recent ring (swizzled BF16 layout).
__global__ void __launch_bounds__(256) k_append(DevPool P, StepDims S, int layer,
                                                const __nv_bfloat16* __restrict__ k_new,
                                                const __nv_bfloat16* __restrict__ v_new) {
  // the step plan, when it fits, is searched in shared memory instead of by dependent global loads
  __shared__ StepSeq sstep[kAppendStepCache];
  const bool cached = S.n_seqs <= kAppendStepCache;
  if (cached) {
    const uint4* src = reinterpret_cast<const uint4*>(P.step);
    uint4* dst = reinterpret_cast<uint4*>(sstep);
    for (int i = threadIdx.x; i < S.n_seqs * (int)(sizeof(StepSeq) / 16); i += blockDim.x) dst[i] = src[i];
    __syncthreads();
  }
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int t = threadIdx.x & 31;
  if (item >= S.total_app * P.Hkv) return;
  const int row = item / P.Hkv, h = item - row * P.Hkv;
  const StepSeq* steps = cached ? sstep : P.step;
  const int i = find_step_index(steps, S.n_seqs, row, 1);
  const StepSeq st = steps[i];
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
    szk[(size_t)w * ng + lane] = sz[sz_index(tau, lane, ng)];
    szv[(size_t)w * ng + lane] = sz[kPage * ng + sz_index(tau, lane, ng)];
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
    const uint32_t szw = sz[sz_index(tau, j / P.G, ng)];
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



cudaError_t launch_append(const DevPool& P, const StepDims& S, int layer, const void* k_new,
                          const void* v_new, cudaStream_t s) {
  if (S.total_app <= 0) return cudaSuccess;
  const int items = S.total_app * P.Hkv;
  k_append<<<(items + 7) / 8, 256, 0, s>>>(P, S, layer, (const __nv_bfloat16*)k_new,
                                            (const __nv_bfloat16*)v_new);
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
