// BF16-only paged KV cache decode: the comparison cache of the same shape as an OSCAR cache, with
// every token in BF16 pages (OSCAR author write-up, m.th-motor.com, serving paragraph and Fig. 6
// paragraph, whose decode speedups are measured against a BF16 paged cache).
//
// Page format: one page = 64 tokens x 128 dims of one KV head, 16-B chunk c of token t at byte
// t*256 + ((c ^ (t & 7)) * 16), the same swizzle as the OSCAR pool's BF16 sink and recent pages.
// Split-K decode: a CTA takes a chunk of up to kChunkPages consecutive pages of one
// (sequence, KV head) pair, streams the K and V pages through shared-memory stages with 1-D bulk
// copies and mbarriers (bounded waits), and its 4 warps (16 tokens of every page each) keep an
// online softmax that the CTA combines into one partial (max, sum, unnormalised output) per
// (pair, chunk). A merge kernel combines the chunks of every (sequence, query head).
#include "device_common.cuh"

namespace oscar {
namespace {

constexpr int kBbWarps = 4;
constexpr int kBbStages = 2;
constexpr int kChunkPages = 32;  // pages of one pair per CTA (2048 tokens)
constexpr int kPageBytes = kPage * kHeadDim * 2;  // 16 KB of one page of K or V
constexpr int kBbSmem = kBbStages * 2 * kPageBytes + kBbStages * 8;

struct Bf16Cache {
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* page_table;
  const int32_t* lengths;
  int32_t n_seqs, Hq, Hkv, max_pages, n_chunks;
  int64_t n_pages_total;
  uint32_t* err;
};

__device__ __forceinline__ size_t page_off(const Bf16Cache& C, int64_t pid, int h) {
  return ((size_t)pid * C.Hkv + h) * kPageBytes;
}

template <int HG>
__global__ void __launch_bounds__(kBbWarps * 32)
    k_bf16_paged_decode(Bf16Cache C, const __nv_bfloat16* __restrict__ q, float* __restrict__ part) {
  constexpr int NT = HG / 4;
  constexpr int SLOT = HG * (2 + kHeadDim);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red_m[kBbWarps][HG], red_l[kBbWarps][HG];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kBbStages * 2 * kPageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int pair = blockIdx.y, chunk = blockIdx.x;
  const int bi = pair / C.Hkv, h = pair - bi * C.Hkv;
  const int L = C.lengths[bi];
  const int n_pages = (L + kPage - 1) / kPage;
  const int p0 = chunk * kChunkPages, p1 = min(n_pages, p0 + kChunkPages);
  float* slot = part + ((size_t)pair * C.n_chunks + chunk) * SLOT;
  if (p0 >= p1) {  // empty chunk
    for (int k = threadIdx.x; k < SLOT; k += blockDim.x) slot[k] = (k < 2 * HG && (k & 1) == 0) ? -INFINITY : 0.f;
    return;
  }
  const int32_t* pt = C.page_table + (size_t)bi * C.max_pages;
  auto issue = [&](int p, int s) {  // thread 0 only
    int64_t pid = pt[p];
    if (pid < 0 || pid >= C.n_pages_total) {
      set_err(C.err, OSCAR_DEVERR_PAGE);
      pid = 0;
    }
    uint8_t* dst = smem + s * 2 * kPageBytes;
    mbar_expect_tx(&bar[s], 2 * kPageBytes);
    const uint64_t pol = policy_evict_first();
    bulk_g2s(dst, C.k + page_off(C, pid, h), kPageBytes, &bar[s], pol);
    bulk_g2s(dst + kPageBytes, C.v + page_off(C, pid, h), kPageBytes, &bar[s], pol);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBbStages; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    for (int s = 0; s < kBbStages && p0 + s < p1; ++s) issue(p0 + s, s);
  }
  __syncthreads();

  // query fragments: column 2h' holds head h' of the n-tile, column 2h'+1 is zero
  uint32_t qf[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(
        q + ((size_t)bi * C.Hq + (size_t)h * HG + nt * 4 + (g >> 1)) * kHeadDim);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      qf[nt][s][0] = (g & 1) ? 0u : qh[(16 * s + 2 * tq) >> 1];
      qf[nt][s][1] = (g & 1) ? 0u : qh[(16 * s + 2 * tq + 8) >> 1];
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
  bool ok = true;
  int s = 0;
  uint32_t par = 0;
  int p = p0;
  for (; p < p1; ++p) {
    ok = __all_sync(0xffffffffu, mbar_wait(&bar[s], par, C.err));
    if (!__syncthreads_and(ok)) break;  // CTA-uniform give-up; copies in flight are drained below
    const uint32_t sK = smem_u32(smem + s * 2 * kPageBytes), sV = sK + kPageBytes;
    const int base = p * kPage + t0;
    const bool v0 = base + g < L, v1 = base + g + 8 < L;
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
        if (mn > mrow[nt]) {  // uniform across the 8 lanes of this head
          const float alpha = fast_exp2(mrow[nt] - mn);
          lrow[nt] *= alpha;
#pragma unroll
          for (int m8 = 0; m8 < 8; ++m8)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][m8][e] *= alpha;
          mrow[nt] = mn;
        }
        const float p0v = fast_exp2(sc0 - mrow[nt]), p1v = fast_exp2(sc1 - mrow[nt]);
        lrow[nt] += p0v + p1v;
        bT[nt] = movmatrix_trans(split_bf16(p0v));
        bB[nt] = movmatrix_trans(split_bf16(p1v));
      }
#pragma unroll
      for (int m8 = 0; m8 < 8; ++m8) {
        uint32_t a[4];
        ldmatrix_x4_trans(a, sV + bf16_chunk_offset(t0 + r + 8 * (mi >> 1), 2 * m8 + (mi & 1)));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt][m8], a[0], a[1], a[2], a[3], bT[nt], bB[nt]);
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (threadIdx.x == 0 && p + kBbStages < p1) {
      fence_proxy_async();
      issue(p + kBbStages, s);
    }
    if (++s == kBbStages) {
      s = 0;
      par ^= 1u;
    }
  }
  if (p < p1) {
    // gave up at page p: bounded waits for the copies issued for pages p .. p+kBbStages-1, then
    // an empty partial (the timeout bit is already set)
    if (threadIdx.x == 0) {
      int sj = s;
      uint32_t pj = par;
      for (int j = 0; j < kBbStages && p + j < p1; ++j) {
        mbar_wait(&bar[sj], pj, C.err);
        if (++sj == kBbStages) {
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
  float* red = reinterpret_cast<float*>(smem);
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
    for (int w = 0; w < kBbWarps; ++w) M = fmaxf(M, red_m[w][head]);
    float o = 0.f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBbWarps; ++w)
        if (red_m[w][head] > -INFINITY) o += fast_exp2(red_m[w][head] - M) * red[(w * HG) * kHeadDim + idx];
    }
    slot[2 * HG + idx] = o;
  }
  if (threadIdx.x < HG) {
    const int head = threadIdx.x;
    float M = -INFINITY, Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kBbWarps; ++w) M = fmaxf(M, red_m[w][head]);
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kBbWarps; ++w)
        if (red_m[w][head] > -INFINITY) Ls += fast_exp2(red_m[w][head] - M) * red_l[w][head];
    }
    slot[2 * head] = M;
    slot[2 * head + 1] = Ls;
  }
}

// One warp per (sequence, query head): LSE-combine the chunk partials; lane l holds dims 4l..4l+3.
template <int HG>
__global__ void __launch_bounds__(256) k_bf16_paged_merge(Bf16Cache C, const float* __restrict__ part,
                                                          float* __restrict__ out) {
  constexpr int SLOT = HG * (2 + kHeadDim);
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= C.n_seqs * C.Hq) return;
  const int bi = row / C.Hq, hq = row - bi * C.Hq, h = hq / HG, hh = hq - h * HG;
  const int pair = bi * C.Hkv + h;
  const float* base = part + (size_t)pair * C.n_chunks * SLOT;
  float M = -INFINITY;
  for (int c = lane; c < C.n_chunks; c += 32) M = fmaxf(M, base[(size_t)c * SLOT + 2 * hh]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, Ls = 0.f;
  if (M > -INFINITY) {
    for (int c = 0; c < C.n_chunks; ++c) {
      const float* sl = base + (size_t)c * SLOT;
      const float mc = sl[2 * hh];
      if (mc == -INFINITY) continue;
      const float w = fast_exp2(mc - M);
      Ls += w * sl[2 * hh + 1];
      const float4 o = *reinterpret_cast<const float4*>(sl + 2 * HG + hh * kHeadDim + 4 * lane);
      acc[0] += w * o.x;
      acc[1] += w * o.y;
      acc[2] += w * o.z;
      acc[3] += w * o.w;
    }
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  *reinterpret_cast<float4*>(out + (size_t)row * kHeadDim + 4 * lane) =
      make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
}

// Rows [n][Hkv][128] of positions pos0 .. pos0+n-1 of one sequence -> its pages (swizzled).
// One thread per 16-B chunk.
__global__ void k_bf16_pack(const __nv_bfloat16* __restrict__ rows, int n, int pos0, int Hkv,
                            const int32_t* __restrict__ pt_row, int64_t n_pages_total, uint8_t* __restrict__ kv,
                            uint32_t* err) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)n * Hkv * 16;
  if (idx >= total) return;
  const int c = (int)(idx & 15);
  const int64_t rh = idx >> 4;
  const int h = (int)(rh % Hkv);
  const int i = (int)(rh / Hkv);
  const int pos = pos0 + i;
  const int64_t pid = pt_row[pos / kPage];
  if (pid < 0 || pid >= n_pages_total) {
    set_err(err, OSCAR_DEVERR_PAGE);
    return;
  }
  const int4 v = *reinterpret_cast<const int4*>(rows + ((size_t)i * Hkv + h) * kHeadDim + 8 * c);
  *reinterpret_cast<int4*>(kv + ((size_t)pid * Hkv + h) * kPageBytes + bf16_chunk_offset(pos & (kPage - 1), c)) = v;
}

oscar_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return OSCAR_OK;
  (void)cudaGetLastError();
  return OSCAR_ECUDA;
}

}  // namespace
}  // namespace oscar

using namespace oscar;

extern "C" {

size_t oscar_bf16_partials_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t n_seqs, int32_t max_len) {
  if (num_kv_heads < 1 || num_q_heads % num_kv_heads || n_seqs < 1 || max_len < 1) return 0;
  const int hg = num_q_heads / num_kv_heads;
  if (hg != 4 && hg != 8) return 0;
  const int64_t n_chunks = ((int64_t)max_len + kPage * kChunkPages - 1) / (kPage * kChunkPages);
  return (size_t)n_seqs * num_kv_heads * n_chunks * (size_t)slot_floats(hg) * 4;
}

oscar_status oscar_bf16_pack(const void* rows, int32_t n, int32_t pos0, int32_t num_kv_heads,
                             const int32_t* page_table_row, int64_t n_pages_total, void* kv_pages,
                             uint32_t* err, void* stream) {
  if (!rows || !page_table_row || !kv_pages || !err || n < 0 || pos0 < 0 || num_kv_heads < 1) return OSCAR_EINVAL;
  if (((reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(kv_pages)) & 15) != 0) return OSCAR_EINVAL;
  if (n == 0) return OSCAR_OK;
  const int64_t total = (int64_t)n * num_kv_heads * 16;
  const int threads = 256;
  k_bf16_pack<<<(unsigned)((total + threads - 1) / threads), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(rows), n, pos0, num_kv_heads, page_table_row, n_pages_total,
      static_cast<uint8_t*>(kv_pages), err);
  return cuda_status(cudaGetLastError());
}

oscar_status oscar_bf16_decode(int32_t num_q_heads, int32_t num_kv_heads, int32_t n_seqs, int32_t max_len,
                               const void* k_pages, const void* v_pages, int64_t n_pages_total,
                               const int32_t* page_table, int32_t max_pages_per_seq, const int32_t* lengths,
                               const void* q, void* partials, size_t partials_bytes, float* out, uint32_t* err,
                               void* stream) {
  const size_t need = oscar_bf16_partials_bytes(num_q_heads, num_kv_heads, n_seqs, max_len);
  if (!need || !k_pages || !v_pages || !page_table || !lengths || !q || !partials || !out || !err) return OSCAR_EINVAL;
  if (((reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages) | reinterpret_cast<uintptr_t>(q) |
        reinterpret_cast<uintptr_t>(partials) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return OSCAR_EINVAL;  // read and written in 16-byte pieces
  if (partials_bytes < need || n_pages_total < 1 ||
      max_pages_per_seq < (max_len + kPage - 1) / kPage)
    return OSCAR_EINVAL;
  Bf16Cache C;
  C.k = static_cast<const uint8_t*>(k_pages);
  C.v = static_cast<const uint8_t*>(v_pages);
  C.page_table = page_table;
  C.lengths = lengths;
  C.n_seqs = n_seqs;
  C.Hq = num_q_heads;
  C.Hkv = num_kv_heads;
  C.max_pages = max_pages_per_seq;
  C.n_chunks = (max_len + kPage * kChunkPages - 1) / (kPage * kChunkPages);
  C.n_pages_total = n_pages_total;
  C.err = err;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(partials);
  const dim3 grid(C.n_chunks, n_seqs * num_kv_heads);
  const unsigned mgrid = (unsigned)((n_seqs * num_q_heads + 7) / 8);
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q);
  if (num_q_heads / num_kv_heads == 4) {
    cudaFuncSetAttribute(k_bf16_paged_decode<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBbSmem);
    k_bf16_paged_decode<4><<<grid, kBbWarps * 32, kBbSmem, st>>>(C, qb, part);
    if (cudaGetLastError() != cudaSuccess) return cuda_status(cudaErrorUnknown);
    k_bf16_paged_merge<4><<<mgrid, 256, 0, st>>>(C, part, out);
  } else {
    cudaFuncSetAttribute(k_bf16_paged_decode<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kBbSmem);
    k_bf16_paged_decode<8><<<grid, kBbWarps * 32, kBbSmem, st>>>(C, qb, part);
    if (cudaGetLastError() != cudaSuccess) return cuda_status(cudaErrorUnknown);
    k_bf16_paged_merge<8><<<mgrid, 256, 0, st>>>(C, part, out);
  }
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
