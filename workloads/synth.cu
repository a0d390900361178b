// Device twin of workloads/synth.py: the same counter-based SplitMix64 + Irwin-Hall(4) draw,
// bf16 round-to-nearest-even, so a cache filled on the GPU can be regenerated on the host.
// Input generation only, plus a read-only bandwidth probe for the benchmark's roofline; none of
// the cache method's arithmetic lives here.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// out[(t * n_heads + h) * 128 + d] for t < n_pos, h < n_heads (kv heads head0 .. head0+n_heads-1)
__global__ void k_synth_kv(__nv_bfloat16* out, uint64_t seed, uint64_t tag, uint64_t seq_key,
                           uint64_t layer, uint64_t kv, int head0, int n_heads, int pos0, int n_pos,
                           const uint8_t* mask, float inv_sigma, float outlier_scale) {
  const size_t total = (size_t)n_pos * n_heads * 128;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const int d = (int)(idx & 127);
    const size_t r = idx >> 7;
    const int h = (int)(r % n_heads);
    const int t = (int)(r / n_heads);
    const uint64_t n = (tag << 51) | (seq_key << 41) | (layer << 34) | ((uint64_t)(head0 + h) << 28) |
                       (kv << 27) | ((uint64_t)(pos0 + t) << 7) | (uint64_t)d;
    const uint64_t hsh = mix64(seed + (n + 1ull) * 0x9E3779B97F4A7C15ull);
    const int64_t s = (int64_t)(hsh & 0xFFFF) + (int64_t)((hsh >> 16) & 0xFFFF) +
                      (int64_t)((hsh >> 32) & 0xFFFF) + (int64_t)(hsh >> 48) - 131070;
    const float scale = (mask && mask[h * 128 + d]) ? outlier_scale : inv_sigma;
    out[idx] = __float2bfloat16_rn(__fmul_rn((float)s, scale));
  }
}

// Read-only stream through the bulk-copy engine: every CTA streams its share of the buffer in
// 32 KB chunks through a ring of shared-memory stages (cp.async.bulk + mbarrier, four chunks in
// flight), the way the decode kernels read their pages; one thread folds one word per chunk so the
// copies are consumed. Waits are bounded (about 2^31 cycles), after which the CTA stops early and
// records the failure in out[blockIdx.x] = 0xFFFFFFFF.
constexpr int kRsChunk = 32768, kRsStages = 4;

__device__ __forceinline__ bool rs_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(bar);
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(a), "r"(parity) : "memory");
    if (ok) return true;
    if (clock64() - t0 > (1ll << 31)) return false;
  }
}

__global__ void __launch_bounds__(128) k_read_stream(const uint8_t* __restrict__ p, size_t n_chunks, uint32_t* out) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kRsStages * kRsChunk);
  const size_t first = blockIdx.x, step = gridDim.x;
  const size_t mine = first < n_chunks ? (n_chunks - first + step - 1) / step : 0;
  uint32_t acc = 0;
  bool failed = false;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRsStages; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&bar[s])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    auto issue = [&](size_t k) {
      const int s = (int)(k % kRsStages);
      const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar[s]);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(kRsChunk) : "memory");
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       (uint32_t)__cvta_generic_to_shared(sm + s * kRsChunk)),
                   "l"(p + (first + k * step) * kRsChunk), "r"(kRsChunk), "r"(b)
                   : "memory");
    };
    size_t issued = 0;
    for (; issued < mine && issued < (size_t)kRsStages; ++issued) issue(issued);
    for (size_t k = 0; k < mine; ++k) {
      const int s = (int)(k % kRsStages);
      if (!rs_wait(&bar[s], (uint32_t)((k / kRsStages) & 1))) {
        failed = true;  // leave once the copies already issued have landed (bounded)
        for (size_t j = k + 1; j < issued; ++j) rs_wait(&bar[j % kRsStages], (uint32_t)((j / kRsStages) & 1));
        break;
      }
      acc ^= *reinterpret_cast<const uint32_t*>(sm + s * kRsChunk + (k & 127) * 4);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the read above before the refill
      if (issued < mine) issue(issued++);
    }
  }
  if (threadIdx.x == 0) out[blockIdx.x] = failed ? 0xFFFFFFFFu : acc;
}

}  // namespace

// Reads `bytes` (a multiple of 32 KB, 16-B aligned) of device memory once; out: device uint32
// array of `blocks` words (0xFFFFFFFF marks a CTA whose bounded wait gave up).
extern "C" int read_stream(const void* buf, unsigned long long bytes, void* out, int blocks, void* stream) {
  if (bytes == 0 || blocks <= 0) return 0;
  const int smem = kRsStages * kRsChunk + kRsStages * 8;
  cudaFuncSetAttribute(k_read_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k_read_stream<<<blocks, 128, smem, (cudaStream_t)stream>>>((const uint8_t*)buf, (size_t)(bytes / kRsChunk),
                                                              (uint32_t*)out);
  return (int)cudaGetLastError();
}

extern "C" int synth_kv_bf16(void* out, unsigned long long seed, int tag, int seq_key, int layer,
                             int kv, int head0, int n_heads, int pos0, int n_pos,
                             const void* mask_dev, float inv_sigma, float outlier_scale,
                             void* stream) {
  if (n_pos <= 0 || n_heads <= 0) return 0;
  const size_t total = (size_t)n_pos * n_heads * 128;
  size_t blocks = (total + 255) / 256;
  if (blocks > 65535u * 8u) blocks = 65535u * 8u;
  k_synth_kv<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      (__nv_bfloat16*)out, seed, (uint64_t)tag, (uint64_t)seq_key, (uint64_t)layer, (uint64_t)kv, head0,
      n_heads, pos0, n_pos, (const uint8_t*)mask_dev, inv_sigma, outlier_scale);
  return (int)cudaGetLastError();
}
