// Device twin of workloads/synth.py: the same counter-based SplitMix64 + Irwin-Hall(4) draw,
// bf16 round-to-nearest-even, so a cache filled on the GPU can be regenerated on the host.
// Input generation only; none of the cache method's arithmetic lives here.
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

}  // namespace

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
