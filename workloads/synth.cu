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

// Read-only stream: every thread loads 16-B words with the streaming cache hint, eight in flight,
// and folds them into one word it writes at the end (so the loads are not optimised away).
__global__ void __launch_bounds__(512) k_read_stream(const uint4* __restrict__ p, size_t n16, uint32_t* out) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldcs(p + i + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(p + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  out[blockIdx.x * (size_t)blockDim.x + threadIdx.x] = acc;
}

}  // namespace

// Reads `bytes` (a multiple of 16, 16-B aligned) of device memory once; out: device uint32 array of
// blocks * 512 words, blocks = 4 * (number of SMs).
extern "C" int read_stream(const void* buf, unsigned long long bytes, void* out, int blocks, void* stream) {
  if (bytes == 0 || blocks <= 0) return 0;
  k_read_stream<<<blocks, 512, 0, (cudaStream_t)stream>>>((const uint4*)buf, (size_t)(bytes / 16), (uint32_t*)out);
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
