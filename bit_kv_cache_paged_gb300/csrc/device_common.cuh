// Device helpers for liboscar's sm_103a kernels: bulk copies with mbarriers (bounded waits),
// warp-level mma/movmatrix/ldmatrix wrappers, the warp-parallel R = U.H.P rotation, and the
// BF16 page swizzle.
#pragma once

#include "oscar_internal.h"

namespace oscar {

// log2(e) / sqrt(128): softmax in base 2 with scale 1/sqrt(head_dim).
constexpr float kScoreLog2 = 0.12751743082459868f;
// 1 / sqrt(128), orthonormal Walsh-Hadamard scale.
constexpr float kInvSqrtD = 0.088388347648318440f;
// A bounded mbarrier wait gives up after this many SM clock cycles (about 0.5 s at 2 GHz).
constexpr long long kWaitCycles = 1ll << 30;

__device__ __forceinline__ void set_err(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// ---------------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.
// Both addresses 16-B aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity`. Returns false (and sets the timeout bit) if it gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 < kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  set_err(err, OSCAR_DEVERR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------------- mma
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 b16 matrix held in the standard fragment layout (thread (g, t) holds
// row g, columns 2t and 2t+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// (hi, lo) split of an fp32 value into two fp16 halves packed as one f16x2 register.
__device__ __forceinline__ uint32_t split_f16(float v) {
  __half h = __float2half_rn(v);
  __half l = __float2half_rn(v - __half2float(h));
  return (uint32_t)__half_as_ushort(h) | ((uint32_t)__half_as_ushort(l) << 16);
}

// Scale of the lo half in split_f16_scaled_lo: |v - fp16(v)| <= 2^-11 |fp16(v)|, so the scaled
// lo half never exceeds the hi half's magnitude.
constexpr float kLoScale = 2048.f;
constexpr float kLoUnscale = 1.f / 2048.f;

// (hi, lo * 2^11) split of an fp32 value into one f16x2 register.
__device__ __forceinline__ uint32_t split_f16_scaled_lo(float v) {
  __half h = __float2half_rn(v);
  __half l = __float2half_rn((v - __half2float(h)) * kLoScale);
  return (uint32_t)__half_as_ushort(h) | ((uint32_t)__half_as_ushort(l) << 16);
}

// split_f16_scaled_lo of two values, with one paired conversion to f16 and one back.
__device__ __forceinline__ void split2_f16_scaled_lo(float a, float b, uint32_t& ra, uint32_t& rb) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 pa = __floats2half2_rn(a, (a - hf.x) * kLoScale);
  const __half2 pb = __floats2half2_rn(b, (b - hf.y) * kLoScale);
  ra = *reinterpret_cast<const uint32_t*>(&pa);
  rb = *reinterpret_cast<const uint32_t*>(&pb);
}

// (low half, high half) of an f16x2 word as floats.
__device__ __forceinline__ float2 half2_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ uint32_t split_bf16(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
  return (uint32_t)__bfloat16_as_ushort(h) | ((uint32_t)__bfloat16_as_ushort(l) << 16);
}

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

__device__ __forceinline__ int bitrev7(int i) { return (int)(__brev((unsigned)i) >> 25); }

// Batch index of step row r: the largest i with offset_i <= r (offsets ascending);
// field 0: dem_offset (demoted rows), 1: app_offset (appended rows).
__device__ __forceinline__ int find_step_index(const StepSeq* st, int n, int r, int field) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int off = field == 0 ? st[mid].dem_offset : st[mid].app_offset;
    if (off <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 2-bit code of a rotated value x in its group frame (zf, sf = fp32 values of the fp16 zero and
// scale), every step one IEEE fp32 operation: u = (x - zf) / sf; uniform levels: rint(u) clamped
// to [0, 3] (round half to even); Lloyd-Max levels (0, a, 3 - a, 3) when lloyd_a > 0: the
// nearest level, [u > a/2] + [u >= 1.5] + [u > 3 - a/2]. A group with sf == 0 codes to 0.
__device__ __forceinline__ int quant_code(float x, float zf, float sf, float lloyd_a) {
  if (sf == 0.f) return 0;
  const float u = __fdiv_rn(__fsub_rn(x, zf), sf);
  if (lloyd_a > 0.f) {
    const float t0 = __fmul_rn(lloyd_a, 0.5f), t2 = __fsub_rn(3.0f, t0);
    return (u > t0 ? 1 : 0) + (u >= 1.5f ? 1 : 0) + (u > t2 ? 1 : 0);
  }
  return min(3, max(0, __float2int_rn(u)));
}
__device__ __forceinline__ int bitrev5(int i) { return (int)(__brev((unsigned)i) >> 27); }

// ---------------------------------------------------------------------------------- rotation
// Lane l holds elements 4l..4l+3 of a 128-vector. In-place orthonormal Walsh-Hadamard
// transform in natural (Sylvester) order: butterflies at distances 1, 2 inside the lane, then
// 4..64 across lanes (xor 1..16).
__device__ __forceinline__ void fwht128(float (&v)[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float o = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = upper ? (o - v[e]) : (v[e] + o);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] *= kInvSqrtD;
}

// NR rows at once: t[r][e] = sum_i x[r][i] * U[i][4*lane + e]; lane holds x[r][4l..4l+3].
// U: row-major 128x128 fp32 in shared or global memory (16-B aligned).
template <int NR>
__device__ __forceinline__ void matvec_u(const float (&x)[NR][4], const float* __restrict__ U,
                                         float (&t)[NR][4], int lane) {
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) t[r][e] = 0.f;
#pragma unroll 4
  for (int i = 0; i < kHeadDim; ++i) {
    const float4 u = *reinterpret_cast<const float4*>(U + i * kHeadDim + 4 * lane);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const float xi = __shfl_sync(0xffffffffu, x[r][i & 3], i >> 2);
      t[r][0] = fmaf(xi, u.x, t[r][0]);
      t[r][1] = fmaf(xi, u.y, t[r][1]);
      t[r][2] = fmaf(xi, u.z, t[r][2]);
      t[r][3] = fmaf(xi, u.w, t[r][3]);
    }
  }
}

// Position (after the bit-reversal permutation) of FWHT output element 4*lane + e.
__device__ __forceinline__ int rot_pos(int lane, int e) { return bitrev7(4 * lane + e); }

// ---------------------------------------------------------------------------------- INT2 (s, z)
// Index (in 32-bit (scale, zero) words) of token tau, group gr of a page's K or V (s, z) array
// (ng groups per token): within each 16-token tile, tokens g and g + 8 of group gr are adjacent,
// so one 64-bit load gives both.
__host__ __device__ constexpr int sz_index(int tau, int gr, int ng) {
  return ((8 * (tau >> 4) + (tau & 7)) * ng + gr) * 2 + ((tau >> 3) & 1);
}

// ---------------------------------------------------------------------------------- BF16 pages
// A BF16 block of 64 tokens x 128 dims stores token t's 16-B chunk c (dims 8c..8c+7) at
// byte t*256 + ((c ^ (t & 7)) * 16), so ldmatrix reads of 8 consecutive tokens hit 8
// distinct bank groups.
__device__ __forceinline__ int bf16_chunk_offset(int t, int c) { return t * 256 + ((c ^ (t & 7)) << 4); }

}  // namespace oscar
