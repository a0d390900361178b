// Demote on the 5th-generation tensor cores: rotate, clip, quantise and pack rows of K or V.
//
// Method (OSCAR author write-up, m.th-motor.com, serving and rotation paragraphs; order of the
// transforms from "oscar-2bit-kv-cache", arddev.tech, section "Аналитика"): a demoted row x is
// rotated by R = U.H.P, clipped, quantised to 2 bits with an fp16 scale and zero point per group
// and packed into the INT2 history page.
//
// The rotation x.R is a dense contraction ([rows x 128] . [128 x 128]) and runs as a tcgen05 GEMM:
//  * R is built once per (layer, KV head, K|V) at pool creation (rows of U through the fp32
//    Walsh-Hadamard transform and the bit-reversal) and split into two bf16 limbs R = R0 + R1
//    (|R - R0 - R1| <= 2^-18 |R| elementwise, so the rotated row is within 2^-18 |x| of x.R, R's
//    columns being unit vectors); x is bf16, so every product is exact and the two GEMMs
//    accumulate x.R in fp32 in tensor memory (smaller limb first);
//  * operands sit in shared memory K-major with the 128-byte swizzle: two halves of 64 columns,
//    row r of a half at r * 128 bytes, its 16-byte chunk c at chunk position c ^ (r & 7); a tile
//    of contiguous rows of the step's new tokens arrives by two tensor copies (TMA), other tiles
//    by per-thread asynchronous copies into the same layout;
//  * one thread per row reads its 128 fp32 results back from tensor memory (tcgen05.ld) and
//    quantises them with the fp32 spec (each step one IEEE operation), then writes codes and
//    (scale, zero) straight into the page layout the decode kernel reads; a decode step's few
//    rows fill the tile four times over instead, and four lanes share each row, one 32-column
//    chunk each.
// A CTA holds the two limbs (64 KB, one bulk copy each) and runs four groups of 4 warps; each group
// owns a 128-row A tile and 128 of the 512 tensor-memory columns and processes every fourth row
// tile, so one group's quantisation overlaps the others' loads and GEMMs. All waits are bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "device_common.cuh"

namespace oscar {
namespace {

constexpr int kTcRows = 128;                       // rows per tile (GEMM M)
constexpr int kTcGroups = 4;                       // groups of 4 warps per CTA
constexpr int kTcThreads = kTcGroups * kTcRows;
constexpr int kLimbBytes = kHeadDim * kHeadDim * 2;  // one bf16 128x128 operand: 32 KB
constexpr int kRBytes = 2 * kLimbBytes;            // R0, R1
constexpr int kATileBytes = kTcRows * kHeadDim * 2;
constexpr int kStepCache = 256;                    // step-plan rows held in shared memory
constexpr int kBarBytes = 128;                     // mbarriers and the tensor-memory address
constexpr int kTcSmem = kRBytes + kTcGroups * kATileBytes + kBarBytes + kStepCache * (int)sizeof(StepSeq);
// Operand layout (A tiles and the R limbs): K-major with the 128-byte swizzle, the layout the
// tensor copies write. The 128 columns are two halves of 64 (16 KB each for 128 rows); in a half,
// row r is 128 contiguous bytes at r * 128, and its 16-byte chunk c sits at chunk position
// c ^ (r & 7) (rows in 1024-byte groups of 8).
constexpr int kSwHalfBytes = kTcRows * 128;
__host__ __device__ constexpr int sw_offset(int r, int k) {
  return (k >> 6) * kSwHalfBytes + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + (k & 7) * 2;
}

// Shared-memory matrix descriptor (tcgen05) of that layout: start address >> 4, leading byte
// offset 16 (not used by a swizzled K-major operand whose K step fits in the 128-byte row), stride
// byte offset 1024 (the next 8 rows), bit 46 = descriptor version of the sm_100 family, swizzle
// mode 2 (128 bytes) at bits 61-63. K step k (16 columns) starts (k >> 2) halves and (k & 3) * 32
// bytes in; the hardware applies the swizzle to the addresses it forms.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)2 << 61);
}
__host__ __device__ constexpr uint32_t kstep_offset(int k) { return (uint32_t)((k >> 2) * kSwHalfBytes + (k & 3) * 32); }

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9,
// 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kHeadDim >> 3) << 17) |
                            ((uint32_t)(kTcRows >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Tensor maps of the step's new K and V rows (k_new / v_new, [token][KV head][128] bf16) as
// 3-D tensors (dim, KV head, token) with a box of 64 dims x 1 head x 128 tokens written with the
// 128-byte swizzle: two copies fill one A tile. ok == 0: no maps (every tile by per-thread copies).
struct TmaRows {
  CUtensorMap k, v;
  int ok;
};

// One box of a 3-D tensor map into shared memory; completion counted on the mbarrier.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// The same load issued without waiting, and the wait that makes an issued load's registers
// readable (the registers pass through the wait, so no use of them can move above it).
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_wait_pass(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tc_ld_wait1(uint32_t (&a)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  tc_ld_wait_pass(a);
}
// 16 columns as 8 pairs (64-bit registers, so that packed f32x2 arithmetic takes them as they are),
// waited for inside the same statement
__device__ __forceinline__ void tc_ld16_pairs(uint32_t taddr, float2 (&v)[8]) {
  uint64_t r[8];
  asm volatile(
      "{\n .reg .b32 t<16>;\n"
      " tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0,t1,t2,t3,t4,t5,t6,t7,t8,t9,t10,t11,t12,t13,t14,t15}, [%8];\n"
      " tcgen05.wait::ld.sync.aligned;\n"
      " mov.b64 %0, {t0, t1};\n mov.b64 %1, {t2, t3};\n mov.b64 %2, {t4, t5};\n mov.b64 %3, {t6, t7};\n"
      " mov.b64 %4, {t8, t9};\n mov.b64 %5, {t10, t11};\n mov.b64 %6, {t12, t13};\n mov.b64 %7, {t14, t15};\n}\n"
      : "=l"(r[0]), "=l"(r[1]), "=l"(r[2]), "=l"(r[3]), "=l"(r[4]), "=l"(r[5]), "=l"(r[6]), "=l"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = *reinterpret_cast<const float2*>(&r[i]);
}
// 16 columns of this warp's 32 lanes, waited for: the wait carries the registers, so that no use
// of them is scheduled before it
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// quant_code with one IEEE reciprocal per group instead of a division per value. The quotient
// ua = (x - zf) * rcp_sf (rcp_sf = correctly rounded 1/sf) is within 2^-22 |u| of the correctly
// rounded u = (x - zf) / sf, so whenever ua is farther than kCodeMargin from every decision
// threshold both give the same code; values within the margin (and NaN) take the exact path, so
// the result always equals quant_code.
constexpr float kCodeMargin = 1e-5f;

// A group whose frame keeps every value's u = (x - zf) / sf inside (-0.5 + 1e-4, 3.5 - 1e-4) needs
// no clamp: rint(u) is already a code. u is monotonic in x and the fast quotient below is within
// 2^-22 |u| of it, so the group's min and max decide this for all its values.
__device__ __forceinline__ bool group_unclamped(float mn, float mx, float zf, float rcp_sf) {
  const float ulo = __fmul_rn(__fsub_rn(mn, zf), rcp_sf), uhi = __fmul_rn(__fsub_rn(mx, zf), rcp_sf);
  return ulo > -0.5f + 1e-4f && uhi < 3.5f - 1e-4f;
}

constexpr float kRoundMagic = 12582912.f;  // 1.5 * 2^23: x + this, rounded, keeps rint(x) in the low mantissa bits
constexpr float kPackBase = 8388608.f;     // 2^23: its bits are 0x4B000000, so integers below 2^8 added to it
                                           // land in the low byte of the bits
constexpr float kMarginSq = (0.5f - kCodeMargin) * (0.5f - kCodeMargin);

// Packed fp32x2 subtract, a - b per lane, round to nearest even.
__device__ __forceinline__ float2 fsub2_rn(float2 a, float2 b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<const float2*>(&r);
}

// Uniform codes of the values of a chunk (dims q) of a group that needs no clamp, fast path. Each
// code is rint of the exact product (x - zf) * rcp_sf: one fused multiply-add with the constant
// 1.5 * 2^23 rounds it, one subtract from the constant gives -rint exactly. The rounding residual
// e of each value enters e^2 - (0.5 - margin)^2, negative exactly when the value is farther than
// the margin from a threshold; the sign bits are ANDed into neg (started at all ones). The codes
// are packed by exact multiply-adds of powers of two into pk2[j] (started at kPackBase; .x: dim q,
// .y: dim q + 1, for the even q with (q & 7) >> 1 == j), code of dim q at bit 2 ((q >> 3) & 3) of
// the low byte of the float's bits. codes_fast2 takes dims q0 .. q0 + N - 1 as pairs (v[i] holds
// dims q0 + 2i and q0 + 2i + 1); codes_fast32 a whole chunk through an accessor, and returns true
// when some value lies within the margin (the caller then takes the exact path for all 32 values).
template <int N>
__device__ __forceinline__ void codes_fast2(const float2 (&v)[N / 2], int q0, float zf, float rcp_sf, float2 (&pk2)[4],
                                           uint32_t& neg) {
  const float2 z2 = make_float2(zf, zf), rc = make_float2(rcp_sf, rcp_sf);
  const float2 mg = make_float2(kRoundMagic, kRoundMagic), nm2 = make_float2(-kMarginSq, -kMarginSq);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const int q = q0 + i;
    const float2 d = fsub2_rn(v[i / 2], z2);
    const float2 nr = fsub2_rn(mg, __ffma2_rn(d, rc, mg));
    const float2 e = __ffma2_rn(d, rc, nr);
    const float2 w = __ffma2_rn(e, e, nm2);
    neg &= __float_as_uint(w.x) & __float_as_uint(w.y);
    const float pw = -(float)(1 << (2 * ((q >> 3) & 3)));
    pk2[(q & 7) >> 1] = __ffma2_rn(nr, make_float2(pw, pw), pk2[(q & 7) >> 1]);
  }
}
template <typename Val>
__device__ __forceinline__ bool codes_fast32(Val val, float zf, float rcp_sf, float2 (&pk2)[4]) {
  uint32_t neg = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < 4; ++j) pk2[j] = make_float2(kPackBase, kPackBase);
  float2 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = make_float2(val(2 * i), val(2 * i + 1));
  codes_fast2<32>(v, 0, zf, rcp_sf, pk2, neg);
  return (int32_t)neg >= 0;
}

// Lloyd-Max levels (0, a, 3 - a, 3): thresholds t0 = a/2, 1.5, t2 = 3 - a/2
__device__ __forceinline__ uint32_t code_lloyd(float x, float zf, float sf, float rcp_sf, float t0, float t2,
                                               float a) {
  const float ua = __fmul_rn(__fsub_rn(x, zf), rcp_sf);
  const bool far = fabsf(ua - t0) > kCodeMargin && fabsf(ua - 1.5f) > kCodeMargin && fabsf(ua - t2) > kCodeMargin;
  if (!far) return (uint32_t)quant_code(x, zf, sf, a);
  return (ua > t0 ? 1u : 0u) + (ua > 1.5f ? 1u : 0u) + (ua > t2 ? 1u : 0u);
}

// Code bytes of one chunk of 32 values of a group with frame (zf, sf, rcp_sf), sf != 0: the low
// byte of b[k] (k = 0..7) holds the codes of dims q with q & 7 == k, the code of dim q at bit
// 2 ((q >> 3) & 3); byte 1 of b[k] is zero (the other bytes are not used). Uniform levels take the
// fast path when the group needs no clamp and no value lies within the margin of a threshold,
// else quant_code itself; Lloyd-Max levels take code_lloyd.
template <typename Val>
__device__ __forceinline__ void chunk_code_bytes(Val val, float zf, float sf, float rcp_sf, bool unclamped,
                                                 float lloyd_a, uint32_t (&b)[8]) {
  if (lloyd_a > 0.f) {
    const float t0 = __fmul_rn(lloyd_a, 0.5f), t2 = __fsub_rn(3.0f, t0);
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = 0;
#pragma unroll
    for (int q = 0; q < 32; ++q) b[q & 7] |= code_lloyd(val(q), zf, sf, rcp_sf, t0, t2, lloyd_a) << (2 * ((q >> 3) & 3));
    return;
  }
  float2 pk2[4];
  if (unclamped && !codes_fast32(val, zf, rcp_sf, pk2)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      b[2 * j] = __float_as_uint(pk2[j].x);
      b[2 * j + 1] = __float_as_uint(pk2[j].y);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) b[k] = 0;
#pragma unroll
  for (int q = 0; q < 32; ++q) b[q & 7] |= (uint32_t)quant_code(val(q), zf, sf, 0.f) << (2 * ((q >> 3) & 3));
}

// 16-B asynchronous copy global -> shared; src_bytes 0 writes zeros (and reads nothing).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// min / max that return NaN when either input is NaN (a NaN anywhere in a row reaches the row's
// frame, which is how a non-finite input row is detected)
__device__ __forceinline__ float fmin_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Bounded wait on an mbarrier phase in which the waiting warp sleeps (a suspend-time hint of 2 us
// per try) instead of spinning, leaving issue slots to the groups that quantise meanwhile.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t* err) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(2000u)
        : "memory");
    if (ok) return true;
    if (clock64() - t0 >= kWaitCycles) break;
  }
  set_err(err, OSCAR_DEVERR_TIMEOUT);
  return false;
}

// AND-reduction over one group's threads (named barrier 1 + group).
__device__ __forceinline__ bool group_and(int group, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(1 + group), "r"(kTcRows)
      : "memory");
  return out != 0;
}

// R = U.H.P of one (layer, KV head, K|V) -> two bf16 limbs in the B operand layout (element
// (n = output position j, k = input dim i)). With v_rot_absorbed, V's R is the identity.
__global__ void __launch_bounds__(128) k_build_rlimbs(DevPool P, uint8_t* __restrict__ rl) {
  const int mat = blockIdx.x;  // (layer * Hkv + h) * 2 + kv
  const int kv = mat & 1, lh = mat >> 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* dst = rl + (size_t)mat * kRBytes;
  const float* U = (kv == 0 ? P.Uk : P.Uv) + (size_t)lh * kHeadDim * kHeadDim;
  const bool identity = kv == 1 && P.absorbed;
  for (int i = warp; i < kHeadDim; i += 4) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = identity ? (4 * lane + e == i ? 1.f : 0.f) : U[i * kHeadDim + 4 * lane + e];
    if (!identity) fwht128(v, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = identity ? 4 * lane + e : rot_pos(lane, e);
      const float r = v[e];
      const __nv_bfloat16 l0 = __float2bfloat16_rn(r);
      const float r1 = r - __bfloat162float(l0);
      const __nv_bfloat16 l1 = __float2bfloat16_rn(r1);
      const int off = sw_offset(j, i);
      *reinterpret_cast<__nv_bfloat16*>(dst + off) = l0;
      *reinterpret_cast<__nv_bfloat16*>(dst + kLimbBytes + off) = l1;

    }
  }
}

// Row source of one tile row: MODE 0 = the step's demoted rows (k_new / v_new or the recent
// ring), quantised into the pages; MODE 2 = the same for a step of at most 32 rows per (KV head,
// K|V), each row repeated four times in the tile (four lanes share a row's epilogue); MODE 1 = n
// contiguous rows of x, fp32 rotated rows out. One kernel per mode keeps each one's code small.
template <int NG, int MODE>
__global__ void __launch_bounds__(MODE == 2 ? kTcRows : kTcThreads, 1)
    k_demote_tc(DevPool P, StepDims S, int layer, int h_fixed, int kv_fixed, const __nv_bfloat16* __restrict__ k_new,
                const __nv_bfloat16* __restrict__ v_new, int n_rows, float* __restrict__ rows_out,
                const __grid_constant__ TmaRows tma) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sR = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRBytes + kTcGroups * kATileBytes);
  uint64_t* bar_r = bars;         // R limbs landed
  uint64_t* bar_mma = bars + 1;   // [group]: this group's GEMM done
  uint64_t* bar_ld = bars + 1 + kTcGroups;  // [group]: this group's tensor copies landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 1 + 2 * kTcGroups);
  // the step plan, when it fits, is searched in shared memory instead of by dependent global loads
  StepSeq* sstep = reinterpret_cast<StepSeq*>(smem + kRBytes + kTcGroups * kATileBytes + kBarBytes);
  constexpr bool kSteps = MODE != 1;  // rows from the step plan
  const bool cached = kSteps && S.n_seqs <= kStepCache;
  if (cached) {
    const uint4* src = reinterpret_cast<const uint4*>(P.step);
    uint4* dst = reinterpret_cast<uint4*>(sstep);
    for (int i = threadIdx.x; i < S.n_seqs * (int)(sizeof(StepSeq) / 16); i += blockDim.x) dst[i] = src[i];
  }
  const int t = threadIdx.x, group = t / kTcRows, gt = t % kTcRows, warp = t >> 5;
  uint8_t* sA = smem + kRBytes + group * kATileBytes;
  const int h = kSteps ? blockIdx.y : h_fixed;
  const int kv = kSteps ? blockIdx.z : kv_fixed;
  const int total = kSteps ? S.total_dem : n_rows;
  const int mat = (layer * P.Hkv + h) * 2 + kv;

  if (t == 0) {
    mbar_init(bar_r, 1);
    for (int g = 0; g < kTcGroups; ++g) {
      mbar_init(&bar_mma[g], 1);
      mbar_init(&bar_ld[g], 1);
    }
    fence_mbar_init();
    mbar_expect_tx(bar_r, kRBytes);
    const uint8_t* src = P.rlimbs + (size_t)mat * kRBytes;
    for (int l = 0; l < 2; ++l) bulk_g2s(sR + l * kLimbBytes, src + l * kLimbBytes, kLimbBytes, bar_r, policy_evict_last());
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot + (uint32_t)(group * 128);
  const uint32_t taddr_row = tmem + ((uint32_t)((warp % 4) * 32) << 16);

  const float clip = (kv == 0 ? P.clip_k : P.clip_v)[layer * P.Hkv + h];
  const float lloyd_a = P.lloyd ? P.cb_a[mat] : 0.f;
  const __nv_bfloat16* src_new = kv == 0 ? k_new : v_new;
  const __nv_bfloat16* ring = (kv == 0 ? P.ring_k : P.ring_v) + (size_t)layer * P.ring_layer_stride;
  uint8_t* int2_layer = P.int2 + (size_t)layer * P.int2_layer_stride;

  bool ok = true, r_ready = false, mma_ok = true;  // mma_ok: this thread saw each GEMM of its group complete
  uint32_t phase = 0;
  // A decode step demotes few rows: up to 32 per (KV head, K|V) fill one tile four times over
  // (A rows 4r .. 4r+3 hold row r), so that four lanes of one warp share the row's epilogue,
  // one 32-column chunk each. The condition is the same for the whole grid.
  constexpr bool rep4 = MODE == 2;
  const int tile_rows = rep4 ? kTcRows / 4 : kTcRows;
  // This thread's row of a tile: source address, and for the pages its position and page id.
  struct RowSrc {
    const uint8_t* src;
    int pos, pid;
    bool have, swz;
    int slot;
  };
  auto row_src = [&](int tile) {
    RowSrc r{reinterpret_cast<const uint8_t*>(kv == 0 ? k_new : v_new), 0, -1, false, false, 0};
    const int row = tile * tile_rows + (rep4 ? gt >> 2 : gt);
    if (row < total) {
      if (kSteps) {
        const StepSeq* steps = cached ? sstep : P.step;
        const int i = find_step_index(steps, S.n_seqs, row, 0);
        const StepSeq& st = steps[i];
        const int p = st.F_old + (row - st.dem_offset);
        r.pos = p;
        r.pid = P.page_table[(size_t)st.seq_id * P.maxp + ((p - kSink) >> 6)];
        if (p < st.L_old) {
          r.slot = p & (kRecent - 1);
          r.src = reinterpret_cast<const uint8_t*>(ring + (((size_t)st.seq_id * P.Hkv + h) * kRecent) * kHeadDim);
          r.swz = true;
        } else {
          r.src = reinterpret_cast<const uint8_t*>(src_new + ((size_t)(st.in_offset + p - st.L_old) * P.Hkv + h) * kHeadDim);
        }
      } else {
        r.src = reinterpret_cast<const uint8_t*>((kv == 0 ? k_new : v_new) + (size_t)row * kHeadDim);
      }
      r.have = true;
    }
    return r;
  };
  // The tile's rows into the A tile (zeros past the end), asynchronously, 16 B per copy. With one
  // row per thread (r is this thread's row), a warp's 32 rows go in as 16 copies of 8 rows x 4
  // chunks: in copy (rb, cb) lane l takes chunk 4 cb + (l >> 3) of the warp's row 8 rb + (l & 7),
  // whose source comes from that row's lane. Each copy then reads 8 runs of 64 B (instead of 32
  // scattered 16 B pieces) and writes 8 rows x 16 B per chunk, one per 16-byte position of the
  // swizzled rows (no bank conflicts). In the four-lane form every lane copies its row whole (the
  // four copies of the row).
  auto load_row = [&](const RowSrc& r) {
    if constexpr (rep4) {
#pragma unroll
      for (int c = 0; c < 16; ++c)
        cp_async16(sA + sw_offset(gt, 8 * c), r.src + (r.have ? (r.swz ? bf16_chunk_offset(r.slot, c) : c * 16) : 0),
                   r.have ? 16u : 0u);
    } else {
      const int lane = gt & 31, wrow = gt - lane;
      const uint32_t meta = (r.have ? 1u : 0u) | (r.swz ? 2u : 0u) | ((uint32_t)r.slot << 2);
#pragma unroll
      for (int rb = 0; rb < 4; ++rb) {
        const int sl = 8 * rb + (lane & 7);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(r.src), sl));
        const uint32_t m = __shfl_sync(0xffffffffu, meta, sl);
        const bool have = (m & 1u) != 0, swz = (m & 2u) != 0;
        const int slot = (int)(m >> 2);
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          const int c = 4 * cb + (lane >> 3);
          cp_async16(sA + sw_offset(wrow + sl, 8 * c), src + (have ? (swz ? bf16_chunk_offset(slot, c) : c * 16) : 0),
                     have ? 16u : 0u);
        }
      }
    }
    cp_async_commit();
  };

  // Codes of the last tile quantised in the bulk form, stored once the next tile's GEMM is issued:
  // the proxy fence at the top of each tile waits for this thread's outstanding global stores,
  // so stores issued a tile earlier have long completed by then.
  uint8_t* pend_blk = nullptr;  // the row's page block (null: nothing to store)
  int pend_tau = 0, pend_pid = -1;
  uint32_t pend_cw[8], pend_sz[NG];
  auto flush = [&]() {
    uint8_t* blk = pend_blk;
    const int tau = pend_tau;
    const uint32_t* cw = pend_cw;
    if (blk) {
      uint32_t* szp = reinterpret_cast<uint32_t*>(blk + 2 * kPage * kCodeBytes + kv * kPage * NG * 4);
#pragma unroll
      for (int k = 0; k < NG; ++k) szp[sz_index(tau, k, NG)] = pend_sz[k];
    }
    if (kv == 1) {
      // V bytes of this token: slice byte 16 (4 g8 + tq) + 4 (2u + (w >> 1)) + 2e + (w & 1); chunks
      // 2j and 2j + 1 are the two bytes of one 16-bit store at + 4j
      const int slice = tau >> 4, ts = tau & 15, tq = (ts >> 1) & 3, e = ts & 1, u = ts >> 3;
      uint8_t* vbase = blk ? blk + kPage * kCodeBytes + slice * 512 + tq * 16 + 8 * u + 2 * e : nullptr;
      if (vbase) {
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          *reinterpret_cast<uint16_t*>(vbase + g8 * 64) = (uint16_t)(cw[g8] & 0xFFFFu);
          *reinterpret_cast<uint16_t*>(vbase + g8 * 64 + 4) = (uint16_t)(cw[g8] >> 16);
        }
      }
    } else if (blk) {
      uint4* d = reinterpret_cast<uint4*>(blk + tau * kCodeBytes);
      d[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      d[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
    }
    pend_blk = nullptr;
  };

  // A bulk tile whose rows (those below total) are all new tokens of one sequence is, in k_new /
  // v_new, 128 consecutive tokens of this KV head: it comes in by two tensor copies (64 dims each),
  // the first token returned here; any other tile returns -1 and goes by per-thread copies.
  const CUtensorMap* tmap = kv == 0 ? &tma.k : &tma.v;
  auto tile_token = [&](int tl) -> int {
    if (MODE != 0 || !tma.ok) return -1;
    const int r0 = tl * tile_rows, rl = min(r0 + tile_rows, total) - 1;
    const StepSeq* steps = cached ? sstep : P.step;
    const StepSeq& st = steps[find_step_index(steps, S.n_seqs, r0, 0)];
    const int p0 = st.F_old + (r0 - st.dem_offset);
    if (rl - st.dem_offset >= st.F_new - st.F_old || p0 < st.L_old) return -1;
    return st.in_offset + (p0 - st.L_old);
  };
  uint32_t ld_phase = 0;    // parity of this group's next tensor-copy completion
  bool ld_pending = false;  // a tensor copy of this group that was not waited for
  auto load_tile = [&](const RowSrc& r, int tok) {
    if (tok >= 0) {
      if (gt == 0) {
        const uint64_t pol = policy_evict_first();
        mbar_expect_tx(&bar_ld[group], kATileBytes);
        tma_load_3d(sA, tmap, 0, h, tok, &bar_ld[group], pol);
        tma_load_3d(sA + kSwHalfBytes, tmap, 64, h, tok, &bar_ld[group], pol);
      }
      ld_pending = true;
    } else {
      load_row(r);
    }
  };

  const int tile_stride = gridDim.x * kTcGroups;
  int tile = blockIdx.x * kTcGroups + group;
  RowSrc cur{};
  int cur_tok = -1;
  if (tile * tile_rows < total) {
    cur = row_src(tile);
    cur_tok = tile_token(tile);
    load_tile(cur, cur_tok);
  }
  for (; tile * tile_rows < total && ok; tile += tile_stride) {
    const bool have = cur.have;
    const int pos = cur.pos, pid = cur.pid;
    const int row = tile * tile_rows + (rep4 ? gt >> 2 : gt);
    bool ld_ok = true;
    if (cur_tok >= 0) {  // tensor copies (async proxy, like the GEMM): the mbarrier is enough
      ld_ok = mbar_wait_sleep(&bar_ld[group], ld_phase, P.err);
      if (ld_ok) {
        ld_phase ^= 1u;
        ld_pending = false;
      }
    } else {
      cp_async_wait_all();
      fence_proxy_async();  // the A tile written by the copies is read by the tensor cores
    }
    tc_fence_before();  // the previous tile's tensor-memory reads come before the barrier
    // One barrier per tile: the group's rows are in, its previous epilogue has left tensor memory,
    // and a failed wait of any of its threads (the rows, the R copy, or the previous GEMM) stops
    // the group.
    ok = group_and(group, mma_ok && ld_ok && (r_ready || mbar_wait_sleep(bar_r, 0, P.err)));
    if (!ok) break;
    r_ready = true;
    // ---- x . (R1 + R0) into this group's tensor-memory columns
    if (gt == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA), r0 = smem_u32(sR);
      uint32_t acc = 0;
      for (int l = 1; l >= 0; --l)
        for (int k = 0; k < kHeadDim / 16; ++k) {
          tc_mma(tmem, smem_desc(a0 + kstep_offset(k)), smem_desc(r0 + l * kLimbBytes + kstep_offset(k)), acc);
          acc = 1;
        }
      tc_commit(&bar_mma[group]);
    }
    if constexpr (MODE == 0) flush();  // the previous tile's codes, while the GEMM runs
    // every thread waits for the GEMM itself; one that gives up (its GEMM may still be in flight)
    // stops the group at the next barrier, and the reads below then see undefined values
    if (mbar_wait_sleep(&bar_mma[group], phase, P.err))
      phase ^= 1u;
    else
      mma_ok = false;
    tc_fence_after();
    // the GEMM has read the A tile: bring in the next tile's rows while this one is quantised
    if ((tile + tile_stride) * tile_rows < total) {
      cur = row_src(tile + tile_stride);
      cur_tok = tile_token(tile + tile_stride);
      load_tile(cur, cur_tok);
    }
    // ---- read the row back in 32-column chunks (every lane takes part in each tcgen05.ld),
    // quantise and store
    if (MODE == 1) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float part[32];
        tc_ld32(taddr_row + (uint32_t)(32 * c), part);
        if (have) {
          float4* o = reinterpret_cast<float4*>(rows_out + (size_t)row * kHeadDim + 32 * c);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = make_float4(part[4 * q], part[4 * q + 1], part[4 * q + 2], part[4 * q + 3]);
        }
      }
    } else if constexpr (rep4) {
      // lane gt handles chunk cq (dims 32cq .. 32cq+31) of row gt >> 2; every lane takes part in
      // every tensor-memory load and shuffle (warp-wide instructions)
      const int cq = gt & 3;
      uint8_t* blk = nullptr;
      int tau = 0;
      if (have) {
        tau = (pos - kSink) & (kPage - 1);
        if (pid < 0 || pid >= P.max_int2_pages) {
          if (cq == 0) set_err(P.err, OSCAR_DEVERR_PAGE);
        } else {
          blk = int2_layer + ((size_t)pid * P.Hkv + h) * P.block_bytes;
        }
      }
      float mine[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) mine[i] = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float part[32];
        tc_ld32(taddr_row + (uint32_t)(32 * cc), part);
        const bool sel = cc == cq;
#pragma unroll
        for (int i = 0; i < 32; ++i) mine[i] = sel ? part[i] : mine[i];
      }
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        mn = fmin_nan(mn, mine[i]);
        mx = fmax_nan(mx, mine[i]);
      }
      if (NG == 1) {  // the row's group spans the four lanes' chunks
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          mn = fmin_nan(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
      }
      // group frame (lo = c*min, hi = c*max, fp16 s and z) of this lane's group
      const float lo = __fmul_rn(clip, mn), hi = __fmul_rn(clip, mx);
      const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
      const __half s16 = __float2half_rn(s32), z16 = __float2half_rn(lo);
      const float sf = __half2float(s16), zf = __half2float(z16);
      const float rcp = sf != 0.f ? __frcp_rn(sf) : 0.f;
      const bool bad = !isfinite(s32) || !isfinite(lo) || !isfinite(sf) || !isfinite(zf);
      if (blk && (NG == 4 || cq == 0)) {
        uint32_t* szp = reinterpret_cast<uint32_t*>(blk + 2 * kPage * kCodeBytes + kv * kPage * NG * 4);
        szp[sz_index(tau, NG == 1 ? 0 : cq, NG)] = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
      }
      // a non-finite input value makes every rotated value of its row non-finite
      if (have && bad && (NG == 4 || cq == 0))
        set_err(P.err, (isfinite(mn) && isfinite(mx)) ? OSCAR_DEVERR_SCALE : OSCAR_DEVERR_INPUT);
      // codes of dims 32cq + q. K: word (q & 7) >> 1 of the chunk pair, bit 16 (q & 1) + 2 ((q >> 3) & 3)
      // + 8 (cq & 1); V: byte (g8 = q & 7, w = cq), bits 2 ((q >> 3) & 3)
      uint32_t kt[4] = {0, 0, 0, 0}, vt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (sf != 0.f) {  // a group with sf == 0 codes to 0
        uint32_t b[8];
        chunk_code_bytes([&](int q) { return mine[q]; }, zf, sf, rcp, group_unclamped(mn, mx, zf, rcp), lloyd_a, b);
#pragma unroll
        for (int j = 0; j < 4; ++j) kt[j] = __byte_perm(b[2 * j], b[2 * j + 1], 0x1410u);  // low bytes to bytes 0, 2
#pragma unroll
        for (int k = 0; k < 8; ++k) vt[k] = b[k] & 0xFFu;
      }
      if (kv == 0) {
        // word (a, j = cq >> 1) of the token's 32 B is kt[a] of chunk 2j OR (kt[a] << 8) of chunk 2j + 1
        uint32_t w[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          w[a] = kt[a] << (8 * (cq & 1));
          w[a] |= __shfl_xor_sync(0xffffffffu, w[a], 1);
        }
        if (blk) {  // the pair's even lane writes a = 0, 1, the odd lane a = 2, 3; word (a, j) at 2a + j
          uint32_t* d = reinterpret_cast<uint32_t*>(blk + tau * kCodeBytes);
          const int a0 = 2 * (cq & 1), j = cq >> 1;
          d[2 * a0 + j] = (cq & 1) ? w[2] : w[0];
          d[2 * (a0 + 1) + j] = (cq & 1) ? w[3] : w[1];
        }
      } else if (blk) {
        const int slice = tau >> 4, ts = tau & 15, tq = (ts >> 1) & 3, e = ts & 1, u = ts >> 3;
        uint8_t* vbase = blk + kPage * kCodeBytes + slice * 512 + tq * 16 + 8 * u + 2 * e;
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) vbase[g8 * 64 + 4 * (cq >> 1) + (cq & 1)] = (uint8_t)vt[g8];
      }
    } else {
      bool bad = false, nonfin = false;
      uint32_t szw[NG];  // the row's (s, z) words, stored with the codes after the last chunk
      // group frame (lo = c*min, hi = c*max, fp16 s and z) of one group's min and max; a
      // non-finite input value makes every rotated value of its row non-finite (NaN-propagating
      // min / max carry it into the frame)
      auto frame = [&](float mn, float mx, int gr, float& zf, float& sf, float& rcp, bool& unclamped) {
        nonfin |= !(isfinite(mn) && isfinite(mx));
        const float lo = __fmul_rn(clip, mn), hi = __fmul_rn(clip, mx);
        const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
        const __half s16 = __float2half_rn(s32), z16 = __float2half_rn(lo);
        sf = __half2float(s16);
        zf = __half2float(z16);
        rcp = sf != 0.f ? __frcp_rn(sf) : 0.f;
        unclamped = group_unclamped(mn, mx, zf, rcp);
        bad |= !isfinite(s32) || !isfinite(lo) || !isfinite(sf) || !isfinite(zf);
        const uint32_t w = (uint32_t)__half_as_ushort(s16) | ((uint32_t)__half_as_ushort(z16) << 16);
#pragma unroll
        for (int k = 0; k < NG; ++k)  // gr is a compile-time constant for NG == 1 and after unrolling
          if (k == gr) szw[k] = w;
      };
      float zf = 0.f, sf = 0.f, rcp = 0.f;
      bool unclamped = false;
      // the row's codes: K word a of chunk pair j at cw[2a + j]; V: byte c of cw[g8] is chunk c's byte g8
      // (a tile holds K rows or V rows only, so one array serves both)
      uint32_t cw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t kt[4] = {0, 0, 0, 0};  // K words of the current chunk pair
      // quantise chunk c (dims 32c .. 32c + 31), held in a. dim j = 32c + q. K: word 2 ((j & 7) >> 1)
      // + (j >> 6), bit 16 (j & 1) + 8 ((j >> 5) & 1) + 2 ((j >> 3) & 3); V: byte (g8 = j & 7, w = j >> 5),
      // bits 2 ((j >> 3) & 3)
      // chunk c's code bytes b (the low byte of b[k] holds dims q with q & 7 == k) into the row's words
      auto place = [&](int c, const uint32_t (&b)[8]) {
        if (kv == 0) {
          // low bytes of b[2j] (even dims) and b[2j + 1] (odd dims) to bytes (0, 2) of K word j for an
          // even chunk, (1, 3) for an odd one; byte 1 of b[2j] is zero
          const uint32_t sel = (c & 1) ? 0x4101u : 0x1410u;
#pragma unroll
          for (int j = 0; j < 4; ++j) kt[j] |= __byte_perm(b[2 * j], b[2 * j + 1], sel);
        } else {
          // low byte of b[g8] to byte c of cw[g8], the other bytes kept
          const uint32_t sel = 0x7654u & ~(0xFu << (4 * c));
#pragma unroll
          for (int g8 = 0; g8 < 8; ++g8) cw[g8] = __byte_perm(b[g8], cw[g8], sel);
        }
      };
      // quantise chunk c (dims 32c .. 32c + 31) of a group of 32, held in a. dim j = 32c + q.
      // K: word 2 ((j & 7) >> 1) + (j >> 6), bit 16 (j & 1) + 8 ((j >> 5) & 1) + 2 ((j >> 3) & 3);
      // V: byte (g8 = j & 7, w = j >> 5), bits 2 ((j >> 3) & 3)
      auto quant_chunk = [&](int c, const uint32_t (&a)[32]) {
        float mn4[4], mx4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) mn4[k] = mx4[k] = __uint_as_float(a[k]);
#pragma unroll
        for (int q = 4; q < 32; ++q) {
          mn4[q & 3] = fmin_nan(mn4[q & 3], __uint_as_float(a[q]));
          mx4[q & 3] = fmax_nan(mx4[q & 3], __uint_as_float(a[q]));
        }
        frame(fmin_nan(fmin_nan(mn4[0], mn4[1]), fmin_nan(mn4[2], mn4[3])),
              fmax_nan(fmax_nan(mx4[0], mx4[1]), fmax_nan(mx4[2], mx4[3])), c, zf, sf, rcp, unclamped);
        if (sf == 0.f) return;  // a group with sf == 0 codes to 0
        uint32_t b[8];
        chunk_code_bytes([&](int q) { return __uint_as_float(a[q]); }, zf, sf, rcp, unclamped, lloyd_a, b);
        place(c, b);
      };
      // K words of chunks c0 and c0 + 1 (c0 even), accumulated in kt
      auto end_pair = [&](int c0) {
        if (kv == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (c0 == 0) cw[2 * k] = kt[k];
            else cw[2 * k + 1] = kt[k];
            kt[k] = 0;
          }
        }
      };
      if constexpr (NG == 1) {
        // one group over all 128 columns. Tensor memory is read 16 columns at a time (a thread's
        // registers are the limit with four groups): the row's min and max first, then per chunk a
        // fast pass, and a second pass (exact or Lloyd-Max codes) only when some lane needs one.
        // Every lane takes part in every load (warp-wide instructions).
        uint32_t r16[16];
        float mn4[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          tc_ld16(taddr_row + (uint32_t)(16 * c), r16);
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            mn4[q & 3] = fmin_nan(mn4[q & 3], __uint_as_float(r16[q]));
            mx4[q & 3] = fmax_nan(mx4[q & 3], __uint_as_float(r16[q]));
          }
        }
        frame(fmin_nan(fmin_nan(mn4[0], mn4[1]), fmin_nan(mn4[2], mn4[3])),
              fmax_nan(fmax_nan(mx4[0], mx4[1]), fmax_nan(mx4[2], mx4[3])), 0, zf, sf, rcp, unclamped);
        // the fast pass runs on every lane (its codes are used only where it applies)
        const bool fast = sf != 0.f && lloyd_a == 0.f && unclamped;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float2 pk2[4];
          uint32_t neg = 0xFFFFFFFFu;
#pragma unroll
          for (int j = 0; j < 4; ++j) pk2[j] = make_float2(kPackBase, kPackBase);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float2 v2[8];
            tc_ld16_pairs(taddr_row + (uint32_t)(32 * c + 16 * hh), v2);
            codes_fast2<16>(v2, 16 * hh, zf, rcp, pk2, neg);
          }
          uint32_t b[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            b[2 * j] = __float_as_uint(pk2[j].x);
            b[2 * j + 1] = __float_as_uint(pk2[j].y);
          }
          const bool redo = sf != 0.f && (!fast || (int32_t)neg >= 0);
          if (__any_sync(0xffffffffu, redo)) {
#pragma unroll
            for (int k = 0; k < 8; ++k) b[k] = redo ? 0u : b[k];
            const float t0 = __fmul_rn(lloyd_a, 0.5f), t2 = __fsub_rn(3.0f, t0);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              tc_ld16(taddr_row + (uint32_t)(32 * c + 16 * hh), r16);
              if (redo) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const int q = 16 * hh + i;
                  const float x = __uint_as_float(r16[i]);
                  const uint32_t cd = lloyd_a > 0.f ? code_lloyd(x, zf, sf, rcp, t0, t2, lloyd_a)
                                                    : (uint32_t)quant_code(x, zf, sf, 0.f);
                  b[q & 7] |= cd << (2 * ((q >> 3) & 3));
                }
              }
            }
          }
          if (sf != 0.f) place(c, b);  // a group with sf == 0 codes to 0
          if (c & 1) end_pair(c - 1);
        }
      } else {
        // four groups of 32 columns: a chunk per iteration (one copy of the quantiser in the code,
        // which keeps the kernel small enough for the instruction cache)
        uint32_t ra[32];
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          tc_ld32_issue(taddr_row + (uint32_t)(32 * c), ra);
          tc_ld_wait1(ra);
          quant_chunk(c, ra);
          if (c & 1) end_pair(c - 1);
        }
      }
      if (have && bad) set_err(P.err, nonfin ? OSCAR_DEVERR_INPUT : OSCAR_DEVERR_SCALE);
      // the row's page block; its codes and (s, z) words are stored by the next flush
      pend_blk = nullptr;
      pend_tau = 0;
      pend_pid = pid;
      if (have) {
        pend_tau = (pos - kSink) & (kPage - 1);
        if (pid < 0 || pid >= P.max_int2_pages)
          set_err(P.err, OSCAR_DEVERR_PAGE);
        else
          pend_blk = int2_layer + ((size_t)pid * P.Hkv + h) * P.block_bytes;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) pend_cw[k] = cw[k];
#pragma unroll
      for (int k = 0; k < NG; ++k) pend_sz[k] = szw[k];
    }
  }
  if constexpr (MODE == 0) flush();
  cp_async_wait_all();  // no row copy in flight when the CTA leaves
  if (!r_ready && t == 0) mbar_wait(bar_r, 0, P.err);  // never leave with the R copy in flight
  if (!mma_ok && gt == 0) mbar_wait(&bar_mma[group], phase, P.err);  // nor free tensor memory under a GEMM
  if (ld_pending && gt == 0) mbar_wait(&bar_ld[group], ld_phase, P.err);  // nor shared memory under a tensor copy
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(*tmem_slot));
}

template <int NG, int MODE>
cudaError_t launch_tc(const DevPool& P, const StepDims& S, int layer, int h, int kv, dim3 grid, const void* k,
                      const void* v, int n, float* out, const TmaRows& tma, cudaStream_t s) {
  cudaFuncSetAttribute(k_demote_tc<NG, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
  // a decode step's rows fill one tile: one warp group (its tile is tile 0, the group's first)
  k_demote_tc<NG, MODE><<<grid, MODE == 2 ? kTcRows : kTcThreads, kTcSmem, s>>>(P, S, layer, h, kv, (const __nv_bfloat16*)k,
                                                           (const __nv_bfloat16*)v, n, out, tma);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled from the driver (looked up once; null when unavailable)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// The rows map of k_new or v_new (n_tokens x hkv x 128 bf16): false when it cannot be made
// (no encoder, an address not 16-byte aligned), and the kernel then copies every tile per thread.
bool encode_rows_map(CUtensorMap* m, const void* base, int hkv, int n_tokens) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || !base || n_tokens <= 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)n_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hkv * kHeadDim * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kTcRows}, estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t rlimb_bytes_per_matrix() { return kRBytes; }

cudaError_t launch_build_rlimbs(const DevPool& P, uint8_t* rl, int n_mats, cudaStream_t s) {
  k_build_rlimbs<<<n_mats, 128, 0, s>>>(P, rl);
  return cudaGetLastError();
}

cudaError_t launch_demote(const DevPool& P, const StepDims& S, int layer, const void* k_new, const void* v_new,
                          cudaStream_t s) {
  if (S.total_dem <= 0) return cudaSuccess;
  const int tiles = (S.total_dem + kTcRows - 1) / kTcRows;
  // one CTA per SM fits (shared memory): at most one wave over all (KV head, K|V) pairs
  const int per_pair = P.num_sms / (2 * P.Hkv) > 0 ? P.num_sms / (2 * P.Hkv) : 1;
  int gx = (tiles + kTcGroups - 1) / kTcGroups;
  gx = gx < per_pair ? gx : per_pair;
  const dim3 grid(gx > 0 ? gx : 1, P.Hkv, 2);
  TmaRows tma;
  std::memset(&tma, 0, sizeof(tma));
  if (S.total_dem <= kTcRows / 4)  // a decode step: at most 32 rows per (KV head, K|V)
    return P.ngroups == 1 ? launch_tc<1, 2>(P, S, layer, 0, 0, grid, k_new, v_new, 0, nullptr, tma, s)
                          : launch_tc<4, 2>(P, S, layer, 0, 0, grid, k_new, v_new, 0, nullptr, tma, s);
  tma.ok = encode_rows_map(&tma.k, k_new, P.Hkv, S.total_new) && encode_rows_map(&tma.v, v_new, P.Hkv, S.total_new);
  return P.ngroups == 1 ? launch_tc<1, 0>(P, S, layer, 0, 0, grid, k_new, v_new, 0, nullptr, tma, s)
                        : launch_tc<4, 0>(P, S, layer, 0, 0, grid, k_new, v_new, 0, nullptr, tma, s);
}

cudaError_t launch_debug_rotate(const DevPool& P, int layer, int head, int kv, const void* x, int n, float* out,
                                cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int tiles = (n + kTcRows - 1) / kTcRows;
  const dim3 grid((tiles + kTcGroups - 1) / kTcGroups, 1, 1);
  StepDims S{};
  // the rows are passed as k (kv = 0) or v (kv = 1)
  TmaRows tma;
  std::memset(&tma, 0, sizeof(tma));
  return launch_tc<1, 1>(P, S, layer, head, kv, grid, x, x, n, out, tma, s);
}

}  // namespace oscar
