// Internal definitions shared by the host pool and the kernels of liboscar.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/oscar.h"

namespace oscar {

constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kSink = 64;
constexpr int kRecent = 256;
constexpr int kRingPages = kRecent / kPage;       // 4 ring pages of 64 slots
constexpr int kBf16PagesPerPair = 1 + kRingPages;  // sink page + ring pages
constexpr int kCodeBytes = kHeadDim / 4;           // 32 B of 2-bit codes per token row
constexpr int kBf16WarpsPerPage = 4;               // BF16 decode: one warp per 16-token tile
constexpr int kBf16SlotsPerPair = 1;              // one BF16 partial per pair
constexpr int kMinUnitsPerWorker = 4;              // INT2 decode: pages per worker, at least
// Range of the Lloyd-Max codebook's interior level a accepted by the pool: the decode's high-bit
// weight 1.5 (1 - a) / a then stays in [-0.46, 1.5], inside the fp16 range of the split query.
constexpr float kLloydMinA = 0.5f;
constexpr float kLloydMaxA = 1.45f;

// INT2 block of one (page, layer, kv head): K codes [64][32 B], V codes [4 slices][512 B],
// K (s, z) fp16 pairs [64][groups], V (s, z) [64][groups].
constexpr int int2_block_bytes(int group_size) {
  return 2 * kPage * kCodeBytes + 2 * kPage * (kHeadDim / group_size) * 4;
}

// Per batch index of the current step (device-visible, 64 B).
struct StepSeq {
  int32_t seq_id;
  int32_t L_old, L_new;    // length before / after this step's tokens
  int32_t F_old, F_new;    // demote frontier before / after (first recent position)
  int32_t sink_page;
  int32_t n_pages;         // INT2 pages covering [64, F_new)
  int32_t in_offset;       // first row of this sequence in k_new / v_new
  int32_t dem_offset;      // prefix sum of demoted rows (positions [F_old, F_new))
  int32_t app_offset;      // prefix sum of appended rows
  int32_t unit_offset;     // prefix sum of INT2 decode units (kv heads x pages)
  int32_t pad[5];
};
static_assert(sizeof(StepSeq) == 64, "StepSeq layout");

// Shape of the current step. The kernels take it as a launch parameter, except the INT2 unit and
// worker counts, which change whenever a sequence starts a new INT2 page: the INT2 decode and the
// merge read those from the device copy (DevPool::dims), so that a captured step graph stays valid
// across page boundaries. nw_max bounds nw for the batch and sizes the INT2 launch and partials.
struct StepDims {
  int32_t n_seqs;
  int32_t total_new;
  int32_t total_dem;
  int32_t total_app;
  int32_t total_units;
  int32_t nw;                      // INT2 decode workers (warps)
  int32_t n_pairs;                 // n_seqs * Hkv
  int32_t nw_max;                  // upper bound of nw for this batch (launch size, partial slots)
  int32_t pad[8];
};
static_assert(sizeof(StepDims) == 64, "StepDims layout");

// Everything a kernel needs to address the pool (passed by value).
struct DevPool {
  int32_t num_layers, Hq, Hkv, G, ngroups, hg;
  int32_t max_seqs, maxp;          // page-table row length
  int64_t max_int2_pages;
  int32_t max_sink_pages;
  int32_t absorbed;
  int32_t block_bytes;
  int32_t num_sms;
  uint32_t* err;
  const float* Uk;                 // [L][Hkv][128][128]
  const float* Uv;
  const float* Utv;                // U_V transposed per (layer, head)
  const float* clip_k;             // [L][Hkv]
  const float* clip_v;
  const float* cb_a;               // Lloyd-Max codebook interior level a, [L][Hkv][K, V]
  const uint8_t* rlimbs;           // R = U.H.P as 3 bf16 limbs per (layer, head, K|V), tensor-core operand layout
  int32_t lloyd;                   // 1: codes index the levels (0, a, 3 - a, 3)
  const int32_t* page_table;       // [max_seqs][maxp]
  const StepSeq* step;             // [n_seqs]
  const StepDims* dims;            // the current step's shape (device copy, uploaded with step)
  uint8_t* int2;                   // [L][max_int2_pages][Hkv][block]
  size_t int2_layer_stride;        // bytes
  __nv_bfloat16* sink_k;           // [L][max_sink_pages][Hkv][64][128]
  __nv_bfloat16* sink_v;
  size_t sink_layer_stride;        // elements
  __nv_bfloat16* ring_k;           // [L][max_seqs][Hkv][256][128]
  __nv_bfloat16* ring_v;
  size_t ring_layer_stride;        // elements
};


// Partials: one slot per BF16 pair, then one per INT2 (worker, pair) segment (at most
// nw_max + n_pairs of them): floats [hg][2] (running max in log2 units, sum) then [hg][128]
// unnormalised output.
inline int slot_floats(int hg) { return hg * (2 + kHeadDim); }
inline size_t partial_slots(const StepDims& S) { return (size_t)S.nw_max + 2 * (size_t)S.n_pairs; }
inline size_t int2_slot_offset(const StepDims& S) { return (size_t)S.n_pairs; }

// Kernel launchers (defined in the .cu files); return cudaGetLastError().
cudaError_t launch_scatter_i32(int32_t* dst, const int32_t* pairs, int n, cudaStream_t s);
size_t rlimb_bytes_per_matrix();
cudaError_t launch_build_rlimbs(const DevPool& P, uint8_t* rl, int n_mats, cudaStream_t s);
cudaError_t launch_transpose_u(const float* U, float* Ut, int n_mats, cudaStream_t s);
cudaError_t launch_demote(const DevPool& P, const StepDims& S, int layer, const void* k_new,
                          const void* v_new, cudaStream_t s);
cudaError_t launch_append(const DevPool& P, const StepDims& S, int layer, const void* k_new,
                          const void* v_new, cudaStream_t s);
cudaError_t launch_rotate_q(const DevPool& P, const StepDims& S, int layer, const void* q,
                            float* q_rot, cudaStream_t s);
cudaError_t launch_decode_int2(const DevPool& P, const StepDims& S, int layer, const float* q_rot,
                               float* partials, cudaStream_t s);
cudaError_t launch_decode_bf16(const DevPool& P, const StepDims& S, int layer, const void* q,
                               float* partials, cudaStream_t s);
cudaError_t launch_merge(const DevPool& P, const StepDims& S, int layer, const float* partials_int2,
                         const float* partials_bf16, float* out, cudaStream_t s);
cudaError_t launch_debug_rotate(const DevPool& P, int layer, int head, int kv, const void* x, int n,
                                float* out, cudaStream_t s);
cudaError_t launch_debug_read_int2(const DevPool& P, int seq, int layer, int head, int pos0, int n,
                                   uint8_t* ck, void* szk, uint8_t* cv, void* szv, cudaStream_t s);
cudaError_t launch_debug_read_bf16(const DevPool& P, int seq, int sink_page, int L, int F,
                                   int layer, int head, int pos0, int n, void* k, void* v,
                                   cudaStream_t s);

cudaError_t launch_debug_int2_scores(const DevPool& P, int seq, int layer, int head, int pos0, int n,
                                     const float* q_rot, float* out, cudaStream_t s);
cudaError_t launch_debug_timeout(uint32_t* err, cudaStream_t s);

// Largest number of INT2 decode workers (warps) resident at once for this geometry.
int decode_int2_max_workers(int hg, int ngroups, int lloyd, int num_sms);

// Load (under CUDA's lazy module loading) the kernel instances that launch_decode_int2, and
// launch_decode_bf16 + launch_merge, use for this geometry on the current device, so that a
// later launch loads nothing.
cudaError_t preload_decode_int2(int hg, int ngroups, int lloyd);
cudaError_t preload_decode_bf16_merge(int hg);

// The parts of a pool that a launcher outside the host pool code needs during a step.
struct PoolStepView {
  const DevPool* P;
  const StepDims* dims;
  int32_t num_layers;
  bool in_step, host_only;
  int device;                      // the device the pool's memory lives on
  int64_t* launch_count;
};
void pool_step_view(oscar_pool* p, PoolStepView* v);

}  // namespace oscar
