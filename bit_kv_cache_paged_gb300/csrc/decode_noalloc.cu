// oscar_decode_merge_noalloc: decode + merge of one layer with the split partials kept in a
// fixed device array that the library owns, for callers that cannot allocate device memory at
// decode time (a host runtime without a device allocator of its own, or code that must not
// allocate between steps). The kernels and launches are those of oscar_decode followed by
// oscar_merge; only the place of the scratch differs. The OSCAR write-ups have no counterpart:
// their split-K decode needs the scratch and leaves open who provides it.
#include <mutex>

#include "oscar_internal.h"

using namespace oscar;

// One array per device for the whole process, shared by every call on that device. It is never
// cleared: the merge reads only slots that the decode kernels of the same call wrote.
static __device__ __align__(256) float g_noalloc_partials[OSCAR_NOALLOC_PARTIALS_MAX_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
// Kernel geometries a call can launch: Hq / Hkv in {4, 8} x groups per row in {1, 4} x Lloyd-Max.
constexpr int kGeoms = 8;

std::mutex g_lookup_mu;
float* g_partials_addr[kMaxDevices];          // set once the lookup on that device has succeeded
bool g_preloaded[kMaxDevices][kGeoms];        // kernels of that geometry loaded on that device

int geom_index(int hg, int ngroups, int lloyd) { return (hg == 8 ? 4 : 0) + (ngroups == 4 ? 2 : 0) + (lloyd ? 1 : 0); }

// Device address of the array on `dev` (the current device), looked up with
// cudaGetSymbolAddress the first time it succeeds there; a failed lookup is not remembered, so a
// later call tries again. The first call for a kernel geometry on a device also loads the
// decode and merge kernels it launches (CUDA loads kernels lazily, on first use), so later calls
// of that geometry load nothing.
oscar_status setup_on_device(int dev, int hg, int ngroups, int lloyd, float** out) {
  if (dev < 0 || dev >= kMaxDevices) return OSCAR_EINVAL;
  std::lock_guard<std::mutex> lock(g_lookup_mu);
  if (!g_partials_addr[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_partials) != cudaSuccess || !addr) {
      (void)cudaGetLastError();
      return OSCAR_ECUDA;
    }
    g_partials_addr[dev] = static_cast<float*>(addr);
  }
  const int gi = geom_index(hg, ngroups, lloyd);
  if (!g_preloaded[dev][gi]) {
    cudaError_t e = preload_decode_int2(hg, ngroups, lloyd);
    if (e == cudaSuccess) e = preload_decode_bf16_merge(hg);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return OSCAR_ECUDA;
    }
    g_preloaded[dev][gi] = true;
  }
  *out = g_partials_addr[dev];
  return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status oscar_decode_merge_noalloc(oscar_pool* pool, int32_t layer, int32_t n_seqs,
                                                   const void* q_bf16, const float* q_rot, float* out,
                                                   void* stream) {
  if (!pool || !q_bf16 || !q_rot || !out) return OSCAR_EINVAL;
  if (((reinterpret_cast<uintptr_t>(q_bf16) | reinterpret_cast<uintptr_t>(q_rot) | reinterpret_cast<uintptr_t>(out)) & 15) != 0)
    return OSCAR_EINVAL;  // read and written in 16-byte pieces
  PoolStepView v{};
  pool_step_view(pool, &v);
  if (layer < 0 || layer >= v.num_layers) return OSCAR_EINVAL;
  if (!v.in_step) return OSCAR_ESTATE;
  if (v.host_only || n_seqs != v.dims->n_seqs) return OSCAR_EINVAL;
  const size_t need = oscar_partials_bytes(pool, n_seqs);
  if (need == 0 || need > OSCAR_NOALLOC_PARTIALS_MAX_BYTES) return OSCAR_EINVAL;
  // the array and the kernels are looked up on the current device, which must be the pool's
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return OSCAR_ECUDA;
  }
  if (dev != v.device) return OSCAR_EINVAL;
  const DevPool& P = *v.P;
  float* part = nullptr;
  const oscar_status r = setup_on_device(dev, P.hg, P.ngroups, P.lloyd, &part);
  if (r != OSCAR_OK) return r;

  const StepDims& S = *v.dims;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* pbf16 = part;
  float* pint2 = part + int2_slot_offset(S) * slot_floats(P.hg);
  cudaError_t e = cudaSuccess;
  if (S.total_units > 0) {
    e = launch_decode_int2(P, S, layer, q_rot, pint2, st);
    if (e == cudaSuccess) ++*v.launch_count;
  }
  if (e == cudaSuccess) {
    e = launch_decode_bf16(P, S, layer, q_bf16, pbf16, st);
    if (e == cudaSuccess) ++*v.launch_count;
  }
  if (e == cudaSuccess) {
    e = launch_merge(P, S, layer, pint2, pbf16, out, st);
    if (e == cudaSuccess) ++*v.launch_count;
  }
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return OSCAR_ECUDA;
  }
  return OSCAR_OK;
}
