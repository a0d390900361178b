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

std::mutex g_lookup_mu;
bool g_looked_up[kMaxDevices];
cudaError_t g_lookup_err[kMaxDevices];
float* g_partials_addr[kMaxDevices];

// Device address of the array on the current device. cudaGetSymbolAddress runs once per device,
// with that device current (the first call there also loads this library's kernels on it); its
// result, success or failure, is kept for every later call.
oscar_status partials_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return OSCAR_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return OSCAR_EINVAL;
  std::lock_guard<std::mutex> lock(g_lookup_mu);
  if (!g_looked_up[dev]) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_noalloc_partials);
    if (e != cudaSuccess) (void)cudaGetLastError();
    g_lookup_err[dev] = e;
    g_partials_addr[dev] = e == cudaSuccess ? static_cast<float*>(addr) : nullptr;
    g_looked_up[dev] = true;
  }
  if (g_lookup_err[dev] != cudaSuccess || !g_partials_addr[dev]) return OSCAR_ECUDA;
  *out = g_partials_addr[dev];
  return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status oscar_decode_merge_noalloc(oscar_pool* pool, int32_t layer, int32_t n_seqs,
                                                   const void* q_bf16, const float* q_rot, float* out,
                                                   void* stream) {
  if (!pool || !q_bf16 || !q_rot || !out) return OSCAR_EINVAL;
  PoolStepView v{};
  pool_step_view(pool, &v);
  if (layer < 0 || layer >= v.num_layers) return OSCAR_EINVAL;
  if (!v.in_step) return OSCAR_ESTATE;
  if (v.host_only || n_seqs != v.dims->n_seqs) return OSCAR_EINVAL;
  const size_t need = oscar_partials_bytes(pool, n_seqs);
  if (need == 0 || need > OSCAR_NOALLOC_PARTIALS_MAX_BYTES) return OSCAR_EINVAL;
  float* part = nullptr;
  const oscar_status r = partials_on_current_device(&part);
  if (r != OSCAR_OK) return r;

  const DevPool& P = *v.P;
  const StepDims& S = *v.dims;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* pint2 = part;
  float* pbf16 = part + ((size_t)S.nw + S.n_pairs) * slot_floats(P.hg);
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
