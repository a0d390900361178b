// liboscar host side: the C ABI, the mixed-precision paged KV pool (page allocator with
// reference counts for shared prefixes, sequence table, per-step work description), launches
// and event timing.
//
// Cache zones follow the OSCAR serving design (first 64 tokens and last 256 tokens in BF16,
// history in INT2 pages that stay compatible with paged KV and prefix caching: OSCAR author
// write-up, m.th-motor.com, serving paragraph; "oscar-2bit-kv-cache", arddev.tech, section
// "Аналитика"). A sequence of length L has sink [0, min(64, L)), INT2 history [64, F) and a
// recent window [F, L), with the demote frontier F = max(64, shared_prefix, L - 256).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "oscar_internal.h"

using namespace oscar;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t err, uk, uv, utv, clip_k, clip_v, cb, rlimb, page_table, step, scatter, sink_k, sink_v, ring_k,
      ring_v, int2, total;
  size_t int2_layer_stride, sink_layer_stride_el, ring_layer_stride_el;
  int32_t maxp, max_sink_pages, block_bytes;
};

bool config_ok(const oscar_config* c) {
  if (!c) return false;
  if (c->num_layers < 1 || c->num_kv_heads < 1 || c->num_q_heads < 1) return false;
  if (c->num_q_heads % c->num_kv_heads) return false;
  const int hg = c->num_q_heads / c->num_kv_heads;
  if (hg != 4 && hg != 8) return false;
  if (c->head_dim != kHeadDim || c->page_size != kPage || c->sink_size != kSink ||
      c->recent_size != kRecent)
    return false;
  if (c->group_size != 128 && c->group_size != 32) return false;
  if (c->max_seqs < 1 || c->max_seqs > (1 << 20)) return false;
  if (c->max_seq_len < 1) return false;
  if (c->max_int2_pages < 1 || c->max_int2_pages > (int64_t)1 << 31) return false;
  if (c->v_rot_absorbed != 0 && c->v_rot_absorbed != 1) return false;
  if (c->flags & ~(OSCAR_FLAG_HOST_ONLY | OSCAR_FLAG_LLOYD_MAX)) return false;
  return true;
}

Layout make_layout(const oscar_config* c) {
  Layout Lt{};
  const size_t L = c->num_layers, H = c->num_kv_heads, D = kHeadDim;
  Lt.maxp = std::max(1, (c->max_seq_len - kSink + kPage - 1) / kPage);
  Lt.max_sink_pages = c->max_seqs;
  Lt.block_bytes = int2_block_bytes(c->group_size);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  Lt.err = take(64);
  Lt.uk = take(L * H * D * D * 4);
  Lt.uv = take(L * H * D * D * 4);
  Lt.utv = take(L * H * D * D * 4);
  Lt.clip_k = take(L * H * 4);
  Lt.clip_v = take(L * H * 4);
  Lt.cb = take(L * H * 2 * 4);
  Lt.rlimb = take(L * H * 2 * rlimb_bytes_per_matrix());
  Lt.page_table = take((size_t)c->max_seqs * Lt.maxp * 4);
  Lt.step = take(sizeof(StepDims) + (size_t)c->max_seqs * sizeof(StepSeq));  // dims, then the batch
  Lt.scatter = take((size_t)c->max_seqs * Lt.maxp * 8);
  Lt.sink_layer_stride_el = (size_t)Lt.max_sink_pages * H * kPage * D;
  Lt.sink_k = take(L * Lt.sink_layer_stride_el * 2);
  Lt.sink_v = take(L * Lt.sink_layer_stride_el * 2);
  Lt.ring_layer_stride_el = (size_t)c->max_seqs * H * kRecent * D;
  Lt.ring_k = take(L * Lt.ring_layer_stride_el * 2);
  Lt.ring_v = take(L * Lt.ring_layer_stride_el * 2);
  Lt.int2_layer_stride = (size_t)c->max_int2_pages * H * Lt.block_bytes;
  Lt.int2 = take(L * Lt.int2_layer_stride);
  Lt.total = off;
  return Lt;
}

struct Seq {
  bool active = false;
  int32_t L = 0, S = 0, F = kSink;
  int32_t sink_page = -1;
  std::vector<int32_t> pages;
  size_t pt_clean = 0;  // page-table entries already on the device
};

}  // namespace

struct oscar_pool {
  oscar_config cfg{};
  bool host_only = false;
  int device = 0;
  int num_sms = 152;
  int max_workers = 152 * 12;
  int hg = 4;
  Layout lay{};
  uint8_t* arena = nullptr;
  bool owns_arena = false;
  DevPool P{};
  std::vector<Seq> seqs;
  std::vector<int32_t> int2_free, int2_ref, sink_free, sink_ref;
  // current step
  bool in_step = false;
  bool stepped = false;  // a step has begun since creation (the codebook is fixed from then on)
  std::vector<StepSeq> step;
  StepDims dims{};
  // pinned staging for step uploads (double-buffered)
  uint8_t* pinned[2] = {nullptr, nullptr};
  size_t pinned_bytes = 0;
  cudaEvent_t pinned_ev[2] = {nullptr, nullptr};
  int pinned_cur = 0;
  // timing
  int32_t timing = 0;  // kernel-kind bitmask
  struct Pending {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_free;
  double total_ms[OSCAR_KERNEL_COUNT] = {};
  int64_t launches[OSCAR_KERNEL_COUNT] = {};
  int64_t launch_count = 0;
  // decode-step graph (oscar_step_graph): instantiated graph, the step shape and pointers it was
  // captured with, and its kernel count
  struct GraphKey {
    StepDims dims;
    const void *k_new, *v_new, *q;
    const void *q_rot, *partials, *out;
    size_t kv_stride, q_stride, out_stride;
  };
  cudaStream_t capture_stream = nullptr;
  cudaStream_t capture_side = nullptr;      // second branch of the captured step (rotate_q)
  cudaEvent_t capture_fork = nullptr, capture_join = nullptr;
  // the BF16 decode's branch when it runs beside the INT2 decode (a step with few sequences):
  // a stream of its own for direct calls (a captured step uses capture_side), and its events
  cudaStream_t dec_side = nullptr;
  cudaEvent_t dec_fork = nullptr, dec_join = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  GraphKey graph_key{};
  bool capturing = false;
  int64_t graph_kernels = 0;
  int64_t graph_captures = 0;  // times the step graph was recorded
};

namespace {

// INT2 decode workers per (sequence, KV head), on average, at most: bounds the merge's work
constexpr int kMaxPartialsPerPair = 64;

oscar_status cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return OSCAR_OK;
  (void)cudaGetLastError();
  return OSCAR_ECUDA;
}

// Brackets one launch with events when timing is on.
template <typename F>
oscar_status timed_launch(oscar_pool* p, int kind, cudaStream_t s, F&& f) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool timed = !p->capturing && ((p->timing >> kind) & 1);
  if (timed) {
    if (!p->ev_free.empty()) {
      a = p->ev_free.back().first;
      b = p->ev_free.back().second;
      p->ev_free.pop_back();
    } else {
      if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return OSCAR_ECUDA;
    }
    cudaEventRecord(a, s);
  }
  const cudaError_t e = f();
  if (timed) {
    cudaEventRecord(b, s);
    p->pending.push_back({kind, a, b});
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (p->capturing)
    p->graph_kernels++;
  else
    p->launch_count++;
  return OSCAR_OK;
}

bool seq_ok(const oscar_pool* p, int32_t id) {
  return id >= 0 && id < p->cfg.max_seqs && p->seqs[id].active;
}

int32_t frontier(int32_t L, int32_t S) { return std::max({(int32_t)kSink, S, L - (int32_t)kRecent}); }

int32_t pages_for(int32_t F) { return F > kSink ? (F - kSink + kPage - 1) / kPage : 0; }

void release_seq_pages(oscar_pool* p, Seq& s) {
  for (int32_t pg : s.pages) {
    if (--p->int2_ref[pg] == 0) p->int2_free.push_back(pg);
  }
  s.pages.clear();
  if (s.sink_page >= 0 && --p->sink_ref[s.sink_page] == 0) p->sink_free.push_back(s.sink_page);
  s.sink_page = -1;
}

// Upload page-table entries [pt_clean, pages.size()) of one sequence synchronously (debug path).
oscar_status flush_seq_table(oscar_pool* p, int32_t id, cudaStream_t st) {
  Seq& s = p->seqs[id];
  if (p->host_only || s.pt_clean >= s.pages.size()) return OSCAR_OK;
  int32_t* dst = reinterpret_cast<int32_t*>(p->arena + p->lay.page_table) + (size_t)id * p->lay.maxp + s.pt_clean;
  const size_t n = s.pages.size() - s.pt_clean;
  if (cudaMemcpyAsync(dst, s.pages.data() + s.pt_clean, n * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return OSCAR_ECUDA;
  s.pt_clean = s.pages.size();
  return OSCAR_OK;
}

// Group frame of fp32 rotated rows, as the demote computes it: lo = c*min, hi = c*max,
// s = fp16((hi - lo) / 3), z = fp16(lo), u = (x - z) / s (every step one IEEE fp32 operation; this
// file is compiled without floating-point contraction), then Lloyd's algorithm for the interior
// level a of the codebook (0, a, 3 - a, 3): nearest-level cells, centroid of the level-a cell
// together with the mirror images 3 - u of the level-(3 - a) cell, a kept in [0.05, 1.45].
double lloyd_fit_rows(const float* r, int64_t n, int G, float clip, int iters) {
  std::vector<double> u;
  u.reserve((size_t)n * kHeadDim);
  for (int64_t i = 0; i < n; ++i) {
    for (int g0 = 0; g0 < kHeadDim; g0 += G) {
      const float* x = r + (size_t)i * kHeadDim + g0;
      float mn = x[0], mx = x[0];
      for (int j = 1; j < G; ++j) {
        mn = std::min(mn, x[j]);
        mx = std::max(mx, x[j]);
      }
      const float lo = clip * mn, hi = clip * mx;
      const float s32 = (hi - lo) / 3.0f;
      const float sf = __half2float(__float2half_rn(s32)), zf = __half2float(__float2half_rn(lo));
      for (int j = 0; j < G; ++j) {
        float v = 0.f;
        if (sf != 0.f) {
          const float d = x[j] - zf;
          v = d / sf;
          if (!std::isfinite(v)) v = 0.f;
        }
        u.push_back((double)v);
      }
    }
  }
  double a = 1.0;
  for (int it = 0; it < iters; ++it) {
    const double t0 = a / 2.0, t2 = 3.0 - a / 2.0;
    double sum = 0.0;
    int64_t cnt = 0;
    for (const double v : u) {
      if (v > t0 && v < 1.5) {
        sum += v;
        ++cnt;
      } else if (v >= 1.5 && v <= t2) {
        sum += 3.0 - v;
        ++cnt;
      }
    }
    if (cnt == 0) break;
    const double next = std::min(1.45, std::max(0.05, sum / (double)cnt));
    const bool done = std::fabs(next - a) < 1e-9;
    a = next;
    if (done) break;
  }
  return a;
}

}  // namespace

void oscar::pool_step_view(oscar_pool* p, PoolStepView* v) {
  v->P = &p->P;
  v->dims = &p->dims;
  v->num_layers = p->cfg.num_layers;
  v->in_step = p->in_step;
  v->host_only = p->host_only;
  v->device = p->device;
  v->launch_count = &p->launch_count;
}

extern "C" {

const char* oscar_version(void) { return "liboscar 0.1 sm_103a"; }

size_t oscar_arena_bytes(const oscar_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return make_layout(cfg).total;
}

oscar_status oscar_pool_create(const oscar_config* cfg, void* dev_arena, size_t arena_bytes,
                               const float* U_k, const float* U_v, const float* clip_k,
                               const float* clip_v, void* stream, oscar_pool** out) {
  if (!out) return OSCAR_EINVAL;
  *out = nullptr;
  if (!config_ok(cfg)) return OSCAR_EINVAL;
  oscar_pool* p = new (std::nothrow) oscar_pool();
  if (!p) return OSCAR_ENOMEM;
  p->cfg = *cfg;
  p->host_only = (cfg->flags & OSCAR_FLAG_HOST_ONLY) != 0;
  p->hg = cfg->num_q_heads / cfg->num_kv_heads;
  p->lay = make_layout(cfg);
  p->seqs.resize(cfg->max_seqs);
  p->int2_ref.assign((size_t)cfg->max_int2_pages, 0);
  p->int2_free.reserve((size_t)cfg->max_int2_pages);
  for (int64_t i = cfg->max_int2_pages - 1; i >= 0; --i) p->int2_free.push_back((int32_t)i);
  p->sink_ref.assign(p->lay.max_sink_pages, 0);
  for (int32_t i = p->lay.max_sink_pages - 1; i >= 0; --i) p->sink_free.push_back(i);
  p->step.reserve(cfg->max_seqs);
  if (p->host_only) {
    if (dev_arena || arena_bytes || U_k || U_v || clip_k || clip_v) {
      delete p;
      return OSCAR_EINVAL;
    }
    p->max_workers = p->num_sms * 12;
    *out = p;
    return OSCAR_OK;
  }
  if (!U_k || !U_v || !clip_k || !clip_v) {
    delete p;
    return OSCAR_EINVAL;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return OSCAR_ECUDA;
  }
  if (dev_arena) {
    if (arena_bytes < p->lay.total || (reinterpret_cast<uintptr_t>(dev_arena) % kAlign) != 0) {
      delete p;
      return OSCAR_ENOMEM;
    }
    p->arena = static_cast<uint8_t*>(dev_arena);
  } else {
    if (arena_bytes != 0) {
      delete p;
      return OSCAR_EINVAL;
    }
    if (cudaMalloc(&p->arena, p->lay.total) != cudaSuccess) {
      (void)cudaGetLastError();
      delete p;
      return OSCAR_ENOMEM;
    }
    p->owns_arena = true;
  }
  const Layout& Lt = p->lay;
  const size_t nmat = (size_t)cfg->num_layers * cfg->num_kv_heads;
  DevPool& P = p->P;
  P.num_layers = cfg->num_layers;
  P.Hq = cfg->num_q_heads;
  P.Hkv = cfg->num_kv_heads;
  P.G = cfg->group_size;
  P.ngroups = kHeadDim / cfg->group_size;
  P.hg = p->hg;
  P.max_seqs = cfg->max_seqs;
  P.maxp = Lt.maxp;
  P.max_int2_pages = cfg->max_int2_pages;
  P.max_sink_pages = Lt.max_sink_pages;
  P.absorbed = cfg->v_rot_absorbed;
  P.block_bytes = Lt.block_bytes;
  P.num_sms = p->num_sms;
  P.err = reinterpret_cast<uint32_t*>(p->arena + Lt.err);
  P.Uk = reinterpret_cast<const float*>(p->arena + Lt.uk);
  P.Uv = reinterpret_cast<const float*>(p->arena + Lt.uv);
  P.Utv = reinterpret_cast<const float*>(p->arena + Lt.utv);
  P.clip_k = reinterpret_cast<const float*>(p->arena + Lt.clip_k);
  P.clip_v = reinterpret_cast<const float*>(p->arena + Lt.clip_v);
  P.cb_a = reinterpret_cast<const float*>(p->arena + Lt.cb);
  P.rlimbs = p->arena + Lt.rlimb;
  P.lloyd = (cfg->flags & OSCAR_FLAG_LLOYD_MAX) ? 1 : 0;
  P.page_table = reinterpret_cast<const int32_t*>(p->arena + Lt.page_table);
  P.dims = reinterpret_cast<const StepDims*>(p->arena + Lt.step);
  P.step = reinterpret_cast<const StepSeq*>(p->arena + Lt.step + sizeof(StepDims));
  P.int2 = p->arena + Lt.int2;
  P.int2_layer_stride = Lt.int2_layer_stride;
  P.sink_k = reinterpret_cast<__nv_bfloat16*>(p->arena + Lt.sink_k);
  P.sink_v = reinterpret_cast<__nv_bfloat16*>(p->arena + Lt.sink_v);
  P.sink_layer_stride = Lt.sink_layer_stride_el;
  P.ring_k = reinterpret_cast<__nv_bfloat16*>(p->arena + Lt.ring_k);
  P.ring_v = reinterpret_cast<__nv_bfloat16*>(p->arena + Lt.ring_v);
  P.ring_layer_stride = Lt.ring_layer_stride_el;

  cudaError_t e = cudaSuccess;
  const size_t ubytes = nmat * kHeadDim * kHeadDim * 4;
  if (e == cudaSuccess) e = cudaMemsetAsync(p->arena + Lt.err, 0, 64, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->arena + Lt.uk, U_k, ubytes, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->arena + Lt.uv, U_v, ubytes, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->arena + Lt.clip_k, clip_k, nmat * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p->arena + Lt.clip_v, clip_v, nmat * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->arena + Lt.page_table, 0xFF, (size_t)cfg->max_seqs * Lt.maxp * 4, st);
  // BF16 sink pages and recent rings start zeroed: the decode multiplies the values of slots that
  // hold no live token by a zero weight, which must not meet a NaN or Inf bit pattern
  if (e == cudaSuccess) e = cudaMemsetAsync(p->arena + Lt.sink_k, 0, Lt.int2 - Lt.sink_k, st);
  if (e == cudaSuccess) e = launch_transpose_u(P.Uv, const_cast<float*>(P.Utv), (int)nmat, st);
  if (e == cudaSuccess) e = launch_build_rlimbs(P, p->arena + Lt.rlimb, (int)nmat * 2, st);
  if (e == cudaSuccess) {  // codebook interior level a = 1 (the uniform levels) until set
    const std::vector<float> ones(nmat * 2, 1.0f);
    e = cudaMemcpyAsync(p->arena + Lt.cb, ones.data(), nmat * 2 * 4, cudaMemcpyHostToDevice, st);
  }
  p->pinned_bytes = align_up(sizeof(StepDims) + (size_t)cfg->max_seqs * sizeof(StepSeq)) + (size_t)cfg->max_seqs * Lt.maxp * 8;
  for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
    e = cudaMallocHost(reinterpret_cast<void**>(&p->pinned[b]), p->pinned_bytes);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->pinned_ev[b], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) p->max_workers = decode_int2_max_workers(p->hg, P.ngroups, P.lloyd, p->num_sms);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    oscar_pool_destroy(p);
    (void)cudaGetLastError();
    return OSCAR_ECUDA;
  }
  *out = p;
  return OSCAR_OK;
}

oscar_status oscar_pool_destroy(oscar_pool* p) {
  if (!p) return OSCAR_OK;
  if (!p->host_only) {
    for (auto& q : p->pending) {
      cudaEventDestroy(q.a);
      cudaEventDestroy(q.b);
    }
    for (auto& q : p->ev_free) {
      cudaEventDestroy(q.first);
      cudaEventDestroy(q.second);
    }
    for (int b = 0; b < 2; ++b) {
      if (p->pinned_ev[b]) {
        cudaEventSynchronize(p->pinned_ev[b]);
        cudaEventDestroy(p->pinned_ev[b]);
      }
      if (p->pinned[b]) cudaFreeHost(p->pinned[b]);
    }
    if (p->graph_exec) cudaGraphExecDestroy(p->graph_exec);
    if (p->capture_stream) cudaStreamDestroy(p->capture_stream);
    if (p->capture_side) cudaStreamDestroy(p->capture_side);
    if (p->capture_fork) cudaEventDestroy(p->capture_fork);
    if (p->capture_join) cudaEventDestroy(p->capture_join);
    if (p->dec_side) cudaStreamDestroy(p->dec_side);
    if (p->dec_fork) cudaEventDestroy(p->dec_fork);
    if (p->dec_join) cudaEventDestroy(p->dec_join);
    if (p->owns_arena && p->arena) cudaFree(p->arena);
  }
  delete p;
  return OSCAR_OK;
}

oscar_status oscar_seq_add(oscar_pool* p, int32_t id, int32_t share_from, int32_t shared_tokens) {
  if (!p || id < 0 || id >= p->cfg.max_seqs || p->seqs[id].active) return OSCAR_EINVAL;
  Seq s;
  if (share_from >= 0) {
    if (!seq_ok(p, share_from) || share_from == id) return OSCAR_EINVAL;
    const Seq& src = p->seqs[share_from];
    if (shared_tokens < kSink || (shared_tokens - kSink) % kPage != 0 || src.F < shared_tokens ||
        shared_tokens > p->cfg.max_seq_len)
      return OSCAR_EINVAL;
    const size_t np = (size_t)(shared_tokens - kSink) / kPage;
    s.pages.assign(src.pages.begin(), src.pages.begin() + np);
    for (int32_t pg : s.pages) p->int2_ref[pg]++;
    s.sink_page = src.sink_page;
    p->sink_ref[s.sink_page]++;
    s.L = shared_tokens;
    s.S = shared_tokens;
    s.F = frontier(s.L, s.S);
  } else {
    if (share_from != -1 || shared_tokens != 0) return OSCAR_EINVAL;
    if (p->sink_free.empty()) return OSCAR_EFULL;
    s.sink_page = p->sink_free.back();
    p->sink_free.pop_back();
    p->sink_ref[s.sink_page] = 1;
  }
  s.active = true;
  s.pt_clean = 0;
  p->seqs[id] = std::move(s);
  return OSCAR_OK;
}

oscar_status oscar_seq_remove(oscar_pool* p, int32_t id) {
  if (!p || !seq_ok(p, id)) return OSCAR_EINVAL;
  // Freed pages are handed out again only by a later oscar_step_begin, so the rest of the
  // current step may still read them.
  release_seq_pages(p, p->seqs[id]);
  p->seqs[id] = Seq();
  return OSCAR_OK;
}

oscar_status oscar_step_begin(oscar_pool* p, const int32_t* seq_ids, const int32_t* n_new,
                              int32_t n_seqs, void* stream) {
  if (!p || !seq_ids || !n_new || n_seqs < 1 || n_seqs > p->cfg.max_seqs) return OSCAR_EINVAL;
  const int Hkv = p->cfg.num_kv_heads;
  std::vector<char> seen(p->cfg.max_seqs, 0);
  int64_t need_pages = 0, tot_new = 0, tot_dem = 0, tot_app = 0, tot_units = 0;
  for (int i = 0; i < n_seqs; ++i) {
    const int32_t id = seq_ids[i];
    if (!seq_ok(p, id) || seen[id] || n_new[i] < 0) return OSCAR_EINVAL;
    seen[id] = 1;
    const Seq& s = p->seqs[id];
    const int64_t Ln = (int64_t)s.L + n_new[i];
    if (Ln > p->cfg.max_seq_len) return OSCAR_EINVAL;
    const int32_t Fn = frontier((int32_t)Ln, s.S);
    need_pages += std::max<int64_t>(0, pages_for(Fn) - (int64_t)s.pages.size());
    tot_new += n_new[i];
  }
  if (tot_new > (int64_t)1 << 30) return OSCAR_EINVAL;
  if (need_pages > (int64_t)p->int2_free.size()) return OSCAR_EFULL;

  // commit: allocate pages, build the step description
  p->step.assign(n_seqs, StepSeq{});
  std::vector<int32_t> scatter;
  for (int i = 0; i < n_seqs; ++i) {
    Seq& s = p->seqs[seq_ids[i]];
    StepSeq& st = p->step[i];
    st.seq_id = seq_ids[i];
    st.L_old = s.L;
    st.L_new = s.L + n_new[i];
    st.F_old = s.F;
    st.F_new = frontier(st.L_new, s.S);
    st.sink_page = s.sink_page;
    const int32_t np = pages_for(st.F_new);
    while ((int32_t)s.pages.size() < np) {
      const int32_t pg = p->int2_free.back();
      p->int2_free.pop_back();
      p->int2_ref[pg] = 1;
      s.pages.push_back(pg);
    }
    st.n_pages = np;
    for (size_t k = s.pt_clean; k < s.pages.size(); ++k) {
      scatter.push_back((int32_t)((size_t)st.seq_id * p->lay.maxp + k));
      scatter.push_back(s.pages[k]);
    }
    s.pt_clean = s.pages.size();
  }
  int64_t in_off = 0;
  for (int i = 0; i < n_seqs; ++i) {
    StepSeq& st = p->step[i];
    st.in_offset = (int32_t)in_off;
    in_off += n_new[i];
    st.dem_offset = (int32_t)tot_dem;
    tot_dem += st.F_new - st.F_old;
    st.app_offset = (int32_t)tot_app;
    const int32_t n_sink_new = std::max(0, std::min((int32_t)kSink, st.L_new) - st.L_old);
    const int32_t n_ring_new = st.L_new - std::max(st.F_new, st.L_old);
    tot_app += n_sink_new + std::max(0, n_ring_new);
    st.unit_offset = (int32_t)tot_units;
    tot_units += (int64_t)Hkv * st.n_pages;
  }
  if (tot_units > (int64_t)1 << 30 || tot_dem > (int64_t)1 << 30) return OSCAR_EINVAL;
  for (int i = 0; i < n_seqs; ++i) {
    Seq& s = p->seqs[seq_ids[i]];
    s.L = p->step[i].L_new;
    s.F = p->step[i].F_new;
  }
  StepDims& D = p->dims;
  std::memset(&D, 0, sizeof(D));
  D.n_seqs = n_seqs;
  D.total_new = (int32_t)tot_new;
  D.total_dem = (int32_t)tot_dem;
  D.total_app = (int32_t)tot_app;
  D.total_units = (int32_t)tot_units;
  D.n_pairs = n_seqs * Hkv;
  D.nw_max = (int32_t)std::max<int64_t>(1, std::min<int64_t>(p->max_workers, (int64_t)n_seqs * Hkv * kMaxPartialsPerPair));
  if (tot_units > 0) {
    // at least kMinUnitsPerWorker pages per worker, and at most kMaxPartialsPerPair partials per
    // (sequence, KV head) on average, which bounds the merge's work when a step has few rows
    const int64_t want = std::min<int64_t>((tot_units + kMinUnitsPerWorker - 1) / kMinUnitsPerWorker,
                                           (int64_t)n_seqs * Hkv * kMaxPartialsPerPair);
    D.nw = (int32_t)std::max<int64_t>(1, std::min<int64_t>(p->max_workers, want));
  } else {
    D.nw = 0;
  }
  p->in_step = true;
  p->stepped = true;
  if (p->host_only) return OSCAR_OK;

  // upload: step description + page-table scatter list through pinned staging
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int b = p->pinned_cur;
  p->pinned_cur ^= 1;
  if (cudaEventSynchronize(p->pinned_ev[b]) != cudaSuccess) return OSCAR_ECUDA;
  const size_t step_bytes = sizeof(StepDims) + (size_t)n_seqs * sizeof(StepSeq);
  std::memcpy(p->pinned[b], &p->dims, sizeof(StepDims));
  std::memcpy(p->pinned[b] + sizeof(StepDims), p->step.data(), (size_t)n_seqs * sizeof(StepSeq));
  const size_t sc_off = align_up(step_bytes);
  const size_t sc_bytes = scatter.size() * 4;
  if (sc_off + sc_bytes > p->pinned_bytes) return OSCAR_EINVAL;
  if (sc_bytes) std::memcpy(p->pinned[b] + sc_off, scatter.data(), sc_bytes);
  cudaError_t e = cudaMemcpyAsync(p->arena + p->lay.step, p->pinned[b], step_bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess && sc_bytes) {
    e = cudaMemcpyAsync(p->arena + p->lay.scatter, p->pinned[b] + sc_off, sc_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) {
      e = launch_scatter_i32(reinterpret_cast<int32_t*>(p->arena + p->lay.page_table),
                             reinterpret_cast<const int32_t*>(p->arena + p->lay.scatter),
                             (int)(scatter.size() / 2), st);
      p->launch_count++;
    }
  }
  if (e == cudaSuccess) e = cudaEventRecord(p->pinned_ev[b], st);
  return cuda_fail(e);
}

// A device pointer the kernels read in 16-byte chunks (null passes: nothing is read then).
static bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

oscar_status oscar_append_and_demote(oscar_pool* p, int32_t layer, const void* k_new,
                                     const void* v_new, void* stream) {
  if (!p || layer < 0 || layer >= p->cfg.num_layers) return OSCAR_EINVAL;
  if (!p->in_step) return OSCAR_ESTATE;
  if (p->host_only) return OSCAR_EINVAL;
  if (p->dims.total_new > 0 && (!k_new || !v_new)) return OSCAR_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return OSCAR_EINVAL;  // the kernels copy 16-byte chunks
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  oscar_status r = OSCAR_OK;
  if (p->dims.total_dem > 0)
    r = timed_launch(p, OSCAR_KERNEL_DEMOTE, st, [&] { return launch_demote(p->P, p->dims, layer, k_new, v_new, st); });
  if (r == OSCAR_OK && p->dims.total_app > 0)
    r = timed_launch(p, OSCAR_KERNEL_APPEND, st, [&] { return launch_append(p->P, p->dims, layer, k_new, v_new, st); });
  return r;
}

oscar_status oscar_rotate_q(oscar_pool* p, int32_t layer, const void* q, float* q_rot, void* stream) {
  if (!p || layer < 0 || layer >= p->cfg.num_layers || !q || !q_rot) return OSCAR_EINVAL;
  if (!aligned16(q) || !aligned16(q_rot)) return OSCAR_EINVAL;
  if (!p->in_step) return OSCAR_ESTATE;
  if (p->host_only) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return timed_launch(p, OSCAR_KERNEL_ROTATE_Q, st, [&] { return launch_rotate_q(p->P, p->dims, layer, q, q_rot, st); });
}

size_t oscar_partials_bytes(const oscar_pool* p, int32_t n_seqs) {
  if (!p || !p->in_step || n_seqs != p->dims.n_seqs) return 0;
  return partial_slots(p->dims) * (size_t)slot_floats(p->hg) * 4;
}

oscar_status oscar_decode(oscar_pool* p, int32_t layer, const void* q, const float* q_rot,
                          void* partials, void* stream) {
  if (!p || layer < 0 || layer >= p->cfg.num_layers || !q || !q_rot || !partials) return OSCAR_EINVAL;
  if (!aligned16(q) || !aligned16(q_rot) || !aligned16(partials)) return OSCAR_EINVAL;
  if (!p->in_step) return OSCAR_ESTATE;
  if (p->host_only) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* pbf16 = static_cast<float*>(partials);
  float* pint2 = pbf16 + int2_slot_offset(p->dims) * slot_floats(p->hg);
  oscar_status r = OSCAR_OK;
  // With few sequences the INT2 grid (4 workers per CTA) and the BF16 grid (a CTA per pair) fit on
  // the SMs side by side: the BF16 kernel then runs on a second branch, beside the INT2 kernel
  // (they write disjoint partials), and the branch joins before the call returns on `stream`.
  const int64_t int2_ctas = p->dims.total_units > 0 ? ((int64_t)p->dims.nw_max + 3) / 4 : 0;
  const bool beside = int2_ctas > 0 && int2_ctas + p->dims.n_pairs <= p->num_sms;
  cudaStream_t bs = st;
  if (beside) {
    if (p->capturing) {
      bs = p->capture_side;
    } else {
      if (!p->dec_side && cudaStreamCreateWithFlags(&p->dec_side, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_fail(cudaErrorUnknown);
      bs = p->dec_side;
    }
    if (!p->dec_fork && cudaEventCreateWithFlags(&p->dec_fork, cudaEventDisableTiming) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    if (!p->dec_join && cudaEventCreateWithFlags(&p->dec_join, cudaEventDisableTiming) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    cudaError_t ce = cudaEventRecord(p->dec_fork, st);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(bs, p->dec_fork, 0);
    if (ce != cudaSuccess) return cuda_fail(ce);
    r = timed_launch(p, OSCAR_KERNEL_DECODE_BF16, bs, [&] { return launch_decode_bf16(p->P, p->dims, layer, q, pbf16, bs); });
    ce = cudaEventRecord(p->dec_join, bs);
    if (r == OSCAR_OK && ce != cudaSuccess) r = cuda_fail(ce);
  }
  if (r == OSCAR_OK && p->dims.total_units > 0)
    r = timed_launch(p, OSCAR_KERNEL_DECODE_INT2, st, [&] { return launch_decode_int2(p->P, p->dims, layer, q_rot, pint2, st); });
  if (beside) {
    const cudaError_t ce = cudaStreamWaitEvent(st, p->dec_join, 0);  // the branch joins even after an error
    if (r == OSCAR_OK && ce != cudaSuccess) r = cuda_fail(ce);
  } else if (r == OSCAR_OK) {
    r = timed_launch(p, OSCAR_KERNEL_DECODE_BF16, st, [&] { return launch_decode_bf16(p->P, p->dims, layer, q, pbf16, st); });
  }
  return r;
}

oscar_status oscar_merge(oscar_pool* p, int32_t layer, const void* partials, float* out, void* stream) {
  if (!p || layer < 0 || layer >= p->cfg.num_layers || !partials || !out) return OSCAR_EINVAL;
  if (!aligned16(partials) || !aligned16(out)) return OSCAR_EINVAL;
  if (!p->in_step) return OSCAR_ESTATE;
  if (p->host_only) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* pbf16 = static_cast<const float*>(partials);
  const float* pint2 = pbf16 + int2_slot_offset(p->dims) * slot_floats(p->hg);
  return timed_launch(p, OSCAR_KERNEL_MERGE, st, [&] { return launch_merge(p->P, p->dims, layer, pint2, pbf16, out, st); });
}

oscar_status oscar_step_graph(oscar_pool* p, const void* k_new, const void* v_new, size_t kv_layer_stride,
                              const void* q, size_t q_layer_stride, float* q_rot, void* partials, float* out,
                              size_t out_layer_stride, void* stream) {
  if (!p || !q || !q_rot || !partials || !out) return OSCAR_EINVAL;
  if (!p->in_step) return OSCAR_ESTATE;
  if (p->host_only || p->capturing) return OSCAR_EINVAL;
  if (p->dims.total_new > 0 && (!k_new || !v_new)) return OSCAR_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || kv_layer_stride % 16 != 0) return OSCAR_EINVAL;
  if (!aligned16(q) || !aligned16(q_rot) || !aligned16(partials) || !aligned16(out) || q_layer_stride % 16 != 0 ||
      out_layer_stride % 16 != 0)
    return OSCAR_EINVAL;
  oscar_pool::GraphKey key;
  std::memset(&key, 0, sizeof(key));  // compared bytewise, padding included
  // the INT2 unit and worker counts are read by the kernels from device memory, so they are not
  // part of the key: only whether the step has INT2 units at all (the decode launch is recorded
  // or not)
  key.dims = p->dims;
  key.dims.total_units = 0;
  key.dims.nw = 0;
  key.dims.pad[0] = p->dims.total_units > 0 ? 1 : 0;
  key.k_new = k_new;
  key.v_new = v_new;
  key.q = q;
  key.q_rot = q_rot;
  key.partials = partials;
  key.out = out;
  key.kv_stride = kv_layer_stride;
  key.q_stride = q_layer_stride;
  key.out_stride = out_layer_stride;
  if (!p->graph_exec || std::memcmp(&key, &p->graph_key, sizeof(key)) != 0) {
    // capture the step's launches on a private stream (nothing runs), then instantiate or update
    if (!p->capture_stream && cudaStreamCreateWithFlags(&p->capture_stream, cudaStreamNonBlocking) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    if (!p->capture_side && cudaStreamCreateWithFlags(&p->capture_side, cudaStreamNonBlocking) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    if (!p->capture_fork && cudaEventCreateWithFlags(&p->capture_fork, cudaEventDisableTiming) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    if (!p->capture_join && cudaEventCreateWithFlags(&p->capture_join, cudaEventDisableTiming) != cudaSuccess)
      return cuda_fail(cudaErrorUnknown);
    cudaStream_t cs = p->capture_stream, side = p->capture_side;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    p->capturing = true;
    p->graph_kernels = 0;
    oscar_status r = OSCAR_OK;
    const char* kb = static_cast<const char*>(k_new);
    const char* vb = static_cast<const char*>(v_new);
    const char* qb = static_cast<const char*>(q);
    char* ob = reinterpret_cast<char*>(out);
    // per layer, rotate_q (which reads only q) runs beside append + demote on a second branch
    // and joins before the decode; q_rot and the partials are reused by the next layer only after
    // this layer's merge, which the next fork follows
    for (int32_t l = 0; l < p->cfg.num_layers && r == OSCAR_OK; ++l) {
      const size_t ko = (size_t)l * kv_layer_stride;
      const void* ql = qb + (size_t)l * q_layer_stride;
      cudaError_t ce = cudaEventRecord(p->capture_fork, cs);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(side, p->capture_fork, 0);
      if (ce != cudaSuccess) r = cuda_fail(ce);
      if (r == OSCAR_OK) r = oscar_rotate_q(p, l, ql, q_rot, side);
      if (r == OSCAR_OK) {
        ce = cudaEventRecord(p->capture_join, side);
        if (ce != cudaSuccess) r = cuda_fail(ce);
      }
      if (r == OSCAR_OK) r = oscar_append_and_demote(p, l, kb ? kb + ko : nullptr, vb ? vb + ko : nullptr, cs);
      if (r == OSCAR_OK) {
        ce = cudaStreamWaitEvent(cs, p->capture_join, 0);
        if (ce != cudaSuccess) r = cuda_fail(ce);
      }
      if (r == OSCAR_OK) r = oscar_decode(p, l, ql, q_rot, partials, cs);
      if (r == OSCAR_OK) r = oscar_merge(p, l, partials, reinterpret_cast<float*>(ob + (size_t)l * out_layer_stride), cs);
    }
    p->capturing = false;
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(cs, &g);
    if (r != OSCAR_OK || e != cudaSuccess || !g) {
      if (g) cudaGraphDestroy(g);
      (void)cudaGetLastError();
      return r != OSCAR_OK ? r : OSCAR_ECUDA;
    }
    if (p->graph_exec) {
      cudaGraphExecUpdateResultInfo info;
      if (cudaGraphExecUpdate(p->graph_exec, g, &info) != cudaSuccess) {
        (void)cudaGetLastError();
        cudaGraphExecDestroy(p->graph_exec);
        p->graph_exec = nullptr;
      }
    }
    cudaError_t ei = cudaSuccess;
    if (!p->graph_exec) ei = cudaGraphInstantiate(&p->graph_exec, g, 0);
    cudaGraphDestroy(g);
    if (ei != cudaSuccess) {
      p->graph_exec = nullptr;
      return cuda_fail(ei);
    }
    std::memcpy(&p->graph_key, &key, sizeof(key));
    p->graph_captures++;
  }
  const cudaError_t e = cudaGraphLaunch(p->graph_exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  p->launch_count += p->graph_kernels;
  return OSCAR_OK;
}

oscar_status oscar_pool_set_codebook(oscar_pool* p, const float* a_host, void* stream) {
  if (!p || !a_host || p->host_only || !(p->cfg.flags & OSCAR_FLAG_LLOYD_MAX)) return OSCAR_EINVAL;
  if (p->stepped) return OSCAR_ESTATE;
  const size_t n = (size_t)p->cfg.num_layers * p->cfg.num_kv_heads * 2;
  for (size_t i = 0; i < n; ++i)
    if (!(a_host[i] >= kLloydMinA && a_host[i] <= kLloydMaxA)) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(p->arena + p->lay.cb, a_host, n * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown);
  return OSCAR_OK;
}

oscar_status oscar_fit_codebook(oscar_pool* p, int32_t layer, int32_t kv_head, int32_t kv, const void* rows,
                                int32_t n, float* scratch, int32_t iters, float* a_out, void* stream) {
  if (!p || p->host_only || layer < 0 || layer >= p->cfg.num_layers || kv_head < 0 ||
      kv_head >= p->cfg.num_kv_heads || (kv != 0 && kv != 1) || !rows || n < 1 || !scratch || iters < 1 || !a_out)
    return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<float> r((size_t)n * kHeadDim);
  float clip = 0.f;
  const size_t ci = (size_t)layer * p->cfg.num_kv_heads + kv_head;
  cudaError_t e = launch_debug_rotate(p->P, layer, kv_head, kv, rows, n, scratch, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(r.data(), scratch, r.size() * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&clip, (kv == 0 ? p->P.clip_k : p->P.clip_v) + ci, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e);
  *a_out = (float)lloyd_fit_rows(r.data(), n, p->cfg.group_size, clip, iters);
  return OSCAR_OK;
}

oscar_status oscar_check(oscar_pool* p, void* stream, uint32_t* detail) {
  if (detail) *detail = 0;
  if (!p) return OSCAR_EINVAL;
  if (p->host_only) return OSCAR_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
  uint32_t w = 0;
  if (cudaMemcpy(&w, p->arena + p->lay.err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
  if (w && cudaMemset(p->arena + p->lay.err, 0, 4) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
  if (detail) *detail = w;
  if (w & OSCAR_DEVERR_TIMEOUT) return OSCAR_ETIMEOUT;
  return w ? OSCAR_EDEVICE : OSCAR_OK;
}

oscar_status oscar_seq_info(const oscar_pool* p, int32_t id, int32_t* length, int32_t* fr, int32_t* np) {
  if (!p || !seq_ok(p, id)) return OSCAR_EINVAL;
  const Seq& s = p->seqs[id];
  if (length) *length = s.L;
  if (fr) *fr = s.F;
  if (np) *np = (int32_t)s.pages.size();
  return OSCAR_OK;
}

oscar_status oscar_pool_get_stats(const oscar_pool* p, oscar_pool_stats* o) {
  if (!p || !o) return OSCAR_EINVAL;
  o->int2_pages_free = (int64_t)p->int2_free.size();
  o->int2_pages_used = p->cfg.max_int2_pages - o->int2_pages_free;
  o->sink_pages_used = p->lay.max_sink_pages - (int32_t)p->sink_free.size();
  int32_t act = 0;
  for (const Seq& s : p->seqs) act += s.active ? 1 : 0;
  o->seqs_active = act;
  const int64_t LH = (int64_t)p->cfg.num_layers * p->cfg.num_kv_heads;
  o->bf16_bytes_per_token = LH * 2 * kHeadDim * 2;
  o->int2_bytes_per_token = LH * (p->lay.block_bytes / kPage);
  return OSCAR_OK;
}

oscar_status oscar_debug_rotate_rows(oscar_pool* p, int32_t layer, int32_t head, int32_t kv,
                                     const void* x, int32_t n, float* out, void* stream) {
  if (!p || p->host_only || layer < 0 || layer >= p->cfg.num_layers || head < 0 ||
      head >= p->cfg.num_kv_heads || (kv != 0 && kv != 1) || n < 0 || (n > 0 && (!x || !out)))
    return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_debug_rotate(p->P, layer, head, kv, x, n, out, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_fail(e);
}

oscar_status oscar_debug_read_int2(oscar_pool* p, int32_t id, int32_t layer, int32_t head, int32_t pos0,
                                   int32_t n, void* ck, void* szk, void* cv, void* szv, void* stream) {
  if (!p || p->host_only || !seq_ok(p, id) || layer < 0 || layer >= p->cfg.num_layers || head < 0 ||
      head >= p->cfg.num_kv_heads || n < 0)
    return OSCAR_EINVAL;
  const Seq& s = p->seqs[id];
  if (n > 0 && (pos0 < kSink || pos0 + n > s.F || !ck || !szk || !cv || !szv)) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  oscar_status r = flush_seq_table(p, id, st);
  if (r != OSCAR_OK) return r;
  cudaError_t e = launch_debug_read_int2(p->P, id, layer, head, pos0, n, static_cast<uint8_t*>(ck), szk,
                                         static_cast<uint8_t*>(cv), szv, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_fail(e);
}

oscar_status oscar_debug_int2_scores(oscar_pool* p, int32_t id, int32_t layer, int32_t head, const float* q_rot,
                                     int32_t pos0, int32_t n, float* out, void* stream) {
  if (!p || p->host_only || !seq_ok(p, id) || layer < 0 || layer >= p->cfg.num_layers || head < 0 ||
      head >= p->cfg.num_kv_heads || n < 0)
    return OSCAR_EINVAL;
  const Seq& s = p->seqs[id];
  if (n > 0 && (pos0 < kSink || pos0 + n > s.F || !q_rot || !out)) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  oscar_status r = flush_seq_table(p, id, st);
  if (r != OSCAR_OK) return r;
  cudaError_t e = launch_debug_int2_scores(p->P, id, layer, head, pos0, n, q_rot, out, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_fail(e);
}

oscar_status oscar_debug_read_bf16(oscar_pool* p, int32_t id, int32_t layer, int32_t head, int32_t pos0,
                                   int32_t n, void* k, void* v, void* stream) {
  if (!p || p->host_only || !seq_ok(p, id) || layer < 0 || layer >= p->cfg.num_layers || head < 0 ||
      head >= p->cfg.num_kv_heads || n < 0)
    return OSCAR_EINVAL;
  const Seq& s = p->seqs[id];
  for (int32_t q = pos0; q < pos0 + n; ++q) {
    const bool in_sink = q >= 0 && q < std::min((int32_t)kSink, s.L);
    const bool in_recent = q >= s.F && q < s.L;
    if (!in_sink && !in_recent) return OSCAR_EINVAL;
  }
  if (n > 0 && (!k || !v)) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_debug_read_bf16(p->P, id, s.sink_page, s.L, s.F, layer, head, pos0, n, k, v, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return cuda_fail(e);
}

oscar_status oscar_debug_set_page_entry(oscar_pool* p, int32_t id, int32_t page, int32_t value, void* stream) {
  if (!p || p->host_only || !seq_ok(p, id)) return OSCAR_EINVAL;
  const Seq& s = p->seqs[id];
  if (page < 0 || page >= (int32_t)s.pages.size()) return OSCAR_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  oscar_status r = flush_seq_table(p, id, st);
  if (r != OSCAR_OK) return r;
  int32_t* dst = reinterpret_cast<int32_t*>(p->arena + p->lay.page_table) + (size_t)id * p->lay.maxp + page;
  if (cudaMemcpyAsync(dst, &value, 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown);
  return OSCAR_OK;
}

oscar_status oscar_debug_restore_page_table(oscar_pool* p, int32_t id, void* stream) {
  if (!p || p->host_only || !seq_ok(p, id)) return OSCAR_EINVAL;
  Seq& s = p->seqs[id];
  if (s.pages.empty()) return OSCAR_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* dst = reinterpret_cast<int32_t*>(p->arena + p->lay.page_table) + (size_t)id * p->lay.maxp;
  if (cudaMemcpyAsync(dst, s.pages.data(), s.pages.size() * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return cuda_fail(cudaErrorUnknown);
  s.pt_clean = s.pages.size();
  return OSCAR_OK;
}

oscar_status oscar_debug_timeout_selftest(oscar_pool* p, void* stream) {
  if (!p || p->host_only) return OSCAR_EINVAL;
  return cuda_fail(launch_debug_timeout(p->P.err, static_cast<cudaStream_t>(stream)));
}

oscar_status oscar_timing_enable(oscar_pool* p, int32_t kernel_mask) {
  if (!p || kernel_mask < 0 || kernel_mask > OSCAR_TIMING_ALL) return OSCAR_EINVAL;
  if (p->host_only) return kernel_mask ? OSCAR_EINVAL : OSCAR_OK;
  for (auto& q : p->pending) {
    cudaEventSynchronize(q.b);
    p->ev_free.push_back({q.a, q.b});
  }
  p->pending.clear();
  for (int k = 0; k < OSCAR_KERNEL_COUNT; ++k) {
    p->total_ms[k] = 0;
    p->launches[k] = 0;
  }
  p->timing = kernel_mask;
  return OSCAR_OK;
}

oscar_status oscar_timing_read(oscar_pool* p, double* total_ms, int64_t* launches) {
  if (!p) return OSCAR_EINVAL;
  for (auto& q : p->pending) {
    if (cudaEventSynchronize(q.b) != cudaSuccess) return cuda_fail(cudaErrorUnknown);
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, q.a, q.b) == cudaSuccess) {
      p->total_ms[q.kind] += ms;
      p->launches[q.kind] += 1;
    }
    p->ev_free.push_back({q.a, q.b});
  }
  p->pending.clear();
  for (int k = 0; k < OSCAR_KERNEL_COUNT; ++k) {
    if (total_ms) total_ms[k] = p->total_ms[k];
    if (launches) launches[k] = p->launches[k];
  }
  return OSCAR_OK;
}

int64_t oscar_launch_count(const oscar_pool* p) { return p ? p->launch_count : 0; }

int64_t oscar_graph_captures(const oscar_pool* p) { return p ? p->graph_captures : 0; }

int32_t oscar_step_int2_workers(const oscar_pool* p) { return (p && p->in_step) ? p->dims.nw : 0; }

}  // extern "C"
