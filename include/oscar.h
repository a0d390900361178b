/*
 * oscar.h -- C ABI of liboscar: OSCAR's mixed-precision paged KV cache and its
 * decode hot path on one NVIDIA GB300 GPU (sm_103a).
 *
 * What the library computes (sources by page title and section):
 *  - Cache zones. The first 64 tokens of a sequence (attention sinks) and the
 *    last 256 tokens stay in BF16; the history between them is stored as
 *    rotated INT2. ("oscar-2bit-kv-cache", arddev.tech, section "Аналитика";
 *    "OSCAR fra Together AI goer 2-bit KV-cache mere praktisk", snilld.dk,
 *    section "Hvad vi ved om resultaterne"; OSCAR author write-up by
 *    Zhongzhu Zhou, m.th-motor.com, serving paragraph.)
 *  - Demote. A new token enters the BF16 recent window; the oldest recent
 *    token is rotated by R = U.H.P (U: attention-aware basis per layer and KV
 *    head; H: Walsh-Hadamard; P: bit-reversal), clipped, quantised to 2 bits
 *    with a per-group scale and zero point, packed 4 codes per byte and moved
 *    to the INT2 history. (Author write-up, serving and rotation paragraphs;
 *    arddev.tech "Аналитика" for the order of the three transforms.)
 *  - Decode. An INT2 kernel unpacks codes, restores scale and zero point and
 *    accumulates in floating point; a BF16 kernel covers sink and recent; an
 *    online-softmax merge combines them. (Author write-up, serving paragraph.)
 *    Keys are compared in the rotated basis: (qR)(kR)^T = qk^T for orthogonal R.
 *
 * Readings where the pages are silent are fixed here and in the oracle:
 * row vectors (x_rot = x R), natural-order orthonormal H_128, one global 7-bit
 * bit-reversal, quant groups along head_dim after rotation, clip ratio c
 * scaling the group min and max, x_hat = code*s + z with fp16 s and z (z =
 * clipped min), codes from the fp16-rounded s and z with IEEE fp32 arithmetic
 * and round-half-even, softmax scale 1/sqrt(head_dim), GQA head h -> KV head
 * h / (Hq/Hkv).
 *
 * Conventions for every entry point:
 *  - Pointers marked "dev" are device (cudaMalloc'd / torch CUDA) addresses;
 *    "host" are host addresses. Streams are cudaStream_t passed as void*.
 *  - The caller owns every buffer it passes (q, k, v, q_rot, partials, out);
 *    the pool owns its arena contents, page tables and copies of U and clip.
 *  - Device buffers of the step calls (k_new, v_new, q, q_rot, partials, out)
 *    and of the BF16-only cache calls (rows, pages, q, partials, out) start on
 *    a 16-byte boundary, as cudaMalloc and torch allocations do; the kernels
 *    read and write them in 16-byte pieces. A call given another address
 *    returns OSCAR_EINVAL and launches nothing.
 *  - Calls that take a stream are asynchronous on it and never synchronise,
 *    except oscar_check and the debug readers (documented). Argument and
 *    capacity errors are returned at once; errors found by kernels (bad page
 *    id, non-finite scale, bounded-wait timeout) set the pool's device error
 *    word and surface from oscar_check.
 *  - No C++ exception crosses this ABI. A pool is not thread-safe: callers
 *    serialise calls on one pool.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum oscar_status {
  OSCAR_OK = 0,
  OSCAR_EINVAL = 1,    /* bad argument or unsupported configuration */
  OSCAR_ENOMEM = 2,    /* arena too small / allocation failed */
  OSCAR_EFULL = 3,     /* no free INT2 page or sink page; step rolled back */
  OSCAR_ECUDA = 4,     /* a CUDA runtime call failed */
  OSCAR_EDEVICE = 5,   /* a kernel set the device error word (see oscar_check) */
  OSCAR_ETIMEOUT = 6,  /* a kernel's bounded wait ran out (device error word) */
  OSCAR_ESTATE = 7     /* call out of order (e.g. decode before step_begin) */
} oscar_status;

/* Device error word bits (reported by oscar_check through *detail). */
#define OSCAR_DEVERR_PAGE 0x1u     /* page id out of range: nothing outside the pool is read or
                                      written; the call's outputs are not valid */
#define OSCAR_DEVERR_SCALE 0x2u    /* demote: non-finite / fp16-overflowing scale or zero */
#define OSCAR_DEVERR_TIMEOUT 0x4u  /* a bounded mbarrier wait gave up */
#define OSCAR_DEVERR_INPUT 0x8u    /* non-finite input row */

/* Config flags. */
#define OSCAR_FLAG_HOST_ONLY 0x1   /* bookkeeping only: no device memory, no launches */
#define OSCAR_FLAG_LLOYD_MAX 0x2   /* INT2 codes index a Lloyd-Max codebook (see oscar_pool_set_codebook) */

typedef struct oscar_config {
  int32_t num_layers;     /* >= 1 */
  int32_t num_q_heads;    /* Hq; Hq / Hkv must be 4 or 8 */
  int32_t num_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;       /* must be 128 */
  int32_t page_size;      /* must be 64 */
  int32_t sink_size;      /* must be 64 */
  int32_t recent_size;    /* must be 256 */
  int32_t group_size;     /* INT2 group along head_dim: 128 or 32 */
  int32_t max_seqs;       /* sequence ids are 0 .. max_seqs-1 */
  int32_t max_seq_len;    /* longest context a sequence may reach */
  int64_t max_int2_pages; /* INT2 page pool capacity; one page = 64 tokens x all layers x all KV heads */
  int32_t v_rot_absorbed; /* 1: V arrives already rotated (R_V folded into W_v / W_o); demote
                             quantises V without rotating it and merge does not un-rotate */
  int32_t flags;          /* OSCAR_FLAG_* */
} oscar_config;

typedef struct oscar_pool oscar_pool; /* opaque, library-owned */

/* Bytes of device arena a pool with this config needs (0 if the config is invalid).
 * Layout (all 256-B aligned): error word, U_K, U_V, U_V^T copies [L][Hkv][128][128] fp32,
 * clip ratios, page tables, step buffers, BF16 sink pool [L][sink pages][Hkv][64][128] x {K,V},
 * BF16 recent ring [L][max_seqs][Hkv][256][128] x {K,V}, INT2 pool
 * [L][max_int2_pages][Hkv][block], block = 4608 B (group 128) or 6144 B (group 32). */
size_t oscar_arena_bytes(const oscar_config* cfg);

/* Create a pool: the BF16 sink pool, the BF16 recent ring and the INT2 page pool of every layer,
 * with per-layer, per-KV-head rotation bases and clipping ratios (OSCAR author write-up,
 * m.th-motor.com: rotation paragraph for the per-layer, per-head rotation and clipping thresholds,
 * decode paragraph before Fig. 2 for the paged layout; "oscar-2bit-kv-cache", arddev.tech,
 * section "Как применить сегодня" for the 64-token sink and 256-token recent sizes). dev_arena: dev buffer of arena_bytes >= oscar_arena_bytes(cfg), owned by the
 * caller and kept alive until destroy; NULL with arena_bytes 0 makes the pool cudaMalloc its own.
 * U_k, U_v: dev fp32 [num_layers][num_kv_heads][128][128], U[i][k] row-major, applied as x.U
 * (columns are the basis vectors). clip_k, clip_v: dev fp32 [num_layers][num_kv_heads] clip
 * ratios. All four are copied (stream-ordered on `stream`); the caller may free them after the
 * stream reaches this point. With OSCAR_FLAG_HOST_ONLY all device arguments must be NULL/0.
 * Returns OSCAR_EINVAL for an unsupported config, OSCAR_ENOMEM for a short arena. */
oscar_status oscar_pool_create(const oscar_config* cfg, void* dev_arena, size_t arena_bytes,
                               const float* U_k, const float* U_v, const float* clip_k,
                               const float* clip_v, void* stream, oscar_pool** out);

/* Destroy a pool (frees what the pool allocated; not the caller's arena). NULL is a no-op.
 * The caller must make sure no work on the pool is still running. */
oscar_status oscar_pool_destroy(oscar_pool* pool);

/* Lloyd-Max codebook (pools created with OSCAR_FLAG_LLOYD_MAX). The author write-up's closing
 * paragraph says the newest OSCAR codebase brings a Lloyd-Max codebook into the attention-aware
 * rotation. Here: the group frame of the uniform quantiser is kept (lo = c*min, hi = c*max,
 * fp16 s = (hi - lo)/3 and z = lo, same storage), and the four levels of a code are
 * (0, a, 3 - a, 3) in units of s above z instead of (0, 1, 2, 3): x_hat = z + s * level[code].
 * Encoding picks the nearest level of u = (x - z)/s (fp32): code = [u > a/2] + [u >= 1.5] +
 * [u > 3 - a/2]. One a per (layer, KV head, K|V); a = 1 (the default) is the uniform quantiser.
 * a_host: host fp32 [num_layers][num_kv_heads][2] (K then V), each in [0.5, 1.45]. Only before the
 * pool's first oscar_step_begin (OSCAR_ESTATE afterwards); synchronous on `stream`. */
oscar_status oscar_pool_set_codebook(oscar_pool* pool, const float* a_host, void* stream);

/* Fit a for (layer, kv_head, kv: 0 = K, 1 = V) by Lloyd's algorithm on calibration rows: rotate
 * rows_bf16 (dev [n][128]) with the pool's R, take each group's frame as the demote does, and
 * iterate nearest-level cells and centroids (the level-(3 - a) cell enters mirrored, 3 - u; the
 * end levels stay fixed; a kept in [0.05, 1.45]; at most `iters` rounds). scratch: dev fp32
 * [n][128]. *a_out receives a (host). Synchronous on `stream`. */
oscar_status oscar_fit_codebook(oscar_pool* pool, int32_t layer, int32_t kv_head, int32_t kv,
                                const void* rows_bf16, int32_t n, float* scratch, int32_t iters,
                                float* a_out, void* stream);

/* Register sequence seq_id with length 0. With share_from >= 0 the new sequence instead starts
 * at length shared_tokens and shares share_from's sink page and the INT2 pages covering positions
 * [64, shared_tokens) (a prefix-cache hit through shared page-table entries; OSCAR author
 * write-up, serving paragraph and Fig. 6 paragraph). shared_tokens must be 64 + a multiple of 64
 * and already demoted in share_from. The sharer's recent window starts empty and refills. */
oscar_status oscar_seq_add(oscar_pool* pool, int32_t seq_id, int32_t share_from,
                           int32_t shared_tokens);

/* Unregister a sequence and release its page references. Host-only bookkeeping: the caller
 * must not remove a sequence that work still in flight on the GPU reads or writes. */
oscar_status oscar_seq_remove(oscar_pool* pool, int32_t seq_id);

/* Start a step: sequence seq_ids[i] (host int32 [n_seqs], distinct, registered) receives
 * n_new[i] >= 0 new tokens (host int32 [n_seqs]; 1 for decode, more for prefill). Advances the
 * host bookkeeping, allocates INT2 pages for the tokens this step demotes, and uploads the step
 * description and page-table changes on `stream`. Batch index i of every later call in the step
 * refers to seq_ids[i]. On OSCAR_EFULL nothing changes. */
oscar_status oscar_step_begin(oscar_pool* pool, const int32_t* seq_ids, const int32_t* n_new,
                              int32_t n_seqs, void* stream);

/* For one layer of the current step: demote the tokens that leave the recent window (rotate,
 * clip, quantise, pack into INT2 pages; fused in one kernel), then append the new tokens to the
 * sink or the recent ring. k_new, v_new: dev bf16 [sum(n_new)][num_kv_heads][128], rows of batch
 * index i first (in seq_ids order), positions ascending, each 16-byte aligned (else OSCAR_EINVAL).
 * Tokens of a long append that would be demoted within the same step go straight from k_new/v_new
 * to INT2. */
oscar_status oscar_append_and_demote(oscar_pool* pool, int32_t layer, const void* k_new_bf16,
                                     const void* v_new_bf16, void* stream);

/* Keys are stored rotated, so the INT2 scores take the rotated query: (q R)(k R)^T = q k^T for
 * the orthogonal R_K, whose basis comes from the query covariance Q^T Q (OSCAR author write-up,
 * rotation paragraph; "OSCAR fra Together AI ...", snilld.dk, section "Hvad OSCAR gør
 * anderledes"). q_rot = q . R_K[layer, kv head of h] for every query head: q dev bf16 [n_seqs][num_q_heads][128]
 * -> q_rot dev fp32, same shape. */
oscar_status oscar_rotate_q(oscar_pool* pool, int32_t layer, const void* q_bf16, float* q_rot,
                            void* stream);

/* Decode attention partials for one layer of the current step (after append_and_demote):
 * the split-K INT2 kernel over the history pages (scores from q_rot) and the BF16 kernel over
 * sink + recent (scores from raw q). The INT2 kernel unpacks the codes, restores scale and zero
 * point and accumulates in floating point; the BF16 kernel covers sink and recent (OSCAR author
 * write-up, decode paragraph before Fig. 2). partials: dev buffer of oscar_partials_bytes(pool, n_seqs)
 * bytes (caller-owned scratch; contents undefined after the call except to oscar_merge). */
oscar_status oscar_decode(oscar_pool* pool, int32_t layer, const void* q_bf16, const float* q_rot,
                          void* partials, void* stream);

/* Merge the partials of oscar_decode into the attention output: LSE-merge the INT2 splits,
 * un-rotate them by R_V^T (unless v_rot_absorbed), LSE-merge with the BF16 part (the online
 * softmax merge of the OSCAR author write-up, decode paragraph before Fig. 2; the value rotation
 * folded into the projection weights instead: "oscar-2bit-kv-cache", section "Аналитика").
 * out: dev fp32 [n_seqs][num_q_heads][128]. */
oscar_status oscar_merge(oscar_pool* pool, int32_t layer, const void* partials, float* out,
                         void* stream);

/* One decode step of every layer as a single CUDA graph launch on `stream` (the fused kernel
 * pipeline the OSCAR decode path runs in: OSCAR author write-up, m.th-motor.com, decode paragraph
 * before Fig. 2, which names SGLang's fused kernel pipeline; the graph is this library's reading of
 * it). For layer l = 0 .. num_layers-1, in order:
 * oscar_append_and_demote, oscar_rotate_q, oscar_decode, oscar_merge, with
 *   k_new, v_new: dev bf16 [Σn_new][num_kv_heads][128] at base + l * kv_layer_stride (bytes; bases
 *                 16-byte aligned and the stride a multiple of 16, else OSCAR_EINVAL),
 *   q:            dev bf16 [n_seqs][num_q_heads][128] at base + l * q_layer_stride,
 *   out:          dev fp32 [n_seqs][num_q_heads][128] at base + l * out_layer_stride,
 *   q_rot, partials: scratch shared by the layers (sizes as for oscar_rotate_q, oscar_partials_bytes).
 * Same results as those calls made one by one. The pool keeps the instantiated graph: while the
 * step's shape (batch, new, demoted and appended rows, whether there are INT2 units) and every
 * pointer and stride stay the same, a call only launches it (the INT2 unit and worker counts,
 * which grow whenever a sequence starts a new INT2 page, are read by the kernels from device
 * memory); otherwise the call first records the launches on a private stream (nothing runs then)
 * and instantiates or updates the graph, which costs host time (oscar_graph_captures counts it). Kernel timing (oscar_timing_enable) does not apply to graph launches; they
 * count in oscar_launch_count. Errors as for the four calls; OSCAR_ECUDA if capture fails. */
oscar_status oscar_step_graph(oscar_pool* pool, const void* k_new_bf16, const void* v_new_bf16,
                              size_t kv_layer_stride, const void* q_bf16, size_t q_layer_stride,
                              float* q_rot, void* partials, float* out, size_t out_layer_stride,
                              void* stream);

/* Bytes of partials scratch that oscar_decode needs for the current step (n_seqs must equal the
 * step's batch): a bound that depends only on the batch size and the pool, so one buffer serves
 * every step of a batch. Returns 0 outside a step or on a mismatch. */
size_t oscar_partials_bytes(const oscar_pool* pool, int32_t n_seqs);

/* ---- Decode + merge with library-owned scratch ----------------------------------------------
 * No counterpart in the OSCAR write-ups: the split-K decode there needs scratch for its per-split
 * partials but says nothing about who provides it. This entry point is for callers that cannot
 * allocate device memory when they decode: a host runtime that has no device allocator of its
 * own, or code that must not allocate between steps. The partials live in one fixed device array
 * of OSCAR_NOALLOC_PARTIALS_MAX_BYTES per device inside liboscar.
 *
 * Computes exactly what oscar_decode followed by oscar_merge computes (same kernels, same
 * launches, same order on `stream`): out dev fp32 [n_seqs][num_q_heads][128]; q, q_rot as for
 * oscar_decode; n_seqs must equal the current step's batch.
 *
 * Size limit: when oscar_partials_bytes(pool, n_seqs) exceeds OSCAR_NOALLOC_PARTIALS_MAX_BYTES
 * (16 MiB: at 4 query heads per KV head about 8 000 partial slots, enough for batch 32 x 8 KV
 * heads with every SM busy), the call returns OSCAR_EINVAL and launches nothing; use oscar_decode
 * with a buffer of your own then.
 *
 * Set-up: the call runs on the current device, which must be the device the pool was created on
 * (OSCAR_EINVAL otherwise). The first call on a device looks up the array's device address there
 * (cudaGetSymbolAddress); the first call for each pool geometry (query heads per KV head, group
 * size, codebook) on a device also makes CUDA load the decode and merge kernels that geometry
 * launches, which CUDA otherwise loads lazily at their first launch. Make those first calls before
 * any stream capture. A failed set-up is not remembered: the next call tries again. After set-up,
 * calls allocate nothing: no device or host memory, no events, no module loads.
 *
 * Sharing: all calls on one device, from every pool, stream and thread of the process, use the
 * same array. Calls whose kernels overlap in time race on it and corrupt each other's outputs;
 * order them (one stream, or an event between them). Nothing in the array has to start at zero:
 * the merge reads only slots that the decode kernels of the same call wrote, so a call clears
 * nothing.
 *
 * Errors: OSCAR_EINVAL (bad argument, batch mismatch, host-only pool, too large, current device
 * not the pool's), OSCAR_ESTATE
 * (outside a step), OSCAR_ECUDA (set-up or launch failed). Launches count in oscar_launch_count;
 * they are not timed by oscar_timing_enable. */
#define OSCAR_NOALLOC_PARTIALS_MAX_BYTES ((size_t)16 << 20)
oscar_status oscar_decode_merge_noalloc(oscar_pool* pool, int32_t layer, int32_t n_seqs,
                                        const void* q_bf16, const float* q_rot, float* out,
                                        void* stream);

/* Synchronise `stream`, then read and clear the device error word. Returns OSCAR_OK,
 * OSCAR_ETIMEOUT (timeout bit set), OSCAR_EDEVICE (other bits) or OSCAR_ECUDA. *detail (may be
 * NULL) receives the OSCAR_DEVERR_* bits. */
oscar_status oscar_check(oscar_pool* pool, void* stream, uint32_t* detail);

/* Current length, demote frontier (first recent position) and INT2 page count of a sequence. */
oscar_status oscar_seq_info(const oscar_pool* pool, int32_t seq_id, int32_t* length,
                            int32_t* frontier, int32_t* int2_pages);

/* Pool occupancy: INT2 pages in use / free, sink pages in use, and stored bytes per token in each
 * zone summed over layers and KV heads (BF16 token: 512 B per layer-head; INT2 token: 72 B at
 * group 128, 96 B at group 32). */
typedef struct oscar_pool_stats {
  int64_t int2_pages_used, int2_pages_free;
  int32_t sink_pages_used, seqs_active;
  int64_t bf16_bytes_per_token, int2_bytes_per_token;
} oscar_pool_stats;
oscar_status oscar_pool_get_stats(const oscar_pool* pool, oscar_pool_stats* out);

/* ---- BF16-only paged cache (the comparison cache of the same shape) -----------------------
 * Every token of every sequence in BF16 pages: the cache the OSCAR write-ups measure their decode
 * speedups against (OSCAR author write-up, m.th-motor.com, serving and Fig. 6 paragraphs). No pool:
 * the caller owns the pages, page table and lengths.
 *   pages: dev bf16, K and V in separate buffers of [n_pages_total][num_kv_heads][64 tokens][128],
 *     token t's 16-B chunk c stored at byte t*256 + ((c ^ (t & 7)) * 16) of its 16 KB page (the
 *     pool's BF16 page swizzle). Token slots past a sequence's length must hold finite values
 *     (zero-initialise the buffers).
 *   page_table: dev int32 [n_seqs][max_pages_per_seq]; page j of sequence i holds positions
 *     64j .. 64j+63. lengths: dev int32 [n_seqs], each in [1, max_len].
 * Out-of-range page ids set OSCAR_DEVERR_PAGE in *err (dev uint32, caller-owned) and the page is
 * replaced by page 0; bounded waits that give up set OSCAR_DEVERR_TIMEOUT. */

/* Scratch bytes of oscar_bf16_decode (0 for an unsupported shape: Hq / Hkv must be 4 or 8). */
size_t oscar_bf16_partials_bytes(int32_t num_q_heads, int32_t num_kv_heads, int32_t n_seqs,
                                 int32_t max_len);

/* Write rows [n][num_kv_heads][128] (dev bf16) of positions pos0 .. pos0+n-1 of one sequence into
 * its pages; page_table_row: dev int32 row of that sequence. Asynchronous on `stream`. */
oscar_status oscar_bf16_pack(const void* rows_bf16, int32_t n, int32_t pos0, int32_t num_kv_heads,
                             const int32_t* page_table_row, int64_t n_pages_total, void* pages,
                             uint32_t* err, void* stream);

/* Decode attention of q (dev bf16 [n_seqs][num_q_heads][128], GQA h -> h / (Hq/Hkv)) over each
 * sequence's BF16 tokens [0, length): split-K over chunks of 32 pages, then an LSE merge into
 * out (dev fp32 [n_seqs][num_q_heads][128]). partials: dev scratch of
 * oscar_bf16_partials_bytes(...) bytes. Asynchronous on `stream`; OSCAR_EINVAL for bad arguments. */
oscar_status oscar_bf16_decode(int32_t num_q_heads, int32_t num_kv_heads, int32_t n_seqs,
                               int32_t max_len, const void* k_pages, const void* v_pages,
                               int64_t n_pages_total, const int32_t* page_table,
                               int32_t max_pages_per_seq, const int32_t* lengths,
                               const void* q_bf16, void* partials, size_t partials_bytes, float* out,
                               uint32_t* err, void* stream);

/* ---- Parity hooks (synchronous on `stream`; for tests, not for the hot path) -------------- */

/* Rotate n bf16 rows (dev [n][128]) by the demote path's fp32 rotation for (layer, kv_head,
 * kv: 0 = K, 1 = V) and write the fp32 rotated rows in position order (dev [n][128]). With
 * v_rot_absorbed and kv = 1 the rows are only converted to fp32. */
oscar_status oscar_debug_rotate_rows(oscar_pool* pool, int32_t layer, int32_t kv_head, int32_t kv,
                                     const void* x_bf16, int32_t n, float* out_f32, void* stream);

/* Read INT2 tokens [pos0, pos0+n) of (seq, layer, kv_head) in canonical layout: codes_k/codes_v
 * dev uint8 [n][32] (byte j>>2, bits 2*(j&3) hold code j), sz_k/sz_v dev fp16 [n][128/G][2]
 * (scale, zero). Positions must lie in [64, frontier). */
oscar_status oscar_debug_read_int2(oscar_pool* pool, int32_t seq_id, int32_t layer,
                                   int32_t kv_head, int32_t pos0, int32_t n, void* codes_k,
                                   void* sz_k, void* codes_v, void* sz_v, void* stream);

/* Diagnostic scores of INT2 tokens [pos0, pos0+n) of (seq, layer, kv_head): for each of the KV
 * head's hg = Hq/Hkv query heads, q_rot[h] . k_hat(token) in fp32, with k_hat = code*s + z the
 * dequantised rotated key (no 1/sqrt(d) scale). q_rot: dev fp32 [hg][128] (rows of oscar_rotate_q's
 * output); out: dev fp32 [hg][n]. Positions must lie in [64, frontier). Used by the quantisation
 * ablation diagnostics (attention-score KL against a BF16 cache). */
oscar_status oscar_debug_int2_scores(oscar_pool* pool, int32_t seq_id, int32_t layer, int32_t kv_head,
                                     const float* q_rot, int32_t pos0, int32_t n, float* out,
                                     void* stream);

/* Read BF16 tokens [pos0, pos0+n) of (seq, layer, kv_head) from the sink page or the recent ring:
 * k_out, v_out dev bf16 [n][128]. Positions must lie in the sink or in [frontier, length). */
oscar_status oscar_debug_read_bf16(oscar_pool* pool, int32_t seq_id, int32_t layer,
                                   int32_t kv_head, int32_t pos0, int32_t n, void* k_out,
                                   void* v_out, void* stream);

/* Fault injection on the host: write `value` into the device page-table entry of INT2 page `page`
 * (0-based, below the sequence's page count) of sequence seq_id, leaving the host's bookkeeping as
 * it is. An out-of-range value (negative, or >= max_int2_pages) must make the kernels that read
 * the entry set OSCAR_DEVERR_PAGE and substitute an in-bounds page (decode) or skip the write
 * (demote); nothing outside the pool is read or written. Synchronous on `stream`. */
oscar_status oscar_debug_set_page_entry(oscar_pool* pool, int32_t seq_id, int32_t page, int32_t value,
                                        void* stream);

/* Rewrite the device page-table row of seq_id from the host's bookkeeping (undoes
 * oscar_debug_set_page_entry). Synchronous on `stream`. */
oscar_status oscar_debug_restore_page_table(oscar_pool* pool, int32_t seq_id, void* stream);

/* Failure-detection self test: launch one CTA that waits on an mbarrier whose transaction count
 * nothing ever completes. Its bounded wait gives up after ~2^30 SM cycles (about half a second),
 * sets OSCAR_DEVERR_TIMEOUT in the device error word and returns; no copy is in flight and nothing
 * faults. Asynchronous on `stream`; read the result with oscar_check (expects OSCAR_ETIMEOUT). */
oscar_status oscar_debug_timeout_selftest(oscar_pool* pool, void* stream);

/* ---- Kernel timing (CUDA events on the launch stream) ------------------------------------- */

#define OSCAR_KERNEL_DEMOTE 0
#define OSCAR_KERNEL_APPEND 1
#define OSCAR_KERNEL_ROTATE_Q 2
#define OSCAR_KERNEL_DECODE_INT2 3
#define OSCAR_KERNEL_DECODE_BF16 4
#define OSCAR_KERNEL_MERGE 5
#define OSCAR_KERNEL_COUNT 6

/* Event timing of launches: bit k of kernel_mask times every launch of kernel kind k
 * (OSCAR_KERNEL_*), e.g. 1 << OSCAR_KERNEL_DECODE_INT2; OSCAR_TIMING_ALL times all kinds; 0
 * disables. Each timed launch is bracketed by two events on its stream. Clears the accumulators. */
#define OSCAR_TIMING_ALL ((1 << OSCAR_KERNEL_COUNT) - 1)
oscar_status oscar_timing_enable(oscar_pool* pool, int32_t kernel_mask);

/* Synchronise the recorded events and return per-kernel total milliseconds and launch counts
 * (host arrays of OSCAR_KERNEL_COUNT entries; either may be NULL). */
oscar_status oscar_timing_read(oscar_pool* pool, double* total_ms, int64_t* launches);

/* Number of this library's kernel launches since the pool was created (all kinds). */
int64_t oscar_launch_count(const oscar_pool* pool);

/* Number of times oscar_step_graph recorded (captured) the step graph since the pool was created.
 * A new INT2 page for some sequence does not force a new recording: the unit and worker counts
 * live in device memory; a change of batch, of new / demoted / appended rows, or of a pointer or
 * stride does. */
int64_t oscar_graph_captures(const oscar_pool* pool);

/* INT2 decode workers of the current step: the step's (sequence, KV head, page) units are split
 * into this many contiguous ranges (split-K segments; each (sequence, KV head) is covered by
 * about workers / (batch x KV heads) of them). 0 outside a step. */
int32_t oscar_step_int2_workers(const oscar_pool* pool);

/* Static description of the library build: "liboscar <version> sm_103a". */
const char* oscar_version(void);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_H_ */
