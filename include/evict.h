/*
 * evict.h — C ABI of libevict: per-block KV-cache token eviction on GB300.
 *
 * One handle = one attention layer's cache ("single-layer, no coordinator",
 * stated on all three pages: "Q-Filters — Query-Agnostic Projection
 * Eviction" §Usage, "L2Norm — Intrinsic Key-Norm Eviction" §Usage,
 * "CurDKV-adapted — Value-Aware Leverage-Score Eviction" §Usage).
 * Each update absorbs one block of m tokens per (batch, KV head), scores it,
 * appends it to the kept set and, over budget, keeps the protected top-k in
 * temporal order (the pages' §How it works sections).
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers unless the name ends in _host.
 *  - Tensors are dense, row-major, innermost dimension last:
 *      K, V blocks        [batch, n_kv_heads, m, head_dim]   (bf16 or fp32)
 *      positions          [batch, m] int32 (shared by the heads of a row)
 *      filters            [n_kv_heads, head_dim] fp32
 *  - Work is enqueued on the handle's CUDA stream and is asynchronous;
 *    caller-owned inputs must stay valid until the stream passes the call.
 *    Update calls never allocate, never synchronise the host and never read
 *    device memory back, so they may be captured in a CUDA graph.
 *  - Every function returns an evict_status (0 = success). On failure a
 *    message is available from evict_last_error() (thread-local) and the
 *    cache state is unchanged, except for EVICT_ECUDA / EVICT_EDEVICE which
 *    leave it undefined.
 *  - Asynchronous device errors surface at the next call that checks
 *    (evict_sync, evict_stats with sync, calibration).
 */
#ifndef EVICT_H
#define EVICT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum evict_status {
  EVICT_OK = 0,
  EVICT_EINVAL = 1,   /* invalid argument or configuration */
  EVICT_ELIMIT = 2,   /* size above a compiled bound: raised, never truncated */
  EVICT_ECUDA = 3,    /* a CUDA runtime call failed */
  EVICT_EDEVICE = 4,  /* a kernel reported an error through the device error word */
  EVICT_ENUM = 5      /* numerically degenerate input (calibration) */
} evict_status;

typedef enum evict_method {
  EVICT_KNORM = 0,     /* "L2Norm — Intrinsic Key-Norm Eviction", §How it works */
  EVICT_QFILTERS = 1,  /* "Q-Filters — Query-Agnostic Projection Eviction", §How it works */
  EVICT_CURDKV = 2,    /* "CurDKV-adapted — Value-Aware Leverage-Score Eviction", §How it works */
  EVICT_H2O = 3        /* H2O-adapted: cumulative proxy-attention mass, the softmax of CurDKV's
                          step 1 ("CurDKV-adapted", §How it works step 1; a new token starts
                          from exactly 0, §The honesty crux item 4). Per block: query t (the
                          incoming key k+t) attends rows i <= k+t with scale 1/sqrt(D); row i
                          gains the weights of the queries after it (a new row not its own
                          query's weight); kept rows add this to their cumulative score, new
                          rows start from it; the budget highest are kept. bf16 only. */
} evict_method;

typedef enum evict_dtype {
  EVICT_BF16 = 0,
  EVICT_FP32 = 1       /* KNorm and Q-Filters only (CurDKV and H2O store bf16) */
} evict_dtype;

/* Compiled bounds (EVICT_ELIMIT above them). */
#define EVICT_HEAD_DIM 128          /* head_dim must equal this */
#define EVICT_MAX_SELECT_ROWS 49152 /* kept + incoming rows per (b,h) in one call */

typedef struct evict_config {
  int method;          /* evict_method */
  int dtype;           /* evict_dtype of K and V */
  int batch;           /* B >= 1 */
  int n_kv_heads;      /* H >= 1 */
  int head_dim;        /* must be EVICT_HEAD_DIM */
  int budget;          /* max rows kept per (b,h) after an update, sinks included */
  int n_sink;          /* leading rows always kept; n_sink + recent < budget */
  int recent;          /* trailing rows always kept (0 = off, the pages' default) */
  int max_block;       /* largest m accepted by an update */
  int max_kept;        /* storage rows per (b,h); 0 means budget. Only evict_set_state
                          can fill more than budget rows. */
  int keep_low;        /* KNorm: 1 keeps the lowest norms (the paper's finding),
                          0 the highest ("L2Norm", §Usage, knorm_keep) */
  int sign;            /* Q-Filters: +1 or -1 ("Q-Filters", §Usage, qfilters_sign) */
  const float* filters;/* Q-Filters: device [n_filter_heads, head_dim] fp32 unit filters,
                          COPIED at init and frozen ("Q-Filters", §How it works step 3).
                          NULL selects the key-SVD fallback (see calib_tokens). */
  int n_filter_heads;  /* Q-Filters: rows of `filters`; must equal n_kv_heads (0 = assume
                          equal). A mismatch raises ("Q-Filters", §Evidence: filters whose
                          head layout disagrees with the layer raise). */
  int rank_cap;        /* CurDKV: leading singular directions (default 16 when 0;
                          "CurDKV-adapted", §Usage, curdkv_rank_cap) */
  void* stream;        /* cudaStream_t for all work of this handle (NULL = legacy default) */
  int calib_tokens;    /* Q-Filters key-SVD fallback (filters == NULL) only: keys seen before
                          the filters freeze (0 = default 128; "Q-Filters", §Usage,
                          qfilters_calib_tokens). While offset + m < calib_tokens an update
                          keeps every row, even over budget, with score 0 (no filter, no
                          eviction). The update that reaches calib_tokens freezes, per
                          (b, h), the top right singular vector of the mean-centred keys
                          present then (kept rows and block), its largest-magnitude
                          component made positive (e_0 when every key is equal), re-scores
                          the kept rows with it and evicts as usual (§How it works step 2,
                          §Key-SVD fallback, §Path dependence: the frozen direction depends
                          on the chunking). Capacity is at least calib_tokens - 1 rows.
                          A non-finite key Gram at the freeze is reported by evict_sync
                          as EVICT_EDEVICE. evict_reset unfreezes. Ignored otherwise. */
  int per_token;       /* CurDKV and H2O: 1 absorbs an m-token update one token at a time,
                          each an m = 1 step ("CurDKV-adapted", §How it works: steps 1-5 per
                          token); a full cache then sheds the unprotected row of lowest
                          score, the lower index of equals (numpy's argmin, step 5). 0 (the
                          default) scores the block at once. EVICT_EINVAL for other methods. */
} evict_config;

/* The kept cache after a call. Pointers are library-owned device memory,
 * valid until the next update / set_state / reset / destroy on the handle.
 * Layout: k, v [batch, n_kv_heads, capacity, head_dim]; pos, score
 * [batch, n_kv_heads, capacity]; rows [0, n_kept) of every (b,h) are valid,
 * in temporal order. pos holds absolute token positions, never renumbered
 * ("Q-Filters", §Adaptation notes). score is the stored fp32 score (KNorm
 * norm, Q-Filters projection, CurDKV cumulative leverage). */
typedef struct evict_view {
  void* k;
  void* v;
  int32_t* pos;
  float* score;
  int32_t n_kept;
  int32_t capacity;
} evict_view;

/* Byte accounting ("L2Norm", §How it works; "Q-Filters", §How it works;
 * "CurDKV-adapted", §Byte accounting). */
typedef struct evict_stats_t {
  int64_t tokens_seen;       /* = offset: absolute tokens passed to updates */
  int64_t tokens_kept;       /* rows per (b,h) */
  int64_t kept_bytes;        /* B*H*tokens_kept*2*D*elem (+ H*D*4 for Q-Filters' filters;
                                the key-SVD fallback counts B*H*D*4 once frozen) */
  int64_t full_seq_bytes;    /* B*H*tokens_seen*2*D*elem */
  double compression_ratio;  /* full_seq_bytes / kept_bytes (0 when nothing kept) */
  int64_t offset;            /* true absolute position of the next token */
} evict_stats_t;

typedef struct evict_handle evict_handle;

/* Create a cache. Validates the configuration ("Q-Filters", §Evidence:
 * n_sink + recent >= budget and an invalid sign raise; filters whose head
 * layout disagrees with the layer raise — the caller states n_kv_heads and
 * the filter buffer must hold exactly n_kv_heads*head_dim floats):
 *   EVICT_EINVAL  bad method/dtype/sizes, head_dim != 128, n_sink+recent >= budget,
 *                 sign not +-1 (Q-Filters), filters NULL (Q-Filters), fp32 with CurDKV;
 *   EVICT_ELIMIT  max(budget,max_kept) + max_block > EVICT_MAX_SELECT_ROWS;
 *   EVICT_ECUDA   device allocation failed.
 * Allocates all device memory the handle will ever use. */
int evict_init(const evict_config* cfg, evict_handle** out);

/* Absorb one block: k, v [B, H, m, D] device, pos [B, m] device int32 or
 * NULL (then positions are offset + [0, m)). Scores the incoming keys
 * once, appends, and over budget keeps the protected top-k in temporal
 * order; then offset += m. m == 0 is a no-op returning the current view.
 * k and v must be 16-byte aligned (they are read with 16-byte vector and
 * TMA loads) and pos 4-byte aligned.
 * EVICT_EINVAL: NULL handle/k/v with m > 0, m < 0, m > max_block, a
 * misaligned k/v/pos, or an append that would exceed capacity without
 * eviction. `out` may be NULL. */
int evict_update_and_fetch(evict_handle* h, const void* k, const void* v, const int32_t* pos,
                           int m, evict_view* out);

/* Grouped update of n_layers (1..32) caches that share every configuration
 * field, their kept-row count, offset and stream — e.g. the layers of one
 * model absorbing the same prompt block. k[l], v[l], pos[l] (pos may be NULL,
 * or hold NULL entries) are layer l's inputs as in evict_update_and_fetch.
 * One set of kernel launches covers all layers, which amortises launch
 * latency for the small per-layer work of a prefill. KNorm and Q-Filters
 * only. `out` (n_layers entries) may be NULL. EVICT_EINVAL if the handles
 * differ or repeat. */
int evict_update_and_fetch_group(evict_handle* const* handles, int n_layers, const void* const* k,
                                 const void* const* v, const int32_t* const* pos, int m,
                                 evict_view* out);

/* Same as evict_update_and_fetch with HOST inputs: copies k_host, v_host
 * (and pos_host if not NULL) to library staging buffers with one
 * cudaMemcpyAsync each on a copy stream of the handle, which the handle's
 * stream then waits for before the update (events on both sides order the
 * staging buffers, so successive calls on different handles overlap one
 * call's kernels with the next call's copies). Host buffers should be
 * pinned; they must stay valid until the handle's stream passes the call. */
int evict_update_and_fetch_host(evict_handle* h, const void* k_host, const void* v_host,
                                const int32_t* pos_host, int m, evict_view* out);

/* The current kept cache (no work enqueued). */
int evict_get_view(const evict_handle* h, evict_view* out);

/* One-shot KNorm / Q-Filters eviction of a single block that allocates
 * nothing. The pages have no counterpart to this call; it exists for callers
 * that cannot call cudaMalloc: code running while a CUDA graph is being
 * captured, serving runtimes that reserve all device memory in their own
 * pool at start-up and forbid later allocations, and plug-ins living inside
 * another framework's memory manager.
 *
 * Same result as a fresh cache created with `cfg` absorbing k, v once
 * through evict_update_and_fetch (offset 0), written to caller buffers:
 *   k, v       [B, H, n, D] device inputs; pos [B, n] device int32 or NULL
 *              (positions 0..n-1); cfg->filters is read in place (not copied);
 *   k_out, v_out [B, H, budget, D], pos_out, score_out [B, H, budget]
 *              device outputs; rows [0, min(n, budget)) of each (b,h) are
 *              written in temporal order.
 * k, v, k_out and v_out must be 16-byte aligned; pos, pos_out, score_out and
 * cfg->filters 4-byte aligned.
 * cfg->max_block, max_kept and rank_cap are ignored; work goes on cfg->stream
 * and the call returns without synchronising.
 * Intermediate data lives in one fixed 8 MiB device array inside the library
 * (held by every GPU that loads it until process exit). A call needs
 * 256 + B*H*(4n + 4*budget + 8 + 4*(ceil(budget/chunk) + 1)) bytes of it plus
 * small rounding (chunk = 64 rows for bf16, 32 for fp32); larger calls return
 * EVICT_ELIMIT. The first call on a device looks up the array's address with
 * that device current — make it before any stream capture. All calls on a
 * device share the array, so calls that overlap on the GPU race.
 *   EVICT_EINVAL  bad configuration (as evict_init), CurDKV, NULL or
 *                 misaligned pointers (nothing is enqueued);
 *   EVICT_ELIMIT  scratch or row bound exceeded;  EVICT_ECUDA  launch failure.
 * A kernel that fails on the device (a bounded wait that gave up, an index
 * outside its bounds) sets the array's error word instead; it stays set until
 * evict_noalloc_status reads it. */
int evict_prefill_noalloc(const evict_config* cfg, const void* k, const void* v, const int32_t* pos, int n,
                          void* k_out, void* v_out, int32_t* pos_out, float* score_out);

/* Device errors of evict_prefill_noalloc calls on the current device: the
 * pages have no counterpart. Synchronises `stream` (cudaStream_t; pass the
 * stream the calls were made on), then reads the error word the calls share.
 * Returns EVICT_OK if no call's kernel has reported an error since the last
 * status call, else EVICT_EDEVICE (with the error named in
 * evict_last_error) and clears the word. Allocates nothing; EVICT_ECUDA if
 * the read fails. */
int evict_noalloc_status(void* stream);

/* Byte accounting from host-side counters (never synchronises). */
int evict_stats(const evict_handle* h, evict_stats_t* out);

/* Load a kept set: k, v [B, H, n, D], pos [B, H, n] int32, score [B, H, n]
 * fp32 (NULL = zeros), all device; n <= capacity. Sets offset. Used to
 * start from a pre-existing cache. EVICT_EINVAL on bad sizes. */
int evict_set_state(evict_handle* h, const void* k, const void* v, const int32_t* pos,
                    const float* score, int n, int64_t offset);

/* Empty the cache and set offset to 0 (host-side only). */
int evict_reset(evict_handle* h);

/* Change the stream of subsequent work. */
int evict_set_stream(evict_handle* h, void* stream);

/* Synchronise the handle's stream and check the device error word:
 * EVICT_ECUDA on a CUDA error, EVICT_EDEVICE if a kernel flagged one
 * (the flag is cleared). */
int evict_sync(evict_handle* h);

void evict_destroy(evict_handle* h);

/* One-time Q-Filters calibration ("Q-Filters", §Calibrated — the paper's
 * actual mechanism): for each query head, the top right singular vector of
 * its uncentered activations q [n_q_heads, n_samples, head_dim] (device,
 * dtype evict_dtype), sign-fixed by sgn(1^T u1); then averaged over
 * contiguous groups of n_q_heads/n_kv_heads query heads and renormalised.
 * Writes filters_out [n_kv_heads, head_dim] fp32 (device). Synchronises the
 * stream (not for use inside graph capture).
 *   EVICT_EINVAL  bad sizes, n_q_heads not a multiple of n_kv_heads;
 *   EVICT_ENUM    a group average shorter than 1e-6 or an all-zero head. */
int evict_qfilters_calibrate(const void* q, int dtype, int n_q_heads, int n_samples, int head_dim,
                             int n_kv_heads, float* filters_out, void* stream);

/* Per-kernel device timing (CUDA events recorded on the handle's stream
 * around each launch). enable != 0 starts recording and clears totals. */
int evict_set_profiling(evict_handle* h, int enable);

typedef struct evict_kernel_time {
  const char* name;     /* static string */
  int64_t launches;
  double total_ms;
} evict_kernel_time;

/* Synchronise, fold the recorded events into per-kernel totals and copy up
 * to max_entries of them to out; *n_out receives the number written. */
int evict_kernel_times(evict_handle* h, evict_kernel_time* out, int max_entries, int* n_out);

/* Rows moved by the handle's last over-budget update, summed over (b,h):
 * *old_moved = kept rows that changed slot, *new_written = incoming rows
 * written into the cache. Synchronises the stream (diagnostic; used to
 * count the compaction's algorithmic bytes). Both are 0 if the last update
 * appended without eviction. */
int evict_compaction_rows(evict_handle* h, int64_t* old_moved, int64_t* new_written);

/* Q-Filters: copy the filters in use to the HOST buffer out_host (may be
 * NULL to query only) and set *n_rows: n_kv_heads rows [H, D] for calibrated
 * filters, B*H rows [B, H, D] once the key-SVD fallback has frozen, 0 before
 * (nothing copied). Synchronises the stream. EVICT_EINVAL for other methods. */
int evict_qfilters_filters(evict_handle* h, float* out_host, int* n_rows);

/* CurDKV / H2O diagnostics: copy the last update's proxy-attention column
 * sums and score increments (CurDKV: leverage; H2O: the mass increment,
 * which leaves out a new row's own weight) of every row of the
 * concatenation (kept rows first, then the block; before compaction) to
 * device buffers attn, leverage [B, H, n] (either may be NULL); *n_rows
 * receives n (0 before the first update). For H2O both buffers receive the
 * mass increment. Enqueued on the handle's stream. EVICT_EINVAL for other
 * methods. */
int evict_curdkv_scores(evict_handle* h, float* attn, float* leverage, int* n_rows);

/* Process-wide count of kernels this library has launched. */
int64_t evict_launch_count(void);

/* Message of the last failed call on this thread ("" if none). */
const char* evict_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EVICT_H */
