// C ABI of libevict: handle lifetime, validation, launch orchestration,
// byte accounting and per-kernel timing. Declarations and contracts are in
// include/evict.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/evict.h"
#include "api_internal.h"
#include "common.cuh"
#include "launch.h"
#include "params.h"

using namespace evict;

namespace evict {

thread_local std::string g_err;
std::atomic<long long> g_launches{0};

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(EVICT_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

const char* const kKernelNames[kKidCount] = {
    "score", "score_append", "select", "compact", "calib_gram", "calib_eig",
    "curdkv_lse", "curdkv_lse_merge", "curdkv_colsum", "curdkv_colsum_merge", "curdkv_gram", "curdkv_eig", "curdkv_leverage",
    "evict1", "qfilters_freeze", "h2o_mass", "curdkv_attn_small",
};

cudaEvent_t take_event(evict_handle* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void fold_events(evict_handle* h) {
  for (auto& r : h->pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      h->total_ms[r.kid] += ms;
      h->launches[r.kid] += 1;
    }
    h->event_pool.push_back(r.start);
    h->event_pool.push_back(r.stop);
  }
  h->pending.clear();
}

}  // namespace evict

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// CurDKV and H2O share the proxy-attention pipeline and its buffers (curdkv.cu).
bool attention_family(int method) { return method == EVICT_CURDKV || method == EVICT_H2O; }

struct Carver {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t bytes) {
    off = align_up(off, 256);
    T* p = reinterpret_cast<T*>(base + off);
    off += bytes;
    return p;
  }
};

// Bytes of the arena for a configuration (carving with base = nullptr).
size_t arena_layout(evict_handle* h, char* base) {
  const evict_config& c = h->cfg;
  const size_t bh = (size_t)c.batch * c.n_kv_heads;
  const size_t e = h->elem;
  Carver cv{base};
  h->kst = cv.take<void>(bh * h->cap * kHeadDim * e);
  h->vst = cv.take<void>(bh * h->cap * kHeadDim * e);
  h->pos_st = cv.take<int32_t>(bh * h->cap * 4);
  h->score_st = cv.take<float>(bh * h->cap * 4);
  h->filters = cv.take<float>((h->fallback ? bh : (size_t)c.n_kv_heads) * kHeadDim * 4);
  h->new_score = cv.take<float>(bh * c.max_block * 4);
  h->src_map = cv.take<int32_t>(bh * h->cap * 4);
  h->meta = cv.take<int2>(bh * sizeof(int2));
  h->flags = cv.take<int>(bh * h->flag_stride * 4);
  h->waits = cv.take<int2>(bh * (h->flag_stride - 1) * sizeof(int2));
  h->err = cv.take<int>(4);
  h->k_stage = cv.take<void>(bh * c.max_block * kHeadDim * e);
  h->v_stage = cv.take<void>(bh * c.max_block * kHeadDim * e);
  h->pos_stage = cv.take<int32_t>((size_t)c.batch * c.max_block * 4);
  if (c.per_token) {
    h->tok_k = cv.take<void>(bh * kHeadDim * e);
    h->tok_v = cv.take<void>(bh * kHeadDim * e);
    h->tok_pos = cv.take<int32_t>((size_t)c.batch * 4);
  }
  if (attention_family(c.method)) curdkv_layout(h, &cv.off, base);
  return align_up(cv.off, 256);
}

// Keys the Q-Filters key-SVD fallback observes before it freezes its filters.
int fallback_tokens(const evict_config* c) { return c->calib_tokens > 0 ? c->calib_tokens : 128; }

int validate(const evict_config* c) {
  if (!c) return fail(EVICT_EINVAL, "config is NULL");
  if (c->method < EVICT_KNORM || c->method > EVICT_H2O) return fail(EVICT_EINVAL, "unknown method %d", c->method);
  if (c->dtype != EVICT_BF16 && c->dtype != EVICT_FP32) return fail(EVICT_EINVAL, "unknown dtype %d", c->dtype);
  if (attention_family(c->method) && c->dtype != EVICT_BF16)
    return fail(EVICT_EINVAL, "CurDKV and H2O store bf16 keys and values only");
  if (c->batch < 1 || c->n_kv_heads < 1) return fail(EVICT_EINVAL, "batch and n_kv_heads must be >= 1");
  if (c->head_dim != EVICT_HEAD_DIM) return fail(EVICT_EINVAL, "head_dim must be %d (got %d)", EVICT_HEAD_DIM, c->head_dim);
  if (c->budget < 1) return fail(EVICT_EINVAL, "budget must be >= 1");
  if (c->n_sink < 0 || c->recent < 0) return fail(EVICT_EINVAL, "n_sink and recent must be >= 0");
  if ((long long)c->n_sink + c->recent >= c->budget)
    return fail(EVICT_EINVAL, "n_sink + recent (%d + %d) must be below the budget %d", c->n_sink, c->recent, c->budget);
  if (c->max_block < 1) return fail(EVICT_EINVAL, "max_block must be >= 1");
  if (c->max_kept < 0) return fail(EVICT_EINVAL, "max_kept must be >= 0");
  if (c->method == EVICT_QFILTERS) {
    if (c->sign != 1 && c->sign != -1) return fail(EVICT_EINVAL, "sign must be +1 or -1 (got %d)", c->sign);
    if (c->calib_tokens < 0) return fail(EVICT_EINVAL, "calib_tokens must be >= 0 (0 = default 128)");
    if (c->filters && c->n_filter_heads != 0 && c->n_filter_heads != c->n_kv_heads)
      return fail(EVICT_EINVAL, "filters hold %d heads but the layer has %d KV heads", c->n_filter_heads, c->n_kv_heads);
  }
  if (c->method == EVICT_KNORM && c->keep_low != 0 && c->keep_low != 1)
    return fail(EVICT_EINVAL, "keep_low must be 0 or 1");
  if (c->per_token != 0 && c->per_token != 1) return fail(EVICT_EINVAL, "per_token must be 0 or 1");
  if (c->per_token && !attention_family(c->method))
    return fail(EVICT_EINVAL, "per-token mode is for CurDKV and H2O (the other scorers are path independent)");
  if (c->method == EVICT_CURDKV && (c->rank_cap < 0 || c->rank_cap > kCurdkvMaxRank))
    return fail(EVICT_ELIMIT, "rank_cap must be in [1, %d] (0 = default 16)", kCurdkvMaxRank);
  long long cap = std::max(c->budget, c->max_kept);
  if (c->method == EVICT_QFILTERS && !c->filters) cap = std::max(cap, (long long)fallback_tokens(c) - 1);
  if (cap + c->max_block > EVICT_MAX_SELECT_ROWS)
    return fail(EVICT_ELIMIT, "capacity %lld + max_block %d exceeds %d rows per (b,h)", cap, c->max_block,
                EVICT_MAX_SELECT_ROWS);
  if ((long long)c->batch * c->n_kv_heads > 65535 / kMaxGroup)
    return fail(EVICT_ELIMIT, "batch * n_kv_heads must be <= %d", 65535 / kMaxGroup);
  return EVICT_OK;
}

}  // namespace

namespace evict {

GroupParams make_group_params(const evict_handle* h, int m, int n_layers) {
  GroupParams P;
  memset(&P, 0, sizeof(P));
  const evict_config& c = h->cfg;
  P.s.batch = c.batch;
  P.s.heads = c.n_kv_heads;
  P.s.m = m;
  P.s.k = h->n_kept;
  P.s.cap = h->cap;
  P.s.budget = c.budget;
  P.s.n_sink = c.n_sink;
  P.s.recent = c.recent;
  P.s.new_stride = h->new_stride;
  P.s.flag_stride = h->flag_stride;
  P.s.chunk = h->chunk;
  P.s.n_layers = n_layers;
  P.s.keep_low = c.method == EVICT_KNORM ? c.keep_low : 0;
  P.s.sign = (float)(c.method == EVICT_QFILTERS ? c.sign : 1);
  P.s.filter_per_unit = h->fallback ? 1 : 0;
  P.s.zero_scores = h->fallback && !h->frozen ? 1 : 0;
  P.s.method = c.method;
  P.s.offset = h->offset;
  P.err = h->err;
  return P;
}

LayerPtrs make_layer_ptrs(evict_handle* h, const void* k, const void* v, const int32_t* pos) {
  LayerPtrs L;
  L.k_in = k;
  L.v_in = v;
  L.pos_in = pos;
  L.kst = h->kst;
  L.vst = h->vst;
  L.pos_st = h->pos_st;
  L.score_st = h->score_st;
  L.filters = h->filters;
  L.new_score = h->new_score;
  L.src_map = h->src_map;
  L.meta = h->meta;
  L.flags = h->flags;
  L.waits = h->waits;
  return L;
}

}  // namespace evict

namespace {

void fill_view(const evict_handle* h, evict_view* out) {
  if (!out) return;
  out->k = h->kst;
  out->v = h->vst;
  out->pos = h->pos_st;
  out->score = h->score_st;
  out->n_kept = h->n_kept;
  out->capacity = h->cap;
}

bool same_shape(const evict_handle* a, const evict_handle* b) {
  const evict_config &x = a->cfg, &y = b->cfg;
  return x.method == y.method && x.dtype == y.dtype && x.batch == y.batch && x.n_kv_heads == y.n_kv_heads &&
         x.budget == y.budget && x.n_sink == y.n_sink && x.recent == y.recent && x.keep_low == y.keep_low &&
         x.sign == y.sign && x.rank_cap == y.rank_cap && a->cap == b->cap && a->new_stride == b->new_stride &&
         a->fallback == b->fallback && a->frozen == b->frozen && x.calib_tokens == y.calib_tokens &&
         a->n_kept == b->n_kept && a->offset == b->offset && a->stream == b->stream;
}

// Enqueue the update of n_layers same-shaped caches (KNorm / Q-Filters).
int run_intrinsic(evict_handle* const* hs, int n_layers, const void* const* k, const void* const* v,
                  const int32_t* const* pos, int m) {
  evict_handle* h = hs[0];
  GroupParams P = make_group_params(h, m, n_layers);
  for (int l = 0; l < n_layers; ++l) P.L[l] = make_layer_ptrs(hs[l], k[l], v[l], pos ? pos[l] : nullptr);
  const long long n = (long long)h->n_kept + m;
  cudaError_t e;
  if (h->fallback && !h->frozen) {
    if (h->offset + m < h->cfg.calib_tokens) {
      // no filter yet: keep every row (n <= offset + m < calib_tokens <= cap + 1)
      e = timed_launch(h, kKidAppend, [&] { return launch_append(P, h->elem, h->stream); });
      if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
      for (int l = 0; l < n_layers; ++l) {
        hs[l]->n_kept = (int)n;
        hs[l]->last_evicted = false;
        hs[l]->offset += m;
      }
      return EVICT_OK;
    }
    e = timed_launch(h, kKidFreeze, [&] { return launch_freeze(P, h->elem, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "fallback freeze kernel launch");
    for (int l = 0; l < n_layers; ++l) hs[l]->frozen = true;
    P.s.zero_scores = 0;
  }
  if (n <= h->cfg.budget) {
    e = timed_launch(h, kKidAppend, [&] { return launch_append(P, h->elem, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
    for (int l = 0; l < n_layers; ++l) {
      hs[l]->n_kept = (int)n;
      hs[l]->last_evicted = false;
    }
  } else if (n == (long long)h->cfg.budget + 1 && m <= evict1_max_block()) {
    // exactly one row leaves: fused score, selection and one-row shift
    e = timed_launch(h, kKidEvict1, [&] { return launch_evict1(P, h->elem, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "single-eviction kernel launch");
    for (int l = 0; l < n_layers; ++l) {
      hs[l]->n_kept = h->cfg.budget;
      hs[l]->last_evicted = true;
    }
  } else {
    e = timed_launch(h, kKidScore, [&] { return launch_score(P, h->elem, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "score kernel launch");
    e = timed_launch(h, kKidSelect, [&] { return launch_select(P, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "select kernel launch");
    e = timed_launch(h, kKidCompact, [&] { return launch_compact(P, h->elem, h->stream); });
    if (e != cudaSuccess) return cuda_fail(e, "compact kernel launch");
    for (int l = 0; l < n_layers; ++l) {
      hs[l]->n_kept = h->cfg.budget;
      hs[l]->last_evicted = true;
    }
  }
  for (int l = 0; l < n_layers; ++l) hs[l]->offset += m;
  return EVICT_OK;
}

// Per-token mode: the block's tokens one at a time, each gathered into the
// handle's token buffers (one strided copy per tensor) and absorbed as an
// m = 1 update.
int per_token_update(evict_handle* h, const void* k, const void* v, const int32_t* pos, int m) {
  const size_t bh = (size_t)h->cfg.batch * h->cfg.n_kv_heads;
  const size_t row = kHeadDim * (size_t)h->elem;
  for (int t = 0; t < m; ++t) {
    cudaError_t e;
    if ((e = cudaMemcpy2DAsync(h->tok_k, row, static_cast<const char*>(k) + t * row, m * row, row, bh,
                               cudaMemcpyDeviceToDevice, h->stream)) != cudaSuccess ||
        (e = cudaMemcpy2DAsync(h->tok_v, row, static_cast<const char*>(v) + t * row, m * row, row, bh,
                               cudaMemcpyDeviceToDevice, h->stream)) != cudaSuccess)
      return cuda_fail(e, "gathering a token");
    if (pos && (e = cudaMemcpy2DAsync(h->tok_pos, sizeof(int32_t), pos + t, m * sizeof(int32_t), sizeof(int32_t),
                                      h->cfg.batch, cudaMemcpyDeviceToDevice, h->stream)) != cudaSuccess)
      return cuda_fail(e, "gathering a position");
    int rc = curdkv_update(h, h->tok_k, h->tok_v, pos ? h->tok_pos : nullptr, 1);
    if (rc) return rc;
  }
  return EVICT_OK;
}

// `device`: k, v (and pos) are read by the kernels directly, so they must be
// aligned for 16-byte vector and TMA loads (4 bytes for positions).
int check_update_args(const evict_handle* h, const void* k, const void* v, const int32_t* pos, int m, bool device) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  if (m < 0) return fail(EVICT_EINVAL, "m must be >= 0 (got %d)", m);
  if (m > h->cfg.max_block) return fail(EVICT_EINVAL, "m = %d exceeds max_block = %d", m, h->cfg.max_block);
  if (m > 0 && (!k || !v)) return fail(EVICT_EINVAL, "k and v must not be NULL");
  if (device && ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15))
    return fail(EVICT_EINVAL, "k and v must be 16-byte aligned");
  if (device && (reinterpret_cast<uintptr_t>(pos) & 3)) return fail(EVICT_EINVAL, "pos must be 4-byte aligned");
  return EVICT_OK;
}

}  // namespace

extern "C" {

int evict_init(const evict_config* cfg, evict_handle** out) {
  if (!out) return fail(EVICT_EINVAL, "out is NULL");
  *out = nullptr;
  int rc = validate(cfg);
  if (rc) return rc;
  evict_handle* h = new evict_handle();
  h->cfg = *cfg;
  if (h->cfg.method == EVICT_CURDKV && h->cfg.rank_cap == 0) h->cfg.rank_cap = 16;
  h->cfg.filters = nullptr;
  h->fallback = cfg->method == EVICT_QFILTERS && !cfg->filters;
  h->cfg.calib_tokens = h->fallback ? fallback_tokens(cfg) : 0;
  h->elem = cfg->dtype == EVICT_BF16 ? 2 : 4;
  h->cap = std::max(cfg->budget, cfg->max_kept);
  if (h->fallback) h->cap = std::max(h->cap, h->cfg.calib_tokens - 1);
  h->new_stride = cfg->max_block;
  h->chunk = compact_chunk_rows(h->elem);
  h->flag_stride = compact_flag_slots(h->cap, h->elem);
  h->stream = static_cast<cudaStream_t>(cfg->stream);
  const size_t bytes = arena_layout(h, nullptr);
  cudaError_t e = cudaMalloc(&h->arena, bytes);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "device allocation of the cache");
  }
  h->arena_bytes = bytes;
  arena_layout(h, static_cast<char*>(h->arena));
  auto bail = [&](cudaError_t err, const char* what) {
    cudaFree(h->arena);
    delete h;
    return cuda_fail(err, what);
  };
  if ((e = cudaMemsetAsync(h->arena, 0, bytes, h->stream)) != cudaSuccess) return bail(e, "clearing the cache");
  if ((e = prepare_select()) != cudaSuccess) return bail(e, "select kernel attribute");
  if ((e = prepare_evict1()) != cudaSuccess) return bail(e, "single-eviction kernel attribute");
  if (h->fallback && (e = prepare_freeze()) != cudaSuccess) return bail(e, "freeze kernel attribute");
  if (cfg->method == EVICT_QFILTERS && !h->fallback) {
    const size_t fb = (size_t)cfg->n_kv_heads * kHeadDim * sizeof(float);
    if ((e = cudaMemcpyAsync(h->filters, cfg->filters, fb, cudaMemcpyDeviceToDevice, h->stream)) != cudaSuccess)
      return bail(e, "copying the filters");
    std::vector<float> hostf((size_t)cfg->n_kv_heads * kHeadDim);
    if ((e = cudaMemcpyAsync(hostf.data(), h->filters, fb, cudaMemcpyDeviceToHost, h->stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(h->stream)) != cudaSuccess)
      return bail(e, "reading back the filters");
    for (float x : hostf) {
      if (!std::isfinite(x)) {
        cudaFree(h->arena);
        delete h;
        return fail(EVICT_EINVAL, "filters contain a non-finite value");
      }
    }
  }
  if (attention_family(cfg->method)) {
    rc = curdkv_prepare(h);
    if (rc) {
      cudaFree(h->arena);
      curdkv_release(h);
      delete h;
      return rc;
    }
  }
  *out = h;
  return EVICT_OK;
}

int evict_update_and_fetch(evict_handle* h, const void* k, const void* v, const int32_t* pos, int m,
                           evict_view* out) {
  int rc = check_update_args(h, k, v, pos, m, true);
  if (rc) return rc;
  if (m > 0) {
    if (attention_family(h->cfg.method)) {
      rc = h->cfg.per_token && m > 1 ? per_token_update(h, k, v, pos, m) : curdkv_update(h, k, v, pos, m);
    } else {
      rc = run_intrinsic(&h, 1, &k, &v, &pos, m);
    }
    if (rc) return rc;
  }
  fill_view(h, out);
  return EVICT_OK;
}

int evict_update_and_fetch_group(evict_handle* const* hs, int n_layers, const void* const* k,
                                 const void* const* v, const int32_t* const* pos, int m, evict_view* out) {
  if (!hs || n_layers < 1 || n_layers > kMaxGroup)
    return fail(EVICT_EINVAL, "need 1..%d handles (got %d)", kMaxGroup, n_layers);
  if (!k || !v) return fail(EVICT_EINVAL, "k and v arrays must not be NULL");
  for (int l = 0; l < n_layers; ++l) {
    int rc = check_update_args(hs[l], k[l], v[l], pos ? pos[l] : nullptr, m, true);
    if (rc) return rc;
    if (l > 0 && !same_shape(hs[0], hs[l]))
      return fail(EVICT_EINVAL, "handle %d differs from handle 0 in shape, state or stream", l);
    for (int j = 0; j < l; ++j)
      if (hs[j] == hs[l]) return fail(EVICT_EINVAL, "handle %d appears twice", l);
  }
  if (attention_family(hs[0]->cfg.method)) return fail(EVICT_EINVAL, "grouped update supports KNorm and Q-Filters");
  if (m > 0) {
    int rc = run_intrinsic(hs, n_layers, k, v, pos, m);
    if (rc) return rc;
  }
  if (out)
    for (int l = 0; l < n_layers; ++l) fill_view(hs[l], &out[l]);
  return EVICT_OK;
}

int evict_update_and_fetch_host(evict_handle* h, const void* k_host, const void* v_host, const int32_t* pos_host,
                                int m, evict_view* out) {
  int rc = check_update_args(h, k_host, v_host, pos_host, m, false);
  if (rc) return rc;
  if (m > 0) {
    // The copies run on the handle's own copy stream, so that a sequence of calls (one per
    // layer) overlaps each call's kernels with the next call's copies; events order the
    // staging buffers between the two streams.
    cudaError_t e = cudaSuccess;
    if (!h->copy_stream) {
      // all three or none: a later call takes a non-null copy stream as fully set up
      cudaStream_t cs = nullptr;
      cudaEvent_t ready = nullptr, freed = nullptr;
      if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&freed, cudaEventDisableTiming)) != cudaSuccess) {
        if (freed) cudaEventDestroy(freed);
        if (ready) cudaEventDestroy(ready);
        if (cs) cudaStreamDestroy(cs);
        return cuda_fail(e, "creating the copy stream");
      }
      h->copy_stream = cs;
      h->stage_ready = ready;
      h->stage_free = freed;
    }
    if (h->stage_used && (e = cudaStreamWaitEvent(h->copy_stream, h->stage_free, 0)) != cudaSuccess)
      return cuda_fail(e, "ordering the staging buffers");
    const size_t bytes = (size_t)h->cfg.batch * h->cfg.n_kv_heads * m * kHeadDim * h->elem;
    if ((e = cudaMemcpyAsync(h->k_stage, k_host, bytes, cudaMemcpyHostToDevice, h->copy_stream)) != cudaSuccess)
      return cuda_fail(e, "copying k to the device");
    if ((e = cudaMemcpyAsync(h->v_stage, v_host, bytes, cudaMemcpyHostToDevice, h->copy_stream)) != cudaSuccess)
      return cuda_fail(e, "copying v to the device");
    if (pos_host) {
      const size_t pb = (size_t)h->cfg.batch * m * sizeof(int32_t);
      if ((e = cudaMemcpyAsync(h->pos_stage, pos_host, pb, cudaMemcpyHostToDevice, h->copy_stream)) != cudaSuccess)
        return cuda_fail(e, "copying positions to the device");
    }
    if ((e = cudaEventRecord(h->stage_ready, h->copy_stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(h->stream, h->stage_ready, 0)) != cudaSuccess)
      return cuda_fail(e, "ordering the staged block");
  }
  rc = evict_update_and_fetch(h, h->k_stage, h->v_stage, pos_host ? h->pos_stage : nullptr, m, out);
  if (rc == EVICT_OK && m > 0) {
    cudaError_t e = cudaEventRecord(h->stage_free, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "ordering the staging buffers");
    h->stage_used = true;
  }
  return rc;
}

int evict_get_view(const evict_handle* h, evict_view* out) {
  if (!h || !out) return fail(EVICT_EINVAL, "handle and out must not be NULL");
  fill_view(h, out);
  return EVICT_OK;
}

int evict_stats(const evict_handle* h, evict_stats_t* out) {
  if (!h || !out) return fail(EVICT_EINVAL, "handle and out must not be NULL");
  const evict_config& c = h->cfg;
  const int64_t per_token = (int64_t)c.batch * c.n_kv_heads * 2 * kHeadDim * h->elem;
  out->tokens_seen = h->offset;
  out->tokens_kept = h->n_kept;
  out->kept_bytes = per_token * h->n_kept;
  if (c.method == EVICT_QFILTERS && !h->fallback) out->kept_bytes += (int64_t)c.n_kv_heads * kHeadDim * 4;
  if (h->fallback && h->frozen) out->kept_bytes += (int64_t)c.batch * c.n_kv_heads * kHeadDim * 4;
  out->full_seq_bytes = per_token * h->offset;
  out->compression_ratio = out->kept_bytes ? (double)out->full_seq_bytes / (double)out->kept_bytes : 0.0;
  out->offset = h->offset;
  return EVICT_OK;
}

int evict_set_state(evict_handle* h, const void* k, const void* v, const int32_t* pos, const float* score, int n,
                    int64_t offset) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  if (n < 0 || n > h->cap) return fail(EVICT_EINVAL, "n = %d outside [0, capacity %d]", n, h->cap);
  if (offset < n) return fail(EVICT_EINVAL, "offset %lld below the kept row count %d", (long long)offset, n);
  if (n > 0 && (!k || !v || !pos)) return fail(EVICT_EINVAL, "k, v and pos must not be NULL");
  const size_t bh = (size_t)h->cfg.batch * h->cfg.n_kv_heads;
  const size_t row = kHeadDim * h->elem;
  cudaError_t e;
  if (n > 0) {
    if ((e = cudaMemcpy2DAsync(h->kst, h->cap * row, k, n * row, n * row, bh, cudaMemcpyDeviceToDevice,
                               h->stream)) != cudaSuccess)
      return cuda_fail(e, "loading k");
    if ((e = cudaMemcpy2DAsync(h->vst, h->cap * row, v, n * row, n * row, bh, cudaMemcpyDeviceToDevice,
                               h->stream)) != cudaSuccess)
      return cuda_fail(e, "loading v");
    if ((e = cudaMemcpy2DAsync(h->pos_st, h->cap * 4, pos, n * 4, n * 4, bh, cudaMemcpyDeviceToDevice,
                               h->stream)) != cudaSuccess)
      return cuda_fail(e, "loading positions");
    if (score)
      e = cudaMemcpy2DAsync(h->score_st, h->cap * 4, score, n * 4, n * 4, bh, cudaMemcpyDeviceToDevice, h->stream);
    else
      e = cudaMemset2DAsync(h->score_st, h->cap * 4, 0, n * 4, bh, h->stream);
    if (e != cudaSuccess) return cuda_fail(e, "loading scores");
  }
  h->n_kept = n;
  h->offset = offset;
  h->last_evicted = false;
  return EVICT_OK;
}

int evict_reset(evict_handle* h) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  h->n_kept = 0;
  h->offset = 0;
  h->last_evicted = false;
  h->frozen = false;          // the fallback estimates new filters for the next sequence
  return EVICT_OK;
}

int evict_set_stream(evict_handle* h, void* stream) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  h->stream = static_cast<cudaStream_t>(stream);
  h->cfg.stream = stream;
  return EVICT_OK;
}

int evict_sync(evict_handle* h) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int err = 0;
  if ((e = cudaMemcpy(&err, h->err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the device error word");
  if (err) {
    cudaMemset(h->err, 0, sizeof(int));
    return fail(EVICT_EDEVICE, "a kernel reported device error %d (%s)", err,
                err == kDevWaitTimeout  ? "bounded wait timed out"
                : err == kDevNonFinite ? "non-finite key Gram at the fallback freeze"
                                       : "index check failed");
  }
  return EVICT_OK;
}

void evict_destroy(evict_handle* h) {
  if (!h) return;
  cudaStreamSynchronize(h->stream);
  for (auto& r : h->pending) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  for (auto ev : h->event_pool) cudaEventDestroy(ev);
  if (h->copy_stream) {
    cudaStreamSynchronize(h->copy_stream);
    cudaEventDestroy(h->stage_ready);
    cudaEventDestroy(h->stage_free);
    cudaStreamDestroy(h->copy_stream);
  }
  cudaFree(h->arena);
  curdkv_release(h);
  delete h;
}

int evict_set_profiling(evict_handle* h, int enable) {
  if (!h) return fail(EVICT_EINVAL, "handle is NULL");
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  fold_events(h);
  h->profiling = enable != 0;
  for (int i = 0; i < kKidCount; ++i) {
    h->total_ms[i] = 0.0;
    h->launches[i] = 0;
  }
  return EVICT_OK;
}

int evict_kernel_times(evict_handle* h, evict_kernel_time* out, int max_entries, int* n_out) {
  if (!h || !n_out) return fail(EVICT_EINVAL, "handle and n_out must not be NULL");
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  fold_events(h);
  int n = 0;
  for (int i = 0; i < kKidCount; ++i) {
    if (!h->launches[i]) continue;
    if (out && n < max_entries) {
      out[n].name = kKernelNames[i];
      out[n].launches = h->launches[i];
      out[n].total_ms = h->total_ms[i];
      ++n;
    }
  }
  *n_out = n;
  return EVICT_OK;
}

int evict_compaction_rows(evict_handle* h, int64_t* old_moved, int64_t* new_written) {
  if (!h || !old_moved || !new_written) return fail(EVICT_EINVAL, "arguments must not be NULL");
  *old_moved = 0;
  *new_written = 0;
  if (!h->last_evicted) return EVICT_OK;
  const size_t bh = (size_t)h->cfg.batch * h->cfg.n_kv_heads;
  std::vector<int2> meta(bh);
  cudaError_t e = cudaStreamSynchronize(h->stream);
  if (e == cudaSuccess) e = cudaMemcpy(meta.data(), h->meta, bh * sizeof(int2), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading compaction metadata");
  for (const int2& m : meta) {
    *old_moved += m.y - m.x;
    *new_written += h->cfg.budget - m.y;
  }
  return EVICT_OK;
}

int evict_qfilters_filters(evict_handle* h, float* out_host, int* n_rows) {
  if (!h || !n_rows) return fail(EVICT_EINVAL, "handle and n_rows must not be NULL");
  if (h->cfg.method != EVICT_QFILTERS) return fail(EVICT_EINVAL, "not a Q-Filters cache");
  const evict_config& c = h->cfg;
  const int rows = h->fallback ? (h->frozen ? c.batch * c.n_kv_heads : 0) : c.n_kv_heads;
  *n_rows = rows;
  if (!out_host || rows == 0) return EVICT_OK;
  cudaError_t e = cudaMemcpyAsync(out_host, h->filters, (size_t)rows * kHeadDim * sizeof(float),
                                  cudaMemcpyDeviceToHost, h->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the filters");
  return EVICT_OK;
}

int evict_curdkv_scores(evict_handle* h, float* attn, float* leverage, int* n_rows) {
  if (!h || !n_rows) return fail(EVICT_EINVAL, "handle and n_rows must not be NULL");
  if (!attention_family(h->cfg.method)) return fail(EVICT_EINVAL, "not a CurDKV or H2O cache");
  return curdkv_last_scores(h, attn, leverage, n_rows);
}

int64_t evict_launch_count(void) { return g_launches.load(); }

const char* evict_last_error(void) { return g_err.c_str(); }

}  // extern "C"
