// Internal definition of the cache handle and host helpers shared by the
// translation units of libevict.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <string>
#include <vector>

#include "../../include/evict.h"
#include "params.h"

namespace evict {

enum KernelId : int {
  kKidScore,
  kKidAppend,
  kKidSelect,
  kKidCompact,
  kKidCalibGram,
  kKidCalibEig,
  kKidCurdkvLse,
  kKidCurdkvLseMerge,
  kKidCurdkvColsum,
  kKidCurdkvColsumMerge,
  kKidCurdkvGram,
  kKidCurdkvEig,
  kKidCurdkvLeverage,
  kKidEvict1,
  kKidFreeze,
  kKidH2oMass,
  kKidCurdkvAttnSmall,
  kKidCount
};

// Largest CurDKV rank cap (leading singular directions) the eigensolver keeps.
constexpr int kCurdkvMaxRank = 32;

struct CurdkvState;   // defined in curdkv.cu

}  // namespace evict

struct evict_handle {
  evict_config cfg;
  int elem = 2;               // bytes per K/V element
  int cap = 0;                // storage rows per (b, h)
  int chunk = 64;             // compaction chunk rows
  int flag_stride = 0;        // compaction flag slots per (b, h): chunk flags + chunk counter
  int new_stride = 0;         // row stride of new_score (= max_block)
  bool fallback = false;      // Q-Filters without calibrated filters: key-SVD fallback
  bool frozen = false;        // fallback: the per-(b, h) filters have been estimated
  cudaStream_t stream = nullptr;

  void* arena = nullptr;      // one device allocation, carved below
  size_t arena_bytes = 0;
  void* kst = nullptr;
  void* vst = nullptr;
  int32_t* pos_st = nullptr;
  float* score_st = nullptr;
  float* filters = nullptr;   // [H, D] calibrated, or [B, H, D] for the fallback
  float* new_score = nullptr;
  int32_t* src_map = nullptr;
  int2* meta = nullptr;
  int* flags = nullptr;
  int2* waits = nullptr;
  int* err = nullptr;
  void* k_stage = nullptr;
  void* v_stage = nullptr;
  int32_t* pos_stage = nullptr;
  cudaStream_t copy_stream = nullptr;   // host-input call: copies into the staging buffers
  cudaEvent_t stage_ready = nullptr;    // the staged block has landed (copy stream)
  cudaEvent_t stage_free = nullptr;     // the last call's kernels are done with the staging (stream)
  bool stage_used = false;
  void* tok_k = nullptr;      // per-token mode: the current token of every (b, h)
  void* tok_v = nullptr;
  int32_t* tok_pos = nullptr;
  evict::CurdkvState* curdkv = nullptr;

  int n_kept = 0;             // rows per (b, h), identical for every (b, h)
  int64_t offset = 0;         // absolute position of the next token
  bool last_evicted = false;  // the last update ran select + compaction

  bool profiling = false;
  struct Rec {
    int kid;
    cudaEvent_t start, stop;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> event_pool;
  double total_ms[evict::kKidCount] = {};
  int64_t launches[evict::kKidCount] = {};
};

namespace evict {

extern thread_local std::string g_err;
extern std::atomic<long long> g_launches;

int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
cudaEvent_t take_event(evict_handle* h);
void fold_events(evict_handle* h);

// Launch through `f` (returns cudaError_t), counting it and, when profiling,
// bracketing it with events on the handle's stream.
template <typename F>
cudaError_t timed_launch(evict_handle* h, int kid, F&& f) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (h->profiling) {
    if (h->pending.size() > 60000) {
      cudaStreamSynchronize(h->stream);
      fold_events(h);
    }
    a = take_event(h);
    b = take_event(h);
    if (a) cudaEventRecord(a, h->stream);
  }
  cudaError_t e = f();
  g_launches.fetch_add(1);
  if (a && b) {
    cudaEventRecord(b, h->stream);
    h->pending.push_back({kid, a, b});
  }
  return e;
}

// Launch parameters of an update of n_layers same-shaped caches (evict_api.cu).
GroupParams make_group_params(const evict_handle* h, int m, int n_layers);
LayerPtrs make_layer_ptrs(evict_handle* h, const void* k, const void* v, const int32_t* pos);

// CurDKV hooks (curdkv.cu).
void curdkv_layout(evict_handle* h, size_t* offset, char* base);
void curdkv_release(evict_handle* h);
int curdkv_prepare(evict_handle* h);
int curdkv_update(evict_handle* h, const void* k, const void* v, const int32_t* pos, int m);
int curdkv_last_scores(const evict_handle* h, float* attn, float* lev, int* n_out);

}  // namespace evict
