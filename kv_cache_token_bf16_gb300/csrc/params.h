// Launch parameters shared by the host orchestration and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace evict {

// Up to this many layer caches can be updated by one set of launches.
constexpr int kMaxGroup = 32;

enum Method : int { kKNorm = 0, kQFilters = 1, kCurDKV = 2 };

// Per-layer device pointers of one grouped update.
struct LayerPtrs {
  const void* k_in;        // [B, H, m, D] incoming keys
  const void* v_in;        // [B, H, m, D] incoming values
  const int32_t* pos_in;   // [B, m] or null (positions = offset + t)
  void* kst;               // [B, H, cap, D] kept keys (in place)
  void* vst;               // [B, H, cap, D] kept values
  int32_t* pos_st;         // [B, H, cap]
  float* score_st;         // [B, H, cap]
  float* filters;          // Q-Filters: [H, D] calibrated, or [B, H, D] frozen by the key-SVD
                           // fallback (written only by the freeze kernel)
  float* new_score;        // [B, H, new_stride] scores of incoming rows
  int32_t* src_map;        // [B, H, cap] source row of each kept destination
  int2* meta;              // [B, H] {first moved destination, old survivors}
  int* flags;              // [B, H, flag_stride] compaction read-done flags, then the chunk counter
  int2* waits;             // [B, H, flag_stride - 1] per destination chunk, the lower chunks whose
                           // reads of kept rows overlap its destinations ({lo, hi}; empty: hi < lo);
                           // written by the select kernel when k > 0
};

// Sizes common to every layer of a grouped update.
struct Shape {
  int batch, heads;        // B, H
  int m;                   // incoming rows
  int k;                   // kept rows before the call
  int cap;                 // storage rows per (b, h)
  int budget;
  int n_sink, recent;
  int new_stride;          // row stride of new_score (max_block)
  int flag_stride;         // flag slots per (b, h): one per chunk + the chunk counter
  int chunk;               // rows per compaction chunk
  int n_layers;
  int keep_low;            // KNorm keep-low: priority = -score
  float sign;              // Q-Filters sign
  int filter_per_unit;     // Q-Filters: filters are [B, H, D] (key-SVD fallback), else [H, D]
  int zero_scores;         // append stores score 0 (key-SVD fallback before its freeze)
  int tie_low;             // single eviction: of equal lowest scores the lower index leaves
  int method;
  long long offset;        // absolute position of the first incoming token
};

struct GroupParams {
  Shape s;
  int* err;                // device error word
  int total_ctas;          // compaction grid size
  LayerPtrs L[kMaxGroup];
};

}  // namespace evict
