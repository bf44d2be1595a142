// Protected top-k selection ("Q-Filters — Query-Agnostic Projection
// Eviction", §How it works step 4 and §Metal kernels; "L2Norm — Intrinsic
// Key-Norm Eviction", §How it works step 3): over budget, every protected row
// (the first n_sink and the trailing recent rows) is kept, then the best
// unprotected rows by priority; rows strictly above the cutoff are always
// admitted and rows equal to it only while quota remains, lowest index first,
// so the budget is never exceeded.
#include "../../include/evict.h"
#include "common.cuh"
#include "launch.h"
#include "params.h"

namespace evict {
namespace {

// ---------------------------------------------------------------------------
// Block-wide exclusive count of a per-thread flag (one tile of THREADS items).
// Returns the flag count of lower-index threads; *total gets the tile total.
// ---------------------------------------------------------------------------
template <int kThreads>
__device__ __forceinline__ uint32_t block_excl_count(bool flag, uint32_t* warp_tot, uint32_t* total) {
  constexpr int kWarps = kThreads / kWarp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const uint32_t in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    uint32_t v = lane < kWarps ? warp_tot[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < kWarps) warp_tot[32 + lane] = incl - v;
    if (lane == 31) warp_tot[64] = incl;
  }
  __syncthreads();
  const uint32_t r = warp_tot[32 + warp] + in_warp;
  *total = warp_tot[64];
  __syncthreads();   // warp_tot is reused by the next call
  return r;
}

// ---------------------------------------------------------------------------
// Protected top-k selection: one CTA per (layer, b, h).
// Order keys of the n = k + m rows live in shared memory. An MSB-first radix
// select (4 passes of 8 bits, warp-aggregated histogram updates) finds the
// key T of the q-th best unprotected row; then one ordered pass admits every
// protected row, every unprotected row above T, and rows equal to T in index
// order while the quota lasts, writing each survivor's source row to
// src_map[destination]. Also resets the compaction read-done flags.
// ---------------------------------------------------------------------------
constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads) select_kernel(const __grid_constant__ GroupParams P) {
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_tot[65];
  __shared__ uint32_t s_prefix, s_rem;
  __shared__ int s_first, s_old_kept;
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = s.k + s.m;
  const float* old_score = L.score_st + (size_t)bh * s.cap;
  const float* new_score = L.new_score + (size_t)bh * s.new_stride;
  for (int i = tid; i < n; i += kSelectThreads) {
    const float sc = i < s.k ? old_score[i] : new_score[i - s.k];
    keys[i] = order_key(s.keep_low ? -sc : sc);
  }
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  for (int j = tid; j < s.flag_stride; j += kSelectThreads) flags[j] = 0;
  if (u == 0 && tid == 0) *P.ticket = 0;          // the compaction that follows draws tickets from 0
  const int lo = s.n_sink, hi = n - s.recent;
  const int q = s.budget - (n - (hi - lo));     // unprotected rows to keep (>= 1)
  if (tid == 0) {
    s_prefix = 0u;
    s_rem = (uint32_t)q;
    s_first = s.k;
    s_old_kept = 0;
  }
  __syncthreads();

  uint32_t prefix = 0u, mask = 0u, rem = (uint32_t)q;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kSelectThreads) hist[b] = 0u;
    __syncthreads();
    for (int base = lo; base < hi; base += kSelectThreads) {
      const int i = base + tid;
      uint32_t bin = 256u;                       // sentinel: not a candidate
      if (i < hi) {
        const uint32_t key = keys[i];
        if ((key & mask) == prefix) bin = (key >> shift) & 255u;
      }
      const unsigned same = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(same) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(same));
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (lane 0 = highest digits)
      uint32_t cnt[8], sum = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) { cnt[j] = hist[255 - 8 * lane - j]; sum += cnt[j]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < rem && rem <= incl);
      if (lane == __ffs(hit) - 1) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= rem) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * lane - j) << shift);
            s_rem = rem - acc;
            break;
          }
          acc += cnt[j];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    rem = s_rem;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix, eq_quota = rem;

  int32_t* src_map = L.src_map + (size_t)bh * s.cap;
  uint32_t eq_carry = 0u, keep_carry = 0u, old_kept = 0u;
  for (int base = 0; base < n; base += kSelectThreads) {
    const int i = base + tid;
    const bool valid = i < n;
    const uint32_t key = valid ? keys[i] : 0u;
    const bool prot = valid && (i < lo || i >= hi);
    const bool eq = valid && !prot && key == T;
    const bool gt = valid && !prot && key > T;
    uint32_t eq_total, keep_total;
    const uint32_t eq_before = eq_carry + block_excl_count<kSelectThreads>(eq, warp_tot, &eq_total);
    const bool keep = prot || gt || (eq && eq_before < eq_quota);
    const uint32_t dest = keep_carry + block_excl_count<kSelectThreads>(keep, warp_tot, &keep_total);
    if (keep) {
      if (dest < (uint32_t)s.budget) src_map[dest] = i;
      else raise_device_error(P.err, kDevBadIndex);
    }
    if (valid && !keep && i < s.k) atomicMin(&s_first, i);
    const unsigned old_bal = __ballot_sync(0xffffffffu, keep && i < s.k);
    if (lane == 0 && old_bal) old_kept += __popc(old_bal);
    eq_carry += eq_total;
    keep_carry += keep_total;
  }
  if (lane == 0 && old_kept) atomicAdd(&s_old_kept, (int)old_kept);
  __syncthreads();
  if (tid == 0) L.meta[bh] = make_int2(s_first, s_old_kept);
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  kernel<<<grid, block, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_select() {
  // Always the compiled maximum: the attribute is per function and device, so
  // a smaller value set for one cache would break launches of a larger one.
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(EVICT_MAX_SELECT_ROWS * sizeof(uint32_t)));
}

cudaError_t launch_select(const GroupParams& P, cudaStream_t st) {
  const int n = P.s.k + P.s.m;
  return launch(select_kernel, dim3(P.s.n_layers * P.s.batch * P.s.heads), dim3(kSelectThreads),
                (size_t)n * sizeof(uint32_t), st, P);
}

}  // namespace evict
