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
// Block-wide exclusive sum of one uint32 per thread; *total gets the sum.
// `scratch` holds 2 * 32 + 1 words.
// ---------------------------------------------------------------------------
template <int kThreads>
__device__ __forceinline__ uint32_t block_excl_sum(uint32_t x, uint32_t* scratch, uint32_t* total) {
  constexpr int kWarps = kThreads / kWarp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = lane < kWarps ? scratch[lane] : 0u;
    uint32_t wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) scratch[32 + lane] = wi - v;
    if (lane == 31) scratch[64] = wi;
  }
  __syncthreads();
  const uint32_t r = scratch[32 + warp] + incl - x;
  *total = scratch[64];
  __syncthreads();   // scratch is reused by the next call
  return r;
}

// ---------------------------------------------------------------------------
// Protected top-k selection: one CTA per (layer, b, h), keys in registers.
//
// Thread t owns the contiguous rows [t*kPer, t*kPer + kPer) and their 32-bit
// order keys. A block min/max over the unprotected keys gives the bits every
// candidate shares; the remaining bits are resolved most-significant first
// in digits of up to 11 bits (a 2048-bin shared histogram per pass, later
// passes only counting keys that still match the prefix), which yields the
// key T of the q-th best unprotected row and how many rows equal to T fit.
// Two block scans then give each segment its count of equal rows and of kept
// rows before it; each thread writes its survivors' source rows to
// src_map[destination] in index order. Also zeroes the unit's compaction
// flags and chunk counter.
// ---------------------------------------------------------------------------
constexpr int kDigitBits = 11;
constexpr int kBins = 1 << kDigitBits;
// destination chunks per (b, h) the wait ranges can describe (smallest chunk: 32 rows)
constexpr int kMaxWaitChunks = (EVICT_MAX_SELECT_ROWS + 31) / 32;

// Wait ranges of the compaction: a survivor with destination d and kept
// source sr (sr < k) is read by chunk d / C and overwritten by chunk sr / C;
// when those differ the overwriting chunk cs must wait for the reading chunks
// [lo, hi].
__device__ __forceinline__ void note_wait_range(int* wlo, int* whi, int cs, int lo, int hi) {
  atomicMin(&wlo[cs], lo);
  atomicMax(&whi[cs], hi);
}
__device__ __forceinline__ void init_waits(int* wlo, int* whi, int chunks) {
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
    wlo[c] = 0x7fffffff;
    whi[c] = -1;
  }
}
__device__ __forceinline__ void store_waits(const int* wlo, const int* whi, int2* out, int chunks) {
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) out[c] = make_int2(wlo[c], whi[c]);
}

template <int kThreads, int kPer, int kMinBlocks = 1>
__global__ void __launch_bounds__(kThreads, kMinBlocks) select_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t scan[65];
  __shared__ uint32_t s_min[32], s_max[32];
  __shared__ uint32_t s_prefix, s_rem;
  __shared__ int s_first, s_old_kept;
  __shared__ int s_wlo[kMaxWaitChunks], s_whi[kMaxWaitChunks];
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kThreads / 32;
  const int chunks = s.flag_stride - 1;
  if (s.k > 0) init_waits(s_wlo, s_whi, chunks);
  const int n = s.k + s.m;
  const int lo = s.n_sink, hi = n - s.recent;
  const int q = s.budget - (n - (hi - lo));      // unprotected rows to keep (>= 1)
  const float* old_score = L.score_st + (size_t)bh * s.cap;
  const float* new_score = L.new_score + (size_t)bh * s.new_stride;
  const int i0 = tid * kPer;

  uint32_t key[kPer];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = i0 + j;
    float sc = 0.f;
    if (i < n) sc = i < s.k ? old_score[i] : new_score[i - s.k];
    key[j] = order_key(s.keep_low ? -sc : sc);
    if (i >= lo && i < hi) {
      kmin = min(kmin, key[j]);
      kmax = max(kmax, key[j]);
    }
  }
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  for (int j = tid; j < s.flag_stride; j += kThreads) flags[j] = 0;   // flags and chunk counter
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    s_min[warp] = kmin;
    s_max[warp] = kmax;
  }
  if (tid == 0) {
    s_first = s.k;
    s_old_kept = 0;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = lane < kWarps ? s_min[lane] : 0xffffffffu;
    uint32_t b = lane < kWarps ? s_max[lane] : 0u;
    a = __reduce_min_sync(0xffffffffu, a);
    b = __reduce_max_sync(0xffffffffu, b);
    if (lane == 0) {
      s_min[0] = a;
      s_max[0] = b;
    }
  }
  __syncthreads();
  const uint32_t all_min = s_min[0], all_max = s_max[0];
  // every unprotected key shares the top `common` bits
  const int common = all_min == all_max ? 32 : __clz(all_min ^ all_max);
  uint32_t mask = common == 0 ? 0u : (common == 32 ? 0xffffffffu : ~(0xffffffffu >> common));
  uint32_t prefix = all_min & mask, rem = (uint32_t)q;
  int low = 32 - common;                          // unresolved low bits
  while (low > 0) {
    const int w = low < kDigitBits ? low : kDigitBits;
    const int shift = low - w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int b = tid; b < kBins; b += kThreads) hist[b] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = i0 + j;
      if (i >= lo && i < hi && (key[j] & mask) == prefix) atomicAdd(&hist[(key[j] >> shift) & dmask], 1u);
    }
    __syncthreads();
    // bins from the top: thread t owns bins (nb-1-t*bpt) downwards
    const int nb = 1 << w;
    constexpr int kBpt = kBins / kThreads;        // bins per thread at full width
    const int bpt = nb >= kThreads ? nb / kThreads : 1;
    uint32_t cnt[kBpt > 0 ? kBpt : 1];
    uint32_t sum = 0u;
    const int top = nb - 1 - tid * bpt;
#pragma unroll
    for (int j = 0; j < (kBpt > 0 ? kBpt : 1); ++j) {
      cnt[j] = (j < bpt && top - j >= 0) ? hist[top - j] : 0u;
      sum += cnt[j];
    }
    uint32_t total;
    const uint32_t above = block_excl_sum<kThreads>(sum, scan, &total);   // counts of higher bins
    if (above < rem && rem <= above + sum) {
      uint32_t acc = above;
#pragma unroll
      for (int j = 0; j < (kBpt > 0 ? kBpt : 1); ++j) {
        if (acc + cnt[j] >= rem) {
          s_prefix = prefix | ((uint32_t)(top - j) << shift);
          s_rem = rem - acc;
          break;
        }
        acc += cnt[j];
      }
    }
    __syncthreads();
    prefix = s_prefix;
    rem = s_rem;
    mask |= dmask << shift;
    low = shift;
  }
  const uint32_t T = prefix, eq_quota = rem;

  // ordered admission over the contiguous per-thread segments
  uint32_t eq_count = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = i0 + j;
    eq_count += (i >= lo && i < hi && key[j] == T) ? 1u : 0u;
  }
  uint32_t total;
  const uint32_t eq_before = block_excl_sum<kThreads>(eq_count, scan, &total);
  uint32_t keep_bits = 0u, eb = eq_before;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = i0 + j;
    if (i >= n) continue;
    const bool prot = i < lo || i >= hi;
    bool keep = prot || key[j] > T;
    if (!prot && key[j] == T) keep = eb++ < eq_quota;
    if (keep) keep_bits |= 1u << j;
  }
  uint32_t dest = block_excl_sum<kThreads>((uint32_t)__popc(keep_bits), scan, &total);
  int32_t* src_map = L.src_map + (size_t)bh * s.cap;
  const int chunk_shift = __ffs(s.chunk) - 1;         // compaction chunks are 32 or 64 rows: a power of two
  int first_drop = s.k;
  uint32_t old_kept = 0u;
  // wait ranges: the thread's rows and destinations both increase, so each source chunk's
  // destination chunks form one run; it is recorded once per run
  int run_cs = -1, run_lo = 0, run_hi = -1;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = i0 + j;
    if (i >= n) continue;
    if (keep_bits & (1u << j)) {
      if (dest < (uint32_t)s.budget) src_map[dest] = i;
      else raise_device_error(P.err, kDevBadIndex);
      if (i < s.k) {
        ++old_kept;
        const int cd = (int)dest >> chunk_shift, cs = i >> chunk_shift;
        if (cd < cs) {
          if (cs != run_cs) {
            if (run_cs >= 0) note_wait_range(s_wlo, s_whi, run_cs, run_lo, run_hi);
            run_cs = cs;
            run_lo = cd;
          }
          run_hi = cd;
        }
      }
      ++dest;
    } else if (i < s.k && i < first_drop) {
      first_drop = i;
    }
  }
  if (run_cs >= 0) note_wait_range(s_wlo, s_whi, run_cs, run_lo, run_hi);
  // the first dropped kept row: one shared atomic per warp (a per-thread atomic on one address
  // serialises hundreds of updates)
  const int wfirst = __reduce_min_sync(0xffffffffu, first_drop);
  if (lane == 0 && wfirst < s.k) atomicMin(&s_first, wfirst);
  const uint32_t wsum = __reduce_add_sync(0xffffffffu, old_kept);
  if (lane == 0 && wsum) atomicAdd(&s_old_kept, (int)wsum);
  __syncthreads();
  if (tid == 0) L.meta[bh] = make_int2(s_first, s_old_kept);
  if (s.k > 0) store_waits(s_wlo, s_whi, L.waits + (size_t)bh * chunks, chunks);
}

// ---------------------------------------------------------------------------
// Protected top-k selection for large n (above the register variant's
// reach): one CTA per (layer, b, h). Order keys of the n = k + m rows live in
// shared memory. An MSB-first radix
// select (4 passes of 8 bits, warp-aggregated histogram updates) finds the
// key T of the q-th best unprotected row. Then each thread takes a contiguous
// segment of rows: a first block scan counts the rows equal to T before each
// segment (equal rows are admitted in index order while the quota lasts), a
// second counts the kept rows before each segment, and each thread writes
// the source row of each of its survivors to src_map[destination]. Also
// zeroes the compaction flags and chunk counter of the unit.
// ---------------------------------------------------------------------------
template <int kThreads>
__global__ void __launch_bounds__(kThreads) select_smem_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scan[65];
  __shared__ uint32_t s_prefix, s_rem;
  __shared__ int s_first, s_old_kept;
  __shared__ int s_wlo[kMaxWaitChunks], s_whi[kMaxWaitChunks];
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = s.k + s.m;
  const int chunks = s.flag_stride - 1;
  if (s.k > 0) init_waits(s_wlo, s_whi, chunks);
  const float* old_score = L.score_st + (size_t)bh * s.cap;
  const float* new_score = L.new_score + (size_t)bh * s.new_stride;
  for (int i = tid; i < n; i += kThreads) {
    const float sc = i < s.k ? old_score[i] : new_score[i - s.k];
    keys[i] = order_key(s.keep_low ? -sc : sc);
  }
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  for (int j = tid; j < s.flag_stride; j += kThreads) flags[j] = 0;   // flags and chunk counter
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
    for (int b = tid; b < 256; b += kThreads) hist[b] = 0u;
    __syncthreads();
    for (int base = lo; base < hi; base += kThreads) {
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

  // ordered admission over contiguous per-thread segments
  const int per = (n + kThreads - 1) / kThreads;
  const int i_begin = min(n, tid * per), i_end = min(n, i_begin + per);
  uint32_t eq_count = 0u;
  for (int i = i_begin; i < i_end; ++i) eq_count += (i >= lo && i < hi && keys[i] == T) ? 1u : 0u;
  uint32_t total;
  uint32_t eq_before = block_excl_sum<kThreads>(eq_count, scan, &total);
  uint32_t keep_count = 0u;
  {
    uint32_t eb = eq_before;
    for (int i = i_begin; i < i_end; ++i) {
      const bool prot = i < lo || i >= hi;
      const uint32_t key = keys[i];
      bool keep = prot || key > T;
      if (!prot && key == T) keep = eb++ < eq_quota;
      keep_count += keep ? 1u : 0u;
    }
  }
  uint32_t dest = block_excl_sum<kThreads>(keep_count, scan, &total);
  int32_t* src_map = L.src_map + (size_t)bh * s.cap;
  const int chunk_shift = __ffs(s.chunk) - 1;         // compaction chunks are 32 or 64 rows: a power of two
  int first_drop = s.k;
  uint32_t old_kept = 0u;
  {
    uint32_t eb = eq_before;
    int run_cs = -1, run_lo = 0, run_hi = -1;           // wait ranges, one record per run (as above)
    for (int i = i_begin; i < i_end; ++i) {
      const bool prot = i < lo || i >= hi;
      const uint32_t key = keys[i];
      bool keep = prot || key > T;
      if (!prot && key == T) keep = eb++ < eq_quota;
      if (keep) {
        if (dest < (uint32_t)s.budget) src_map[dest] = i;
        else raise_device_error(P.err, kDevBadIndex);
        if (i < s.k) {
          ++old_kept;
          const int cd = (int)dest >> chunk_shift, cs = i >> chunk_shift;
          if (cd < cs) {
            if (cs != run_cs) {
              if (run_cs >= 0) note_wait_range(s_wlo, s_whi, run_cs, run_lo, run_hi);
              run_cs = cs;
              run_lo = cd;
            }
            run_hi = cd;
          }
        }
        ++dest;
      } else if (i < s.k && i < first_drop) {
        first_drop = i;
      }
    }
    if (run_cs >= 0) note_wait_range(s_wlo, s_whi, run_cs, run_lo, run_hi);
  }
  // the first dropped kept row: one shared atomic per warp (a per-thread atomic on one address
  // serialises hundreds of updates)
  const int wfirst = __reduce_min_sync(0xffffffffu, first_drop);
  if (lane == 0 && wfirst < s.k) atomicMin(&s_first, wfirst);
  const uint32_t wsum = __reduce_add_sync(0xffffffffu, old_kept);
  if (lane == 0 && wsum) atomicAdd(&s_old_kept, (int)wsum);
  __syncthreads();
  if (tid == 0) L.meta[bh] = make_int2(s_first, s_old_kept);
  if (s.k > 0) store_waits(s_wlo, s_whi, L.waits + (size_t)bh * chunks, chunks);
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  return launch_pdl(kernel, grid, block, smem, st, nullptr, P);
}

}  // namespace

cudaError_t prepare_select() {
  // The shared-memory variant serves the largest row counts. The attribute is
  // always the compiled maximum: it is per function and device, so a smaller
  // value set for one cache would break launches of a larger one.
  const int bytes = (int)(EVICT_MAX_SELECT_ROWS * sizeof(uint32_t));
  return cudaFuncSetAttribute(select_smem_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

cudaError_t launch_select(const GroupParams& P, cudaStream_t st) {
  const int n = P.s.k + P.s.m;
  const dim3 grid(P.s.n_layers * P.s.batch * P.s.heads);
  if (n <= 256 * 4) return launch(select_kernel<256, 4>, grid, dim3(256), 0, st, P);
  if (n <= 256 * 8) return launch(select_kernel<256, 8>, grid, dim3(256), 0, st, P);
  if (n <= 512 * 16) {
    // more (b, h) units than SMs: 512-thread CTAs, two per SM, keep every unit in one wave
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((int)grid.x > sms && (int)grid.x <= 2 * sms)
      return launch(select_kernel<512, 16, 2>, grid, dim3(512), 0, st, P);
  }
  if (n <= 1024 * 8) return launch(select_kernel<1024, 8>, grid, dim3(1024), 0, st, P);
  // the fewest keys per thread that hold n: less serial work per pass, no register spills
  if (n <= 1024 * 12) return launch(select_kernel<1024, 12>, grid, dim3(1024), 0, st, P);
  if (n <= 1024 * 17) return launch(select_kernel<1024, 17>, grid, dim3(1024), 0, st, P);
  if (n <= 1024 * 24) return launch(select_kernel<1024, 24>, grid, dim3(1024), 0, st, P);
  return launch(select_smem_kernel<1024>, grid, dim3(1024), (size_t)n * sizeof(uint32_t), st, P);
}

}  // namespace evict
