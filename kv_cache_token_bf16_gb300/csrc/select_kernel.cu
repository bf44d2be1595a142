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
// order keys; bit j of its masks stands for row t*kPer + j. A block min/max
// over the unprotected keys gives the bits every candidate shares; the
// remaining bits are resolved most-significant first in digits of up to 11
// bits: each pass counts the candidates still matching the prefix in a
// 2048-bin shared histogram, and one warp scans it for the bin holding the
// rem-th best. Passes stop once every bit is resolved or once the whole bin
// is admitted (rem equals its count): then every row of the bin is kept and
// its low bits never decide anything. The result is a masked threshold: rows
// whose masked key is above the prefix are kept, and of the rows whose masked
// key equals it, the first eq_quota in index order. One block scan of the
// per-thread counts of both classes gives each thread its first destination;
// each thread then writes the source row of each of its survivors to a
// shared copy of src_map (budget words of dynamic shared memory), which the
// block stores coalesced at the end. Also zeroes the unit's compaction flags
// and chunk counter.
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

// Bits [a, b) of a 32-bit mask (0 <= a, b <= 31).
__device__ __forceinline__ uint32_t bit_range(int a, int b) {
  return b > a ? ((1u << (b - a)) - 1u) << a : 0u;
}

// Inclusive warp sum.
__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// One warp finds the bin holding the rem-th candidate counted from the top of
// a 2048-bin histogram: lane l sums the 64 bins of group 31 - l (groups from
// the top; its 16 vector loads are rotated by l so that no two lanes of a
// quarter-warp share a bank), a warp scan picks the group, and the group's
// bins, two per lane from its top, a second scan picks the bin. Returns the
// bin; *above gets the candidates in higher bins, *count the bin's count.
__device__ __forceinline__ int warp_find_bin(const uint32_t* h, uint32_t rem, uint32_t* above, uint32_t* count) {
  const int lane = threadIdx.x & 31;
  const int g = 31 - lane;                        // this lane's group: bins [64g, 64g + 64)
  const uint4* gv = reinterpret_cast<const uint4*>(h + 64 * g);
  uint32_t sum = 0u;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 v = gv[(c + lane) & 15];
    sum += (v.x + v.y) + (v.z + v.w);
  }
  const uint32_t incl = warp_incl_sum(sum);
  const unsigned hit = __ballot_sync(0xffffffffu, incl - sum < rem && rem <= incl);
  const int src = __ffs(hit) - 1;
  const uint32_t gabove = __shfl_sync(0xffffffffu, incl - sum, src);
  const int top = 64 * (31 - src) + 63 - 2 * lane;  // this lane's two bins: top, top - 1
  const uint32_t c0 = h[top], c1 = h[top - 1];
  const uint32_t pair = c0 + c1;
  const uint32_t pincl = warp_incl_sum(pair);
  const uint32_t pexcl = gabove + pincl - pair;
  const unsigned phit = __ballot_sync(0xffffffffu, pexcl < rem && rem <= pexcl + pair);
  const int psrc = __ffs(phit) - 1;
  const bool first = pexcl + c0 >= rem;           // the rem-th lies in the higher bin of the pair
  const int bin = first ? top : top - 1;
  const uint32_t bab = first ? pexcl : pexcl + c0;
  const uint32_t bcnt = first ? c0 : c1;
  *above = __shfl_sync(0xffffffffu, bab, psrc);
  *count = __shfl_sync(0xffffffffu, bcnt, psrc);
  return __shfl_sync(0xffffffffu, bin, psrc);
}

template <int kThreads, int kPer, int kMinBlocks = 1>
__global__ void __launch_bounds__(kThreads, kMinBlocks) select_kernel(const __grid_constant__ GroupParams P) {
  constexpr int kWarps = kThreads / kWarp;
  static_assert(kPer < 32, "row masks are 32-bit");
  static_assert(kThreads * kPer < 65536, "block counts are packed in 16-bit halves");
  pdl_wait();
  __shared__ __align__(16) uint32_t hist[2][kBins];   // this pass's histogram and the next one's
  __shared__ uint32_t s_red[2][32];               // per-warp min / max
  __shared__ uint32_t s_cnt[32];                  // per-warp totals of the admission counts
  __shared__ uint32_t s_prefix, s_rem, s_nbin;
  __shared__ int s_first, s_old_kept;
  __shared__ int s_kb[kMaxWaitChunks];            // per source chunk holding kept rows: survivors before it
  extern __shared__ int32_t s_map[];              // [budget] source row of each destination
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = s.flag_stride - 1;
  const int n = s.k + s.m;
  const int lo = s.n_sink, hi = n - s.recent;
  const int q = s.budget - (n - (hi - lo));      // unprotected rows to keep (>= 1)
  const float* old_score = L.score_st + (size_t)bh * s.cap;
  const float* new_score = L.new_score + (size_t)bh * s.new_stride;
  const int i0 = tid * kPer;
  auto clampj = [&](int r) { return min(max(r - i0, 0), kPer); };
  const uint32_t valid = bit_range(0, clampj(n));          // rows below n
  const uint32_t cand = bit_range(clampj(lo), clampj(hi)); // unprotected rows
  const uint32_t prot = valid & ~cand;
  const uint32_t old = bit_range(0, clampj(s.k));          // rows kept before the call

  auto score_at = [&](int i) { return i < n ? (i < s.k ? old_score[i] : new_score[i - s.k]) : 0.f; };
  auto to_key = [&](float x) { return order_key(s.keep_low ? -x : x); };
  uint32_t key[kPer];
  bool vec = false;
  if constexpr (kPer % 4 == 0) {
    // 16-byte loads when no group of 4 rows straddles k and both score planes are 16-byte aligned
    vec = ((s.k | s.cap | s.new_stride) & 3) == 0 &&
          ((reinterpret_cast<uintptr_t>(L.score_st) | reinterpret_cast<uintptr_t>(L.new_score)) & 15) == 0;
  }
  if (vec) {
#pragma unroll
    for (int g = 0; g < kPer / 4; ++g) {
      const int i = i0 + 4 * g;
      float4 v;
      if (i + 4 <= n) {
        v = i < s.k ? *reinterpret_cast<const float4*>(old_score + i)
                    : *reinterpret_cast<const float4*>(new_score + (i - s.k));
      } else {
        v = make_float4(score_at(i), score_at(i + 1), score_at(i + 2), score_at(i + 3));
      }
      key[4 * g] = to_key(v.x);
      key[4 * g + 1] = to_key(v.y);
      key[4 * g + 2] = to_key(v.z);
      key[4 * g + 3] = to_key(v.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kPer; ++j) key[j] = to_key(score_at(i0 + j));
  }
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (cand & (1u << j)) {
      kmin = min(kmin, key[j]);
      kmax = max(kmax, key[j]);
    }
  }
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  for (int j = tid; j < s.flag_stride; j += kThreads) flags[j] = 0;   // flags and chunk counter
  for (int b = tid; b < kBins; b += kThreads) hist[0][b] = 0u;
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    s_red[0][warp] = kmin;
    s_red[1][warp] = kmax;
  }
  if (tid == 0) {
    s_first = s.k;
    s_old_kept = 0;
  }
  __syncthreads();
  const uint32_t all_min = __reduce_min_sync(0xffffffffu, lane < kWarps ? s_red[0][lane] : 0xffffffffu);
  const uint32_t all_max = __reduce_max_sync(0xffffffffu, lane < kWarps ? s_red[1][lane] : 0u);
  // every unprotected key shares the top `common` bits
  const int common = all_min == all_max ? 32 : __clz(all_min ^ all_max);
  uint32_t mask = common == 0 ? 0u : (common == 32 ? 0xffffffffu : ~(0xffffffffu >> common));
  uint32_t prefix = all_min & mask, rem = (uint32_t)q, nbin = (uint32_t)(hi - lo);
  int low = 32 - common;                          // unresolved low bits
  int cur = 0;
  while (low > 0 && rem < nbin) {
    const int w = low < kDigitBits ? low : kDigitBits;
    const int shift = low - w;
    const uint32_t dmask = (1u << w) - 1u;
    uint32_t* h = hist[cur];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if ((cand & (1u << j)) && (key[j] & mask) == prefix) atomicAdd(&h[(key[j] >> shift) & dmask], 1u);
    for (int b = tid; b < kBins; b += kThreads) hist[cur ^ 1][b] = 0u;   // the next pass's histogram
    __syncthreads();
    if (warp == 0) {
      uint32_t above, count;
      const int bin = warp_find_bin(h, rem, &above, &count);
      if (lane == 0) {
        s_prefix = prefix | ((uint32_t)bin << shift);
        s_rem = rem - above;
        s_nbin = count;
      }
    }
    __syncthreads();
    prefix = s_prefix;
    rem = s_rem;
    nbin = s_nbin;
    mask |= dmask << shift;
    low = shift;
    cur ^= 1;
  }
  const uint32_t eq_quota = rem;                  // rows of the final bin admitted in index order

  // rows kept outright (protected, or masked key above the prefix) and rows of the final bin
  uint32_t gt = prot, eq = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (cand & (1u << j)) {
      const uint32_t mk = key[j] & mask;
      if (mk > prefix) gt |= 1u << j;
      else if (mk == prefix) eq |= 1u << j;
    }
  }
  const uint32_t n_gt = (uint32_t)__popc(gt), n_eq = (uint32_t)__popc(eq);
  const uint32_t packed = n_gt | (n_eq << 16);
  const uint32_t pincl = warp_incl_sum(packed);
  if (lane == 31) s_cnt[warp] = pincl;
  __syncthreads();
  const uint32_t wtot = lane < kWarps ? s_cnt[lane] : 0u;
  const uint32_t wbefore = __shfl_sync(0xffffffffu, warp_incl_sum(wtot) - wtot, warp);
  const uint32_t before = wbefore + pincl - packed;
  const uint32_t eq_before = before >> 16;
  const uint32_t dest = (before & 0xffffu) + min(eq_quota, eq_before);
  // the first r rows of the final bin are admitted
  const uint32_t r = eq_quota > eq_before ? min(n_eq, eq_quota - eq_before) : 0u;
  uint32_t eq_keep = eq;
  if (r < n_eq) {
    uint32_t rest = eq;
    for (uint32_t t = 0; t < r; ++t) rest &= rest - 1u;
    eq_keep = eq & ~rest;
  }
  const uint32_t keep = gt | eq_keep;

  {
    uint32_t kb = keep;
    uint32_t d = dest;
    while (kb) {
      const int j = __ffs(kb) - 1;
      kb &= kb - 1u;
      if (d < (uint32_t)s.budget) s_map[d] = i0 + j;
      else raise_device_error(P.err, kDevBadIndex);
      ++d;
    }
  }
  // kept rows below k. Survivors keep their order, so the kept rows of source chunk c take the
  // destinations [kb(c), kb(c + 1)), kb(c) being the survivors before the chunk's first row (and
  // kb at k the kept rows that survive); the thread holding a chunk's first row records kb(c).
  const int chunk_shift = __ffs(s.chunk) - 1;     // compaction chunks are a power of two
  for (int c0 = ((i0 + s.chunk - 1) >> chunk_shift) << chunk_shift; c0 < min(i0 + kPer, s.k); c0 += s.chunk)
    s_kb[c0 >> chunk_shift] = (int)(dest + (uint32_t)__popc(keep & bit_range(0, c0 - i0)));
  const uint32_t old_keep = keep & old;
  const uint32_t drop = old & ~keep;
  // the first dropped kept row and the survivor count: one shared atomic per warp
  const int wfirst = __reduce_min_sync(0xffffffffu, drop ? i0 + __ffs(drop) - 1 : s.k);
  const uint32_t wkept = __reduce_add_sync(0xffffffffu, (uint32_t)__popc(old_keep));
  if (lane == 0) {
    if (wfirst < s.k) atomicMin(&s_first, wfirst);
    if (wkept) atomicAdd(&s_old_kept, (int)wkept);
  }
  __syncthreads();
  int32_t* src_map = L.src_map + (size_t)bh * s.cap;
  for (int d = tid; d < s.budget; d += kThreads) src_map[d] = s_map[d];
  if (tid == 0) L.meta[bh] = make_int2(s_first, s_old_kept);
  if (s.k > 0) {
    // wait ranges of the compaction: the kept rows of source chunk c are read by the destination
    // chunks [kb(c) / C, (kb(c + 1) - 1) / C]; those below c must read them before chunk c is
    // overwritten (empty: hi < lo)
    int2* out = L.waits + (size_t)bh * chunks;
    const int old_chunks = (s.k + s.chunk - 1) >> chunk_shift;
    for (int c = tid; c < chunks; c += kThreads) {
      int2 wr = make_int2(0x7fffffff, -1);
      if (c < old_chunks) {
        const int a = s_kb[c], b = c + 1 < old_chunks ? s_kb[c + 1] : s_old_kept;
        if (b > a) {
          const int lo_c = a >> chunk_shift, hi_c = min((b - 1) >> chunk_shift, c - 1);
          if (lo_c <= hi_c) wr = make_int2(lo_c, hi_c);
        }
      }
      out[c] = wr;
    }
  }
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

// The register variants take budget words of dynamic shared memory (budget < n <= kThreads * kPer).
template <int kThreads, int kPer, int kMinBlocks>
cudaError_t allow_map(cudaError_t e) {
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(select_kernel<kThreads, kPer, kMinBlocks>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(kThreads * kPer * sizeof(int32_t)));
}

cudaError_t prepare_select() {
  // The shared-memory variant serves the largest row counts. The attributes are
  // always the compiled maxima: they are per function and device, so a smaller
  // value set for one cache would break launches of a larger one.
  const int bytes = (int)(EVICT_MAX_SELECT_ROWS * sizeof(uint32_t));
  cudaError_t e = cudaFuncSetAttribute(select_smem_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  e = allow_map<256, 4, 1>(e);
  e = allow_map<256, 8, 1>(e);
  e = allow_map<512, 16, 2>(e);
  e = allow_map<1024, 8, 1>(e);
  e = allow_map<1024, 12, 1>(e);
  e = allow_map<1024, 17, 1>(e);
  return allow_map<1024, 24, 1>(e);
}

cudaError_t launch_select(const GroupParams& P, cudaStream_t st) {
  const int n = P.s.k + P.s.m;
  const dim3 grid(P.s.n_layers * P.s.batch * P.s.heads);
  const size_t map = (size_t)P.s.budget * sizeof(int32_t);   // register variants: the shared src_map
  if (n <= 256 * 4) return launch(select_kernel<256, 4>, grid, dim3(256), map, st, P);
  if (n <= 256 * 8) return launch(select_kernel<256, 8>, grid, dim3(256), map, st, P);
  if (n <= 512 * 16) {
    // more (b, h) units than SMs: 512-thread CTAs, two per SM, keep every unit in one wave
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((int)grid.x > sms && (int)grid.x <= 2 * sms)
      return launch(select_kernel<512, 16, 2>, grid, dim3(512), map, st, P);
  }
  if (n <= 1024 * 8) return launch(select_kernel<1024, 8>, grid, dim3(1024), map, st, P);
  // the fewest keys per thread that hold n: less serial work per pass, no register spills
  if (n <= 1024 * 12) return launch(select_kernel<1024, 12>, grid, dim3(1024), map, st, P);
  if (n <= 1024 * 17) return launch(select_kernel<1024, 17>, grid, dim3(1024), map, st, P);
  if (n <= 1024 * 24) return launch(select_kernel<1024, 24>, grid, dim3(1024), map, st, P);
  return launch(select_smem_kernel<1024>, grid, dim3(1024), (size_t)n * sizeof(uint32_t), st, P);
}

}  // namespace evict
