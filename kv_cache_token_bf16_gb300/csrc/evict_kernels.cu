// Score, protected top-k selection and order-preserving compaction kernels.
//
// Method sources (the three documentation pages):
//  * "L2Norm — Intrinsic Key-Norm Eviction", §How it works: fp32 L2 norm of
//    each incoming key, once; over budget keep the budget lowest (or highest)
//    norms with sinks / recent window forced, temporal order kept.
//  * "Q-Filters — Query-Agnostic Projection Eviction", §How it works step 3:
//    score = sign * (key . filter) in fp32, once; §Metal kernels: the tie
//    rule (strictly-greater rows always, equal rows lowest index first,
//    never more than budget) and the compaction that keeps temporal order;
//    §Adaptation notes: keys copied bit-identically, positions not renumbered.
//
// Score evaluation order (fixed so that a key's score is a pure function of
// its bits, independent of block length or launch shape): a half-warp owns
// one key; lane c holds elements 8c..8c+7 and sums their products left to
// right with round-to-nearest multiplies and adds (no FMA contraction), then
// the 16 lane sums are combined by an xor butterfly with strides 8, 4, 2, 1.
// The norm is the IEEE square root of that sum.
#include "common.cuh"
#include "launch.h"
#include "params.h"

namespace evict {

namespace {

constexpr int kScoreThreads = 256;
constexpr int kRowsPerHalfWarp = 4;
constexpr int kScoreRowsPerCta = (kScoreThreads / 16) * kRowsPerHalfWarp;   // 64

// Load the 8 elements lane `c` owns of one key row, widened to fp32.
template <bool kBf16>
struct RowLoad;

template <>
struct RowLoad<true> {
  uint4 r;
  __device__ __forceinline__ void load(const char* row, int c) { r = ld_stream(row + 16 * c); }
  __device__ __forceinline__ void zero() { r = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void widen(float (&x)[8]) const { bf16x8_to_f32(r, x); }
};

template <>
struct RowLoad<false> {
  uint4 a, b;
  __device__ __forceinline__ void load(const char* row, int c) {
    a = ld_stream(row + 32 * c);
    b = ld_stream(row + 32 * c + 16);
  }
  __device__ __forceinline__ void zero() { a = b = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void widen(float (&x)[8]) const {
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  }
};

// Canonical fp32 score of the half-warp's key; every lane returns the same value.
template <int kMethod>
__device__ __forceinline__ float canonical_score(const float (&x)[8], const float (&f)[8], float sign) {
  float a;
  if (kMethod == kKNorm) {
    a = __fmul_rn(x[0], x[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j) a = __fadd_rn(a, __fmul_rn(x[j], x[j]));
  } else {
    a = __fmul_rn(x[0], f[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j) a = __fadd_rn(a, __fmul_rn(x[j], f[j]));
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
  if (kMethod == kKNorm) return __fsqrt_rn(a);
  return __fmul_rn(sign, a);
}

template <int kMethod>
__device__ __forceinline__ void load_filter(const float* filters, int h, int c, float (&f)[8]) {
  if (kMethod == kQFilters) {
    const float4* fp = reinterpret_cast<const float4*>(filters + h * kHeadDim + 8 * c);
    float4 a = fp[0], b = fp[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = 0.f;
  }
}

// ---------------------------------------------------------------------------
// Score: one CTA covers 64 incoming rows of one (layer, b, h); writes new_score.
// grid = (ceil(m / 64), n_layers * B * H)
// ---------------------------------------------------------------------------
template <bool kBf16, int kMethod>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const __grid_constant__ GroupParams P) {
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.y;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, h = bh % s.heads;
  constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  const int c = threadIdx.x & 15, hw = threadIdx.x >> 4;
  float f[8];
  load_filter<kMethod>(L.filters, h, c, f);
  const char* base = static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes;
  const int row0 = blockIdx.x * kScoreRowsPerCta + hw;
  RowLoad<kBf16> ld[kRowsPerHalfWarp];
#pragma unroll
  for (int j = 0; j < kRowsPerHalfWarp; ++j) {
    const int t = row0 + 16 * j;
    if (t < s.m) ld[j].load(base + (size_t)t * kRowBytes, c); else ld[j].zero();
  }
  float* out = L.new_score + (size_t)bh * s.new_stride;
#pragma unroll
  for (int j = 0; j < kRowsPerHalfWarp; ++j) {
    float x[8];
    ld[j].widen(x);
    const float sigma = canonical_score<kMethod>(x, f, s.sign);
    const int t = row0 + 16 * j;
    if (c == 0 && t < s.m) out[t] = sigma;
  }
}

// ---------------------------------------------------------------------------
// Score + append (the concatenation stays within budget): copies each
// incoming K/V row to storage row k + t, with its score and position.
// grid = (ceil(m / 64), n_layers * B * H)
// ---------------------------------------------------------------------------
template <bool kBf16, int kMethod>
__global__ void __launch_bounds__(kScoreThreads) append_kernel(const __grid_constant__ GroupParams P) {
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.y;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, h = bh % s.heads, b = bh / s.heads;
  constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  constexpr int kLaneBytes = kRowBytes / 16;
  const int c = threadIdx.x & 15, hw = threadIdx.x >> 4;
  float f[8];
  load_filter<kMethod>(L.filters, h, c, f);
  const char* kin = static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes;
  const char* vin = static_cast<const char*>(L.v_in) + (size_t)bh * s.m * kRowBytes;
  char* kout = static_cast<char*>(L.kst) + ((size_t)bh * s.cap + s.k) * kRowBytes;
  char* vout = static_cast<char*>(L.vst) + ((size_t)bh * s.cap + s.k) * kRowBytes;
  const int row0 = blockIdx.x * kScoreRowsPerCta + hw;
#pragma unroll
  for (int j = 0; j < kRowsPerHalfWarp; ++j) {
    const int t = row0 + 16 * j;
    RowLoad<kBf16> kr, vr;
    if (t < s.m) {
      kr.load(kin + (size_t)t * kRowBytes, c);
      vr.load(vin + (size_t)t * kRowBytes, c);
    } else {
      kr.zero();
      vr.zero();
    }
    float x[8];
    kr.widen(x);
    const float sigma = canonical_score<kMethod>(x, f, s.sign);
    if (t < s.m) {
      // kLaneBytes = 16 (bf16) or 32 (fp32) bytes per lane, contiguous per lane
      uint4* kd = reinterpret_cast<uint4*>(kout + (size_t)t * kRowBytes + kLaneBytes * c);
      uint4* vd = reinterpret_cast<uint4*>(vout + (size_t)t * kRowBytes + kLaneBytes * c);
      if constexpr (kBf16) {
        kd[0] = kr.r;
        vd[0] = vr.r;
      } else {
        kd[0] = kr.a; kd[1] = kr.b;
        vd[0] = vr.a; vd[1] = vr.b;
      }
      if (c == 0) {
        const size_t dst = (size_t)bh * s.cap + s.k + t;
        L.score_st[dst] = sigma;
        L.pos_st[dst] = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      }
    }
  }
}

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

// ---------------------------------------------------------------------------
// Order-preserving in-place compaction.
//
// Destination rows are cut into chunks of kChunk rows; a CTA moves one chunk
// of one (layer, b, h). Every survivor moves to a destination at or below
// its source, so a chunk's writes can only clobber storage rows that lower
// chunks still have to read. Each CTA therefore (1) draws a ticket that
// orders chunks low-to-high (a lower ticket is already running), (2) reads
// its sources into shared memory and publishes a read-done flag (release),
// (3) waits (acquire, bounded) for the lower chunks whose storage sources
// overlap its destination range, and (4) writes. Rows below the first
// eviction never move and are not touched. Incoming survivors are read
// straight from the caller's K/V blocks.
// ---------------------------------------------------------------------------
constexpr int kCompactThreads = 256;

template <int kRowBytes, int kChunk>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ GroupParams P) {
  constexpr int kVpr = kRowBytes / 16;   // 16-byte vectors per row
  __shared__ uint4 sk[kChunk * kVpr];
  __shared__ uint4 sv[kChunk * kVpr];
  __shared__ int32_t spos[kChunk];
  __shared__ float sscore[kChunk];
  __shared__ int s_ticket, s_abort;
  const Shape& s = P.s;
  const int tid = threadIdx.x;
  if (tid == 0) {
    const int t = atomicAdd(P.ticket, 1);
    if (t == P.total_ctas - 1) atomicExch(P.ticket, 0);
    s_ticket = t;
    s_abort = 0;
  }
  __syncthreads();
  if (s_ticket >= P.total_ctas) {                // a stale counter: never index past the flags
    if (tid == 0) raise_device_error(P.err, kDevBadIndex);
    return;
  }
  const int bhn = s.batch * s.heads;
  const int units = bhn * s.n_layers;
  const int u = s_ticket % units;
  const int c = s_ticket / units;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, b = bh / s.heads;
  const int2 meta = L.meta[bh];
  const int first = meta.x, old_kept = meta.y;
  const int d_lo = max(c * kChunk, first);
  const int d_hi = min(c * kChunk + kChunk, s.budget);
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  if (d_lo >= d_hi) {
    if (tid == 0) st_release(&flags[c], 1);
    return;
  }
  const int32_t* src = L.src_map + (size_t)bh * s.cap;
  const size_t plane = (size_t)bh * s.cap;
  const char* kst = static_cast<const char*>(L.kst);
  const char* vst = static_cast<const char*>(L.vst);
  const char* kin = static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes;
  const char* vin = static_cast<const char*>(L.v_in) + (size_t)bh * s.m * kRowBytes;
  const int rows = d_hi - d_lo;
  const int n_rows = s.k + s.m;
  for (int r = tid; r < rows; r += kCompactThreads) {
    const int sr = src[d_lo + r];
    if (sr < 0 || sr >= n_rows) s_abort = 1;
  }
  __syncthreads();
  if (s_abort) {                                  // corrupt map: record it, move nothing
    if (tid == 0) {
      raise_device_error(P.err, kDevBadIndex);
      st_release(&flags[c], 1);
    }
    return;
  }

  // (2) read phase
  for (int idx = tid; idx < rows * kVpr; idx += kCompactThreads) {
    const int r = idx / kVpr, vec = idx - r * kVpr;
    const int sr = src[d_lo + r];
    const char* kp;
    const char* vp;
    if (sr < s.k) {
      kp = kst + (plane + sr) * kRowBytes;
      vp = vst + (plane + sr) * kRowBytes;
    } else {
      kp = kin + (size_t)(sr - s.k) * kRowBytes;
      vp = vin + (size_t)(sr - s.k) * kRowBytes;
    }
    sk[idx] = reinterpret_cast<const uint4*>(kp)[vec];
    sv[idx] = reinterpret_cast<const uint4*>(vp)[vec];
  }
  for (int r = tid; r < rows; r += kCompactThreads) {
    const int sr = src[d_lo + r];
    if (sr < s.k) {
      spos[r] = L.pos_st[plane + sr];
      sscore[r] = L.score_st[plane + sr];
    } else {
      const int t = sr - s.k;
      spos[r] = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      sscore[r] = L.new_score[(size_t)bh * s.new_stride + t];
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    st_release(&flags[c], 1);
    // (3) wait for lower chunks whose storage sources overlap [d_lo, d_hi)
    for (int j = c - 1; j >= 0; --j) {
      if (j * kChunk + kChunk <= first) break;             // this and all lower chunks read nothing
      const int j_lo = max(j * kChunk, first);
      const int j_hi = min(j * kChunk + kChunk, old_kept); // storage-sourced destinations of chunk j
      if (j_lo >= j_hi) continue;                          // chunk j reads only incoming rows
      if (src[j_hi - 1] < d_lo) break;                     // chunk j (and lower) read below our range
      if (src[j_lo] >= d_hi) continue;                     // chunk j reads above our range
      int spins = 0;
      while (ld_acquire(&flags[j]) == 0) {
        if (++spins > kSpinLimit) {
          raise_device_error(P.err, kDevWaitTimeout);
          s_abort = 1;
          break;
        }
        __nanosleep(100);
      }
      if (s_abort) break;
    }
  }
  __syncthreads();
  if (s_abort) return;

  // (4) write phase
  char* kdst = static_cast<char*>(L.kst) + (plane + d_lo) * kRowBytes;
  char* vdst = static_cast<char*>(L.vst) + (plane + d_lo) * kRowBytes;
  for (int idx = tid; idx < rows * kVpr; idx += kCompactThreads) {
    reinterpret_cast<uint4*>(kdst)[idx] = sk[idx];
    reinterpret_cast<uint4*>(vdst)[idx] = sv[idx];
  }
  for (int r = tid; r < rows; r += kCompactThreads) {
    L.pos_st[plane + d_lo + r] = spos[r];
    L.score_st[plane + d_lo + r] = sscore[r];
  }
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  kernel<<<grid, block, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

int compact_chunk_rows(int dtype_bytes) { return dtype_bytes == 2 ? 32 : 16; }

cudaError_t launch_score(const GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const dim3 grid((P.s.m + kScoreRowsPerCta - 1) / kScoreRowsPerCta, P.s.n_layers * P.s.batch * P.s.heads);
  const bool bf = dtype_bytes == 2;
  if (P.s.method == kKNorm)
    return launch(bf ? score_kernel<true, kKNorm> : score_kernel<false, kKNorm>, grid, kScoreThreads, 0, st, P);
  return launch(bf ? score_kernel<true, kQFilters> : score_kernel<false, kQFilters>, grid, kScoreThreads, 0, st, P);
}

cudaError_t launch_append(const GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const dim3 grid((P.s.m + kScoreRowsPerCta - 1) / kScoreRowsPerCta, P.s.n_layers * P.s.batch * P.s.heads);
  const bool bf = dtype_bytes == 2;
  if (P.s.method == kKNorm)
    return launch(bf ? append_kernel<true, kKNorm> : append_kernel<false, kKNorm>, grid, kScoreThreads, 0, st, P);
  return launch(bf ? append_kernel<true, kQFilters> : append_kernel<false, kQFilters>, grid, kScoreThreads, 0, st, P);
}

cudaError_t prepare_select(int max_rows) {
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)(max_rows * sizeof(uint32_t)));
}

cudaError_t launch_select(const GroupParams& P, cudaStream_t st) {
  const int n = P.s.k + P.s.m;
  return launch(select_kernel, dim3(P.s.n_layers * P.s.batch * P.s.heads), dim3(kSelectThreads),
                (size_t)n * sizeof(uint32_t), st, P);
}

cudaError_t launch_compact(GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const int chunk = compact_chunk_rows(dtype_bytes);
  const int chunks = (P.s.budget + chunk - 1) / chunk;
  P.total_ctas = chunks * P.s.n_layers * P.s.batch * P.s.heads;
  if (dtype_bytes == 2)
    return launch(compact_kernel<kHeadDim * 2, 32>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
  return launch(compact_kernel<kHeadDim * 4, 16>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
}

}  // namespace evict
