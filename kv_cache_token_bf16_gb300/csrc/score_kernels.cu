// Score kernels: fused per-key score (KNorm norm / Q-Filters projection) and
// the score + append path used while the cache stays within budget.
//
// Sources: "L2Norm — Intrinsic Key-Norm Eviction", §How it works step 1 (fp32
// L2 norm of each incoming key, computed once at insertion); "Q-Filters —
// Query-Agnostic Projection Eviction", §How it works step 3 (score =
// sign * (key . filter) in fp32, once) and §Metal kernels (fp32 accumulation
// over the stored keys).
//
// Every key is scored in the canonical evaluation order of score.cuh.
#include "common.cuh"
#include "launch.h"
#include "params.h"
#include "score.cuh"
#include "tcgen05.cuh"

namespace evict {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kRowsPerHalfWarp = 4;
constexpr int kScoreRowsPerCta = (kScoreThreads / 16) * kRowsPerHalfWarp;   // 64

// ---------------------------------------------------------------------------
// Score: one CTA covers 64 incoming rows of one (layer, b, h); writes new_score.
// grid = (ceil(m / 64), n_layers * B * H)
// ---------------------------------------------------------------------------
template <bool kBf16, int kMethod>
__global__ void __launch_bounds__(kScoreThreads) score_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.y;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  const int c = threadIdx.x & 15, hw = threadIdx.x >> 4;
  float f[8];
  load_filter<kMethod>(L.filters, filter_row(s, bh), c, f);
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
  pdl_wait();
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.y;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, b = bh / s.heads;
  constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  constexpr int kLaneBytes = kRowBytes / 16;
  const int c = threadIdx.x & 15, hw = threadIdx.x >> 4;
  float f[8];
  load_filter<kMethod>(L.filters, filter_row(s, bh), c, f);
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
        L.score_st[dst] = s.zero_scores ? 0.f : sigma;     // zero: no filter frozen yet
        L.pos_st[dst] = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      }
    }
  }
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  return launch_pdl(kernel, grid, block, smem, st, nullptr, P);
}

}  // namespace

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

}  // namespace evict

namespace evict {
namespace {

// ---------------------------------------------------------------------------
// Single eviction, fused ("L2Norm — Intrinsic Key-Norm Eviction" and
// "Q-Filters — Query-Agnostic Projection Eviction", §How it works: score the
// incoming rows once, keep the budget best with the protected rows forced,
// compact in temporal order). Used when the concatenation exceeds the budget
// by exactly one row (decode steps): the evicted row is the unprotected row
// of lowest priority, the last one in (priority desc, index asc) order, i.e.
// the largest index among the lowest keys; with tie_low (the per-token
// argmin of "CurDKV-adapted — Value-Aware Leverage-Score Eviction", §How it
// works step 5) the smallest index among them. Every row after it moves down
// by one. One CTA per (layer, b, h):
//   1. score the m incoming rows (same canonical order as score_kernel); the
//      kCurDKV variant (CurDKV and H2O per-token steps) takes the scores the
//      attention pipeline left in new_score instead;
//   2. block-wide max of (~key << 32 | tag) over the unprotected rows, the
//      tag being the index (or its complement with tie_low);
//   3. destinations [min(e, k), n - 1) take row d below e and row d + 1 from
//      e on: the kept rows behind e stream through a shared-memory ring of
//      bulk copies (step 3 below), positions and scores through shared
//      memory, then the incoming rows are copied from the block.
// grid = n_layers * B * H, block = 256.
// ---------------------------------------------------------------------------
constexpr int kE1Threads = 256;
constexpr int kE1Warps = kE1Threads / 32;
constexpr int kE1MaxBlock = 64;          // incoming rows scored by one CTA
constexpr int kE1Stages = 3;             // bulk-copy ring stages
constexpr int kE1StageBytes = 32768;     // one chunk of K rows and the same rows of V
constexpr int kE1PsChunk = 1024;         // positions / scores moved per shared-memory round
constexpr int kE1Smem = kE1Stages * kE1StageBytes;

// Bounded wait on a bulk-copy barrier (the thread sleeps between polls; 2 s at most); raises
// the device error on timeout.
__device__ __forceinline__ bool e1_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_ns();
  do {
    if (tc::mbar_try_wait_sleep(bar, parity, 20000)) return true;
  } while (tc::global_ns() - t0 < 2000000000ull);
  raise_device_error(err, kDevWaitTimeout);
  return false;
}

template <bool kBf16, int kMethod>
__global__ void __launch_bounds__(kE1Threads, 2) evict1_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  extern __shared__ __align__(128) unsigned char e1_smem[];   // kE1Stages x (K chunk, V chunk)
  __shared__ float s_new[kE1MaxBlock];
  __shared__ unsigned long long s_best[kE1Warps];
  __shared__ uint64_t s_bar[kE1Stages];
  __shared__ int32_t s_pos[kE1PsChunk];
  __shared__ float s_sc[kE1PsChunk];
  const Shape& s = P.s;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, b = bh / s.heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  const int n = s.k + s.m;                              // = budget + 1
  const size_t plane = (size_t)bh * s.cap;
  const char* kin = static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes;
  const char* vin = static_cast<const char*>(L.v_in) + (size_t)bh * s.m * kRowBytes;
  if (tid == 0)
    for (int i = 0; i < kE1Stages; ++i) tc::mbar_init(&s_bar[i], 1);

  // the kept rows' candidates first (their loads overlap the scoring below)
  const int lo = s.n_sink, hi = n - s.recent;
  // (~key << 32 | tag), largest = evicted; the tag is the index, or its complement when equal
  // scores evict the lower index (tie_low)
  const uint32_t tag_mask = s.tie_low ? 0xffffffffu : 0u;
  unsigned long long best = 0ull;
  for (int i = lo + tid; i < min(hi, s.k); i += kE1Threads) {
    const float sc = L.score_st[plane + i];
    const uint32_t key = order_key(s.keep_low ? -sc : sc);
    const unsigned long long v = ((unsigned long long)(~key) << 32) | ((uint32_t)i ^ tag_mask);
    best = v > best ? v : best;
  }
  // 1. scores of the incoming rows (half-warp per row); given by the caller for kCurDKV
  if constexpr (kMethod == kCurDKV) {
    for (int t = tid; t < s.m; t += kE1Threads) s_new[t] = L.new_score[(size_t)bh * s.new_stride + t];
  } else {
    const int c = tid & 15, hw = tid >> 4;
    float f[8];
    load_filter<kMethod>(L.filters, filter_row(s, bh), c, f);
    for (int t0 = 0; t0 < s.m; t0 += kE1Threads / 16) {
      const int t = t0 + hw;
      RowLoad<kBf16> ld;
      if (t < s.m) ld.load(kin + (size_t)t * kRowBytes, c); else ld.zero();
      float x[8];
      ld.widen(x);
      const float sigma = canonical_score<kMethod>(x, f, s.sign);
      if (c == 0 && t < s.m) s_new[t] = sigma;
    }
  }
  __syncthreads();

  // 2. the evicted row: largest (~key, index) over the unprotected rows
  for (int i = max(lo, s.k) + tid; i < hi; i += kE1Threads) {
    const uint32_t key = order_key(s.keep_low ? -s_new[i - s.k] : s_new[i - s.k]);
    const unsigned long long v = ((unsigned long long)(~key) << 32) | ((uint32_t)i ^ tag_mask);
    best = v > best ? v : best;
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, best, o);
    best = w > best ? w : best;
  }
  if (lane == 0) s_best[warp] = best;
  __syncthreads();
  unsigned long long all = s_best[0];
#pragma unroll
  for (int w = 1; w < kE1Warps; ++w) all = s_best[w] > all ? s_best[w] : all;
  const int e = (int)((uint32_t)all ^ tag_mask);         // lo <= e < hi

  // 3. destinations [min(e, k), n - 1): d takes source d below e and d + 1
  // from e on. Kept rows behind e move down by one row in place: one thread
  // streams them through a shared-memory ring with bulk copies (every later
  // chunk's sources lie above every earlier chunk's destinations, so the
  // loads may run ahead and only the stores keep their order). Meanwhile
  // warps 1-7 move positions and scores through shared memory chunk by
  // chunk; the incoming rows' K / V follow once the ring has drained.
  const int d_begin = min(e, s.k), d_end = n - 1;
  auto srow = [&](int d) { return d < e ? d : d + 1; };
  const int R = e < s.k ? s.k - 1 - e : 0;              // kept rows that move
  if (warp == 0) {
    if (lane == 0 && R > 0) {
      constexpr int kC = kE1StageBytes / 2 / kRowBytes;   // rows per chunk
      const int nch = (R + kC - 1) / kC;
      const char* kplane = static_cast<const char*>(L.kst) + plane * kRowBytes;
      const char* vplane = static_cast<const char*>(L.vst) + plane * kRowBytes;
      const uint32_t ring = tc::smem_u32(e1_smem);
      bool ok = true;
      auto issue_load = [&](int i) {
        const int r0 = e + 1 + i * kC, rows = min(kC, R - i * kC);
        const uint32_t bytes = (uint32_t)(rows * kRowBytes), st = (uint32_t)(i % kE1Stages);
        tc::mbar_arrive_expect_tx(&s_bar[st], 2 * bytes);
        tc::bulk_load(ring + st * kE1StageBytes, kplane + (size_t)r0 * kRowBytes, bytes, &s_bar[st]);
        tc::bulk_load(ring + st * kE1StageBytes + kE1StageBytes / 2, vplane + (size_t)r0 * kRowBytes, bytes,
                      &s_bar[st]);
      };
      const int pre = min(kE1Stages, nch);
      for (int i = 0; i < pre; ++i) issue_load(i);
      int waited = 0;
      for (int i = 0; i < nch && ok; ++i) {
        const int st = i % kE1Stages;
        ok = e1_wait(&s_bar[st], (uint32_t)((i / kE1Stages) & 1), P.err);
        if (!ok) break;
        waited = i + 1;
        const int r0 = e + 1 + i * kC, rows = min(kC, R - i * kC);
        const uint32_t bytes = (uint32_t)(rows * kRowBytes);
        char* kd = static_cast<char*>(L.kst) + (plane + r0 - 1) * kRowBytes;
        char* vd = static_cast<char*>(L.vst) + (plane + r0 - 1) * kRowBytes;
        tc::bulk_store(kd, ring + st * kE1StageBytes, bytes);
        tc::bulk_store(vd, ring + st * kE1StageBytes + kE1StageBytes / 2, bytes);
        tc::bulk_commit();
        if (i >= 1 && i - 1 + kE1Stages < nch) {         // refill the previous chunk's stage
          tc::bulk_wait_read<1>();
          issue_load(i - 1 + kE1Stages);
        }
      }
      // loads issued but not consumed (only after a failed wait) land before exit
      const int issued = min(nch, waited >= 1 ? waited + kE1Stages - 1 : pre);
      for (int i = waited; i < issued; ++i) e1_wait(&s_bar[i % kE1Stages], (uint32_t)((i / kE1Stages) & 1), P.err);
      tc::bulk_wait_all();
    }
    __syncwarp();
  } else {
    // positions and scores: read a chunk of sources, then write it (in order)
    constexpr int kPsThreads = kE1Threads - 32;
    for (int c0 = d_begin; c0 < d_end; c0 += kE1PsChunk) {
      const int c1 = min(d_end, c0 + kE1PsChunk);
      for (int d = c0 + tid - 32; d < c1; d += kPsThreads) {
        const int sr = srow(d);
        if (sr < s.k) {
          s_pos[d - c0] = L.pos_st[plane + sr];
          s_sc[d - c0] = L.score_st[plane + sr];
        } else {
          const int t = sr - s.k;
          s_pos[d - c0] = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
          s_sc[d - c0] = s_new[t];
        }
      }
      tc::named_sync(1, kPsThreads);
      for (int d = c0 + tid - 32; d < c1; d += kPsThreads) {
        L.pos_st[plane + d] = s_pos[d - c0];
        L.score_st[plane + d] = s_sc[d - c0];
      }
      tc::named_sync(1, kPsThreads);
    }
  }
  __syncthreads();
  // incoming rows: source k + t (t != e - k) to destination k + t (before e) or k + t - 1
  {
    constexpr int kVpr = kRowBytes / 16;
    for (int idx = tid; idx < s.m * kVpr * 2; idx += kE1Threads) {
      const int t = idx / (kVpr * 2), rem = idx - t * kVpr * 2;
      const int sr = s.k + t;
      if (sr == e) continue;
      const bool is_v = rem >= kVpr;
      const int c = is_v ? rem - kVpr : rem;
      const int d = sr < e ? sr : sr - 1;
      const char* src = (is_v ? vin : kin) + (size_t)t * kRowBytes;
      char* dst = static_cast<char*>(is_v ? L.vst : L.kst) + (plane + d) * kRowBytes;
      reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
    }
  }
  if (tid == 0) L.meta[bh] = make_int2(min(e, s.k), e < s.k ? s.k - 1 : s.k);
}

}  // namespace

int evict1_max_block() { return kE1MaxBlock; }

cudaError_t prepare_evict1() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(evict1_kernel<true, kKNorm>, cudaFuncAttributeMaxDynamicSharedMemorySize, kE1Smem)) ||
      (e = cudaFuncSetAttribute(evict1_kernel<false, kKNorm>, cudaFuncAttributeMaxDynamicSharedMemorySize, kE1Smem)) ||
      (e = cudaFuncSetAttribute(evict1_kernel<true, kQFilters>, cudaFuncAttributeMaxDynamicSharedMemorySize, kE1Smem)) ||
      (e = cudaFuncSetAttribute(evict1_kernel<false, kQFilters>, cudaFuncAttributeMaxDynamicSharedMemorySize, kE1Smem)) ||
      (e = cudaFuncSetAttribute(evict1_kernel<true, kCurDKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kE1Smem)))
    return e;
  return cudaSuccess;
}

cudaError_t launch_evict1(const GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const dim3 grid(P.s.n_layers * P.s.batch * P.s.heads);
  const bool bf = dtype_bytes == 2;
  if (P.s.method == kKNorm)
    return launch(bf ? evict1_kernel<true, kKNorm> : evict1_kernel<false, kKNorm>, grid, kE1Threads, kE1Smem, st, P);
  if (P.s.method >= kCurDKV)          // CurDKV and H2O: scores already in new_score, bf16 storage
    return launch(evict1_kernel<true, kCurDKV>, grid, kE1Threads, kE1Smem, st, P);
  return launch(bf ? evict1_kernel<true, kQFilters> : evict1_kernel<false, kQFilters>, grid, kE1Threads, kE1Smem, st,
                P);
}

}  // namespace evict
