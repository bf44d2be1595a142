// CurDKV-adapted block scoring ("CurDKV-adapted — Value-Aware Leverage-Score
// Eviction", §How it works steps 1-4 and §The honesty crux items 1-4).
//
// For every (b, h) with k kept rows and an incoming block of m rows
// (n = k + m rows in total):
//   1. proxy attention: the incoming keys are the queries; query t (row k+t)
//      attends rows i <= k+t with logits (q_t . k_i) / sqrt(D);
//      attn[i] = sum_t softmax_t[i]                       (two tensor-core passes)
//   2. weighted values w_i = attn[i] * v_i and G = W^T W = sum_i w_i w_i^T
//   3. the top r = min(rank_cap, n, D) eigenvectors e_j of G (the right
//      singular vectors of W; lambda_j = s_j^2) and E = trace G = sum_j s_j^2
//   4. leverage l_i = sum_{j<r} (w_i . e_j)^2 / E  (= sum_j (s_j^2/sum s^2) U_ij^2);
//      kept rows accumulate it into their stored score, incoming rows are
//      seeded with it.
// The block is then cut to budget by the shared protected top-k (keep high)
// and compaction.
//
// Kernels:
//   curdkv_lse_kernel      pass 1: per query and key split, running max and sum of
//                          2^logit (tcgen05 MMA, 256 queries x 128 keys per step, pipelined)
//   curdkv_lse_merge_kernel  log2-sum-exp per query from the splits
//   curdkv_colsum_kernel   pass 2: per key, sum over queries of 2^(logit - lse)
//                          (tcgen05 MMA, 256 keys x 128 queries per step, pipelined)
//   curdkv_gram_kernel     partial G over a slice of rows (tcgen05, split bf16)
//   curdkv_eig_kernel      sum of partials (fp64), Householder tridiagonalisation,
//                          multisection bisection for the top r eigenvalues,
//                          inverse iteration, orthonormalisation, back-transform
//   curdkv_leverage_kernel l_i (projections on tcgen05) and the cumulative-score update
//   curdkv_append_kernel   copy of the block when the cache stays within budget
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cfloat>
#include <cmath>
#include <cstring>

#include "api_internal.h"
#include "common.cuh"
#include "launch.h"
#include "params.h"
#include "tcgen05.cuh"

namespace evict {

struct CurdkvState {
  float* lse = nullptr;        // [BH, lse_stride]  log2-sum-exp per query
  float2* lse_part = nullptr;  // [BH, 8, lse_stride] per-split (max, sum)
  int lse_stride = 0;          // max_block rounded up to 4 (16-byte rows)
  int sm_count = 0;
  float* attn = nullptr;       // [BH, rows]        column sums
  float* lev = nullptr;        // [BH, rows]        leverage of the last call
  float* gram_part = nullptr;  // [BH, splits, 128*128]
  float* evec = nullptr;       // [BH, kCurdkvMaxRank, 128]
  float* inv_e = nullptr;      // [BH]
  int rows = 0;                // cap + max_block
  int splits = 0;              // gram partials per (b, h)
  int last_n = 0;              // rows of the last update
};

namespace {

constexpr int kTile = 128;                  // rows of a query or key tile
constexpr int kAttnThreads = 128;           // 4 warps: one TMEM lane per thread
constexpr int kTileBytes = kTile * kHeadDim * 2;
constexpr int kGramRows = 2048;             // rows per Gram partial
constexpr int kEigThreads = 1024;
constexpr int kMbarSpin = 1 << 22;          // bounded MMA wait (well above a tile's time)
constexpr float kLog2e = 1.4426950408889634f;

struct CurdkvParams {
  const void* k_in;      // [BH, m, D] bf16
  const void* v_in;
  const void* kst;       // [BH, cap, D] bf16
  const void* vst;
  int k, m, n, cap, heads, rank;
  float scale2;          // log2(e) / sqrt(D)
  float* lse;
  float2* lse_part;       // [BH, kMaxLseSplit, lse_stride] per-split (max, sum)
  int lse_stride;         // max_block rounded up to 4
  float* attn;
  float* lev;
  int rows;
  float* gram_part;
  int splits;
  float* evec;
  float* inv_e;
  float* score_st;
  float* new_score;
  int new_stride;
  int32_t* pos_st;
  const int32_t* pos_in;
  long long offset;
  int* err;
};

__device__ __forceinline__ const char* key_row(const CurdkvParams& p, int bh, int i) {
  if (i < p.k) return static_cast<const char*>(p.kst) + ((size_t)bh * p.cap + i) * (kHeadDim * 2);
  return static_cast<const char*>(p.k_in) + ((size_t)bh * p.m + (i - p.k)) * (kHeadDim * 2);
}
__device__ __forceinline__ const char* value_row(const CurdkvParams& p, int bh, int i) {
  if (i < p.k) return static_cast<const char*>(p.vst) + ((size_t)bh * p.cap + i) * (kHeadDim * 2);
  return static_cast<const char*>(p.v_in) + ((size_t)bh * p.m + (i - p.k)) * (kHeadDim * 2);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Wait for an MMA commit (bounded); returns false on timeout.
__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity, int* err) {
  for (int spin = 0; spin < kMbarSpin; ++spin)
    if (tc::mbar_try_wait(bar, parity)) return true;
  raise_device_error(err, kDevWaitTimeout);
  return false;
}

// 8 MMAs (K = 128 in steps of 16): D[128 x 128] = A[128 x 128] * B[128 x 128]^T.
__device__ __forceinline__ void issue_tile_mma(uint32_t tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kTile, kTile);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t off = (uint32_t)((s >> 2) * kTile * 128 + (s & 3) * 32);
    tc::mma_bf16(tmem, tc::sw128_desc(a + off), tc::sw128_desc(b + off), idesc, s > 0 ? 1u : 0u);
  }
}

// ---------------------------------------------------------------------------
// Pipelined attention passes. Each CTA holds two fixed 128-row operand tiles
// (256 queries in pass 1, 256 keys in pass 2) and streams the other operand
// through a 3-stage cp.async ring; every streamed tile feeds two 128 x 128
// MMAs. TMEM holds two buffers of two fp32 accumulators (512 columns), so
// the MMAs of tile i+1 run while tile i is read. 512 threads: warp w reads
// TMEM lanes 32*(w%4)..+31 (one accumulator row per thread) and, with
// g = w/4, accumulator g/2, columns 64*(g%2)..+63.
// ---------------------------------------------------------------------------
constexpr int kPipeThreads = 512;
constexpr int kColGroups = 4;                     // column groups of 64 over the two accumulators
constexpr int kStages = 3;
constexpr int kPipeSmem = (2 + kStages) * kTileBytes + 1024;
constexpr int kMaxLseSplit = 8;

// cp.async of one 128-row tile (rows >= row_end are zero) by all threads.
__device__ __forceinline__ void pipe_load_rows(const CurdkvParams& p, int bh, uint32_t tile, int row0, int row_end) {
#pragma unroll
  for (int q = 0; q < kTile * 16 / kPipeThreads; ++q) {
    const int c = threadIdx.x + q * kPipeThreads;
    const int r = c >> 4, j = c & 15;
    const int row = row0 + r;
    const bool ok = row < row_end;
    const char* src = key_row(p, bh, ok ? row : 0) + j * 16;
    tc::cp_async16(tile + tc::sw128_offset(r, j, kTile), src, ok ? 16u : 0u);
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Warp-uniform bounded wait for an MMA commit; every lane returns the same answer.
__device__ __forceinline__ bool warp_wait_mma(uint64_t* bar, uint32_t parity, int* err) {
  bool ok = false;
  for (int spin = 0; spin < kMbarSpin && !ok; ++spin) ok = tc::mbar_try_wait(bar, parity);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) raise_device_error(err, kDevWaitTimeout);
  return ok;
}

// MMAs of one streamed tile into buffer `buf`: accumulator a = fixed tile a x streamed tile.
// `two` = the second fixed tile holds real rows. Pass 1 puts the fixed tiles
// on the A side (rows = queries), pass 2 too (rows = keys).
__device__ __forceinline__ void issue_pair(uint32_t tmem, int buf, uint32_t fixed0, uint32_t streamed, bool two,
                                           uint64_t* bar) {
  tc::fence_after_sync();
  issue_tile_mma(tmem + (uint32_t)(buf * 2 * kTile), fixed0, streamed);
  if (two) issue_tile_mma(tmem + (uint32_t)(buf * 2 * kTile + kTile), fixed0 + kTileBytes, streamed);
  tc::mma_commit(bar);
}

// ---------------------------------------------------------------------------
// Pass 1 (split over keys): for query t of the CTA's 256 and key split s,
//   (m, s) = (max_i x_i, sum_i 2^(x_i - max)),  x_i = scale2 * q_t . k_i,
// over the split's share of the keys i <= k + t. grid = (ceil(m/256), S, B*H).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPipeThreads, 1) curdkv_lse_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  __shared__ float s_m[kColGroups][kTile], s_s[kColGroups][kTile];
  const int t0 = blockIdx.x * 2 * kTile, split = blockIdx.y, n_split = gridDim.y, bh = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 2, a = g >> 1, col0 = 64 * (g & 1);
  const int row = 32 * (warp & 3) + lane;
  const int t = t0 + a * kTile + row;                // this thread's query
  const bool two = t0 + kTile < p.m;                 // the second query tile exists
  const int t_last = min(p.m, t0 + 2 * kTile) - 1;
  const int key_end = p.k + t_last + 1;
  const int n_kt = (key_end + kTile - 1) / kTile;
  const int per = (n_kt + n_split - 1) / n_split;
  const int kt_begin = split * per, kt_end = min(n_kt, kt_begin + per);
  float2* part = p.lse_part + ((size_t)bh * kMaxLseSplit + split) * p.lse_stride;
  if (kt_begin >= kt_end) {                          // nothing to see in this split
    if ((g & 1) == 0 && t < p.m) part[t] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int T = kt_end - kt_begin;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t q_tiles = tc::smem_u32(smem), stage0 = q_tiles + 2 * kTileBytes;
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    s_fail = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 4 * kTile);
  pipe_load_rows(p, bh, q_tiles, p.k + t0, p.k + p.m);                  // queries = incoming rows
  pipe_load_rows(p, bh, q_tiles + kTileBytes, p.k + t0 + kTile, p.k + p.m);
  cp_async_commit();
  pipe_load_rows(p, bh, stage0, kt_begin * kTile, key_end);
  cp_async_commit();
  if (T > 1) pipe_load_rows(p, bh, stage0 + kTileBytes, (kt_begin + 1) * kTile, key_end);
  cp_async_commit();
  cp_async_wait_1();
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  if (tid == 0) issue_pair(tmem, 0, q_tiles, stage0, two, &bar[0]);
  const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
  const bool active = a == 0 || two;                 // warp-uniform: this warp's accumulator exists
  float run_max = -INFINITY, run_sum = 0.f;
  int consumed = 0, issued = 1;
  for (int it = 0; it < T; ++it) {
    if (it + 2 < T) pipe_load_rows(p, bh, stage0 + ((it + 2) % kStages) * kTileBytes, (kt_begin + it + 2) * kTile, key_end);
    cp_async_commit();
    cp_async_wait_1();
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) break;
    if (it + 1 < T) {
      if (tid == 0) issue_pair(tmem, (it + 1) & 1, q_tiles, stage0 + ((it + 1) % kStages) * kTileBytes, two,
                               &bar[(it + 1) & 1]);
      ++issued;
    }
    if (!warp_wait_mma(&bar[it & 1], (uint32_t)((it >> 1) & 1), p.err)) {
      if (lane == 0) s_fail = 1;
      continue;                                      // the next barrier sees s_fail
    }
    ++consumed;
    tc::fence_after_sync();
    if (active) {
      const int i0 = (kt_begin + it) * kTile;
      const bool full = i0 + kTile - 1 <= p.k + t0 + a * kTile;   // every key visible to every query
      const uint32_t acc = tmem + (uint32_t)((it & 1) * 2 * kTile + a * kTile + col0) + tlane;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float v[32];
        tc::tmem_ld32(acc + c0, v);
        if (!full) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (i0 + col0 + c0 + c > p.k + t) v[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mx[c] = fmaxf(fmaxf(v[c], v[c + 8]), fmaxf(v[c + 16], v[c + 24]));
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
        if (mx[0] > -INFINITY) {
          const float nm = fmaxf(run_max, mx[0] * p.scale2);
          float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < 32; ++c) sm[c & 3] += ex2(fmaf(v[c], p.scale2, -nm));
          run_sum = (run_max > -INFINITY ? run_sum * ex2(run_max - nm) : 0.f) + ((sm[0] + sm[1]) + (sm[2] + sm[3]));
          run_max = nm;
        }
      }
    }
    tc::fence_before_sync();
  }
  // a failure can leave MMAs in flight: wait for them (bounded) before freeing TMEM
  if (issued > consumed) warp_wait_mma(&bar[consumed & 1], (uint32_t)((consumed >> 1) & 1), p.err);
  s_m[g][row] = run_max;
  s_s[g][row] = run_sum;
  tc::fence_before_sync();
  __syncthreads();
  if ((g & 1) == 0 && active && !s_fail && t < p.m) {
    const float m0 = s_m[g][row], m1 = s_m[g + 1][row];
    const float mm = fmaxf(m0, m1);
    float ss = 0.f;
    if (mm > -INFINITY)
      ss = (m0 > -INFINITY ? s_s[g][row] * ex2(m0 - mm) : 0.f) + (m1 > -INFINITY ? s_s[g + 1][row] * ex2(m1 - mm) : 0.f);
    part[t] = make_float2(mm, ss);
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 4 * kTile);
}

// Merge the key splits: lse2[t] = log2 sum_s s_s 2^(m_s). grid = ceil(m / 256) x B*H.
__global__ void __launch_bounds__(256) curdkv_lse_merge_kernel(const __grid_constant__ CurdkvParams p, int n_split) {
  const int bh = blockIdx.y, t = blockIdx.x * 256 + threadIdx.x;
  if (t >= p.m) return;
  const float2* part = p.lse_part + (size_t)bh * kMaxLseSplit * p.lse_stride + t;
  float mm = -INFINITY;
  for (int s = 0; s < n_split; ++s) mm = fmaxf(mm, part[(size_t)s * p.lse_stride].x);
  float ss = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float2 v = part[(size_t)s * p.lse_stride];
    if (v.x > -INFINITY) ss += v.y * ex2(v.x - mm);
  }
  p.lse[(size_t)bh * p.lse_stride + t] = mm + log2f(ss);
}

// ---------------------------------------------------------------------------
// Pass 2: attn[i] = sum_{t : k+t >= i} 2^(scale2 * q_t . k_i - lse2[t]).
// The CTA's 256 keys are fixed (MMA operand A); query tiles stream through
// the ring with their lse2 values. grid = (ceil(n / 256), B*H).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPipeThreads, 1) curdkv_colsum_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  __shared__ __align__(16) float s_lse[kStages][kTile];
  __shared__ float s_acc[kColGroups][kTile];
  const int i0 = blockIdx.x * 2 * kTile, bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = warp >> 2, a = g >> 1, col0 = 64 * (g & 1);
  const int row = 32 * (warp & 3) + lane;
  const int i = i0 + a * kTile + row;              // this thread's key
  const int key_end = min(p.n, i0 + 2 * kTile);
  const bool two = i0 + kTile < p.n;               // the second key tile exists
  const int t_first = max(0, i0 - p.k);            // first query that sees a key of the CTA
  const int tq0 = (t_first / kTile) * kTile;
  const int T = (p.m - tq0 + kTile - 1) / kTile;   // >= 1: the last key is seen by the last query
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t k_tiles = tc::smem_u32(smem), stage0 = k_tiles + 2 * kTileBytes;
  const float* lse = p.lse + (size_t)bh * p.lse_stride;
  auto load_stage = [&](int it) {
    const int tq = tq0 + it * kTile, st = it % kStages;
    pipe_load_rows(p, bh, stage0 + st * kTileBytes, p.k + tq, p.k + p.m);
    if (tid < kTile / 4) {
      const bool ok = tq + 4 * tid < p.m;          // values past m are never read
      tc::cp_async16(tc::smem_u32(&s_lse[st][4 * tid]), lse + (ok ? tq + 4 * tid : 0), ok ? 16u : 0u);
    }
  };
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    s_fail = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 4 * kTile);
  pipe_load_rows(p, bh, k_tiles, i0, key_end);
  pipe_load_rows(p, bh, k_tiles + kTileBytes, i0 + kTile, key_end);
  cp_async_commit();
  load_stage(0);
  cp_async_commit();
  if (T > 1) load_stage(1);
  cp_async_commit();
  cp_async_wait_1();
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  if (tid == 0) issue_pair(tmem, 0, k_tiles, stage0, two, &bar[0]);
  const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
  const bool active = a == 0 || two;               // warp-uniform: this warp's accumulator exists
  const int key_base = i0 + a * kTile;             // first key of this warp's accumulator
  float acc4[4] = {0.f, 0.f, 0.f, 0.f};
  int consumed = 0, issued = 1;
  for (int it = 0; it < T; ++it) {
    if (it + 2 < T) load_stage(it + 2);
    cp_async_commit();
    cp_async_wait_1();
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) break;
    if (it + 1 < T) {
      if (tid == 0) issue_pair(tmem, (it + 1) & 1, k_tiles, stage0 + ((it + 1) % kStages) * kTileBytes, two,
                               &bar[(it + 1) & 1]);
      ++issued;
    }
    if (!warp_wait_mma(&bar[it & 1], (uint32_t)((it >> 1) & 1), p.err)) {
      if (lane == 0) s_fail = 1;
      continue;
    }
    ++consumed;
    tc::fence_after_sync();
    if (active) {
      const int tq = tq0 + it * kTile;
      const float* l = s_lse[it % kStages] + col0;
      // every query of the tile exists and sees every key of the accumulator
      const bool full = tq + kTile <= p.m && key_base + kTile - 1 <= p.k + tq;
      const uint32_t acc = tmem + (uint32_t)((it & 1) * 2 * kTile + a * kTile + col0) + tlane;
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        float v[32];
        tc::tmem_ld32(acc + c0, v);
        if (full) {
#pragma unroll
          for (int c = 0; c < 32; ++c) acc4[c & 3] += ex2(fmaf(v[c], p.scale2, -l[c0 + c]));
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int tt = tq + col0 + c0 + c;
            if (tt < p.m && i <= p.k + tt) acc4[c & 3] += ex2(fmaf(v[c], p.scale2, -l[c0 + c]));
          }
        }
      }
    }
    tc::fence_before_sync();
  }
  if (issued > consumed) warp_wait_mma(&bar[consumed & 1], (uint32_t)((consumed >> 1) & 1), p.err);
  s_acc[g][row] = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
  tc::fence_before_sync();
  __syncthreads();
  if ((g & 1) == 0 && active && !s_fail && i < key_end) p.attn[(size_t)bh * p.rows + i] = s_acc[g][row] + s_acc[g + 1][row];
  if (warp == 0) tc::tmem_dealloc(tmem, 4 * kTile);
}

// ---------------------------------------------------------------------------
// Partial Gram of the weighted values on the tensor cores:
//   G_part = sum over the split's rows i of a_i^2 v_i v_i^T
//          = V^T (a^2 V)_hi + V^T (a^2 V)_lo,
// V exact in bf16 and a_i^2 v_i split into two bf16 terms (hi + lo carries
// ~16 significant bits; the dropped lo*lo-free remainder is below 2^-17 of
// each term). The MMA contracts over tokens, so each 128-token tile is
// transposed on the way into shared memory: a thread loads 8 tokens x 8
// features (eight 16-byte rows) and rearranges them with byte permutes into
// 8 features x 8 tokens. grid = (ceil(n / 2048), B*H), block = 128; the next
// tile's loads overlap the running MMAs.
// ---------------------------------------------------------------------------
constexpr int kGramTcSmem = 3 * kTileBytes + 1024;

// 8 x 8 transpose of bf16 values: in[t] holds 8 features of token t, out[f]
// holds 8 tokens of feature f.
__device__ __forceinline__ void transpose8x8(const uint4 (&in)[8], uint4 (&out)[8]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(in);   // w[4*t + k]: features 2k, 2k+1 of token t
#pragma unroll
  for (int f = 0; f < 8; ++f) {
    const uint32_t sel = (f & 1) ? 0x7632u : 0x5410u;
    const int k = f >> 1;
    out[f].x = __byte_perm(w[4 * 0 + k], w[4 * 1 + k], sel);
    out[f].y = __byte_perm(w[4 * 2 + k], w[4 * 3 + k], sel);
    out[f].z = __byte_perm(w[4 * 4 + k], w[4 * 5 + k], sel);
    out[f].w = __byte_perm(w[4 * 6 + k], w[4 * 7 + k], sel);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo_elem, hi_elem);   // .x (low half) = lo_elem
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(kAttnThreads) curdkv_gram_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const int split = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t a_tile = tc::smem_u32(smem), bhi_tile = a_tile + kTileBytes, blo_tile = bhi_tile + kTileBytes;
  const int r_begin = split * kGramRows, r_end = min(p.n, r_begin + kGramRows);
  const float* attn = p.attn + (size_t)bh * p.rows;
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    s_fail = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTile);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  // thread -> two 8x8 blocks of the tile: token block tb, feature blocks fb and fb + 8
  const int tb = tid & 15, fb0 = tid >> 4;
  uint4 raw[2][8];
  float asq[8];
  auto load_tile = [&](int t0) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int row = t0 + 8 * tb + t;
      const bool ok = row < r_end;
      const uint4* src = reinterpret_cast<const uint4*>(value_row(p, bh, ok ? row : r_begin));
      raw[0][t] = ok ? __ldg(src + fb0) : make_uint4(0, 0, 0, 0);
      raw[1][t] = ok ? __ldg(src + fb0 + 8) : make_uint4(0, 0, 0, 0);
      const float a = ok ? attn[row] : 0.f;
      asq[t] = a * a;
    }
  };
  uint32_t parity = 0;
  int pending = 0;                                          // commits not yet waited for
  load_tile(r_begin);
  for (int t0 = r_begin; t0 < r_end; t0 += kTile) {
    if (pending) {                                          // smem tiles are free once the last MMAs finished
      if (!wait_mma(&bar, parity, p.err)) s_fail = 1;
      else pending = 0;
      parity ^= 1u;
      tc::fence_after_sync();
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int fb = fb0 + 8 * h;
      uint4 tr[8];
      transpose8x8(raw[h], tr);
#pragma unroll
      for (int f = 0; f < 8; ++f)
        *reinterpret_cast<uint4*>(smem + tc::sw128_offset(8 * fb + f, tb, kTile)) = tr[f];
      uint4 hi[8], lo[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        float x[8];
        bf16x8_to_f32(raw[h][t], x);
        float y[8], yh[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) y[q] = x[q] * asq[t];
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hw[q] = pack_bf16x2(y[2 * q], y[2 * q + 1]);
          yh[2 * q] = __uint_as_float(hw[q] << 16);
          yh[2 * q + 1] = __uint_as_float(hw[q] & 0xffff0000u);
          lw[q] = pack_bf16x2(y[2 * q] - yh[2 * q], y[2 * q + 1] - yh[2 * q + 1]);
        }
        hi[t] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        lo[t] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      transpose8x8(hi, tr);
#pragma unroll
      for (int f = 0; f < 8; ++f)
        *reinterpret_cast<uint4*>(smem + kTileBytes + tc::sw128_offset(8 * fb + f, tb, kTile)) = tr[f];
      transpose8x8(lo, tr);
#pragma unroll
      for (int f = 0; f < 8; ++f)
        *reinterpret_cast<uint4*>(smem + 2 * kTileBytes + tc::sw128_offset(8 * fb + f, tb, kTile)) = tr[f];
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    if (s_fail) break;
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTile, kTile);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint32_t off = (uint32_t)((st >> 2) * kTile * 128 + (st & 3) * 32);
        const uint64_t ad = tc::sw128_desc(a_tile + off);
        tc::mma_bf16(tmem, ad, tc::sw128_desc(bhi_tile + off), idesc, (t0 > r_begin || st > 0) ? 1u : 0u);
        tc::mma_bf16(tmem, ad, tc::sw128_desc(blo_tile + off), idesc, 1u);
      }
      tc::mma_commit(&bar);
    }
    pending = 1;
    if (t0 + kTile < r_end) load_tile(t0 + kTile);          // overlaps with the MMAs
  }
  // the last commit (also on a failure path, so no MMA is in flight at dealloc)
  if (pending && !wait_mma(&bar, parity, p.err)) s_fail = 1;
  __syncthreads();
  tc::fence_after_sync();
  if (!s_fail) {
    float* out = p.gram_part + ((size_t)bh * p.splits + split) * kHeadDim * kHeadDim + (size_t)tid * kHeadDim;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < kTile; c0 += 32) {
      float v[32];
      tc::tmem_ld32(trow + c0, v);
#pragma unroll
      for (int c = 0; c < 32; c += 4)
        *reinterpret_cast<float4*>(out + c0 + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTile);
}

// ---------------------------------------------------------------------------
// Top-r eigenvectors of G (symmetric, 128 x 128), one CTA of 512 threads per
// (b, h). G is normalised by its trace and held in registers: kGroup threads
// share a row, thread t owning row t/kGroup and the columns c = t%kGroup
// (mod kGroup).
// ---------------------------------------------------------------------------
constexpr int kGroup = kEigThreads / kHeadDim; // threads per row
constexpr int kEigPer = kHeadDim / kGroup;     // columns per thread

struct EigSmem {
  double trace;
  double diag64[kHeadDim];
  float hv[kHeadDim - 2][kHeadDim];   // Householder vector of step j (zeros up to index j)
  float x[2][kHeadDim], pv[2][kHeadDim];
  float gram[kCurdkvMaxRank][kCurdkvMaxRank + 1];
  float d[kHeadDim], e[kHeadDim], e2[kHeadDim], beta[kHeadDim];
  float lam[kCurdkvMaxRank];
  float z[kCurdkvMaxRank][kHeadDim];  // eigenvectors (tridiagonal basis, then original)
  float lu[kCurdkvMaxRank][5][kHeadDim];  // per-vector LU factors: diag^-1, sup1, sup2, mult, pivot flag
  float tnorm;
};

// Number of eigenvalues of the (normalised) tridiagonal T that are <= x.
__device__ __forceinline__ int sturm_count(const EigSmem& s, float x, float pivmin) {
  int cnt = 0;
  float q = s.d[0] - x;
  if (fabsf(q) < pivmin) q = -pivmin;
  if (q <= 0.f) ++cnt;
#pragma unroll 4
  for (int i = 1; i < kHeadDim; ++i) {
    q = s.d[i] - __fdividef(s.e2[i - 1], q) - x;
    if (fabsf(q) < pivmin) q = -pivmin;
    if (q <= 0.f) ++cnt;
  }
  return cnt;
}

__device__ __forceinline__ float hash_unit(int i, int j) {
  uint32_t h = (uint32_t)i * 2654435761u ^ (uint32_t)(j + 1) * 2246822519u;
  h ^= h >> 15;
  h *= 2654435761u;
  h ^= h >> 13;
  return (float)(h & 0xFFFFu) * (1.f / 65536.f) - 0.5f;
}

__global__ void __launch_bounds__(kEigThreads, 1) curdkv_eig_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(16) unsigned char eig_raw[];
  EigSmem& s = *reinterpret_cast<EigSmem*>(eig_raw);
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int n = kHeadDim;
  constexpr int kWarps = kEigThreads / 32;
  const int r = p.rank;
  float* evec_out = p.evec + (size_t)bh * kCurdkvMaxRank * n;
  const int row = tid / kGroup, q4 = tid % kGroup;   // q4: this thread's column class

  // G = sum of the partials in a fixed order: fp32, except the diagonal terms
  // that form E = trace G (fp64; GB300's fp64 rate is low, so only those)
  const int splits_used = (p.n + kGramRows - 1) / kGramRows;
  const float* part = p.gram_part + (size_t)bh * p.splits * n * n + row * n + q4;
  float a[kEigPer];
#pragma unroll
  for (int i = 0; i < kEigPer; ++i) a[i] = 0.f;
  for (int sp = 0; sp < splits_used; ++sp) {        // branch-free so the loads overlap
    const float* src = part + (size_t)sp * n * n;
#pragma unroll
    for (int i = 0; i < kEigPer; ++i) a[i] += src[kGroup * i];
  }
  if (row % kGroup == q4) {                          // this thread holds G[row][row]
    const float* src = p.gram_part + (size_t)bh * p.splits * n * n + row * n + row;
    double diag = 0.0;
    for (int sp = 0; sp < splits_used; ++sp) diag += src[(size_t)sp * n * n];
    s.diag64[row] = diag;
  }
  __syncthreads();
  if (tid == 0) {
    double tr = 0.0;
    for (int i = 0; i < n; ++i) tr += s.diag64[i];
    s.trace = tr;
  }
  __syncthreads();
  if (!(s.trace > 0.0)) {
    for (int el = tid; el < kCurdkvMaxRank * n; el += kEigThreads) evec_out[el] = 0.f;
    if (tid == 0) p.inv_e[bh] = 0.f;
    return;
  }
  if (tid == 0) p.inv_e[bh] = (float)(1.0 / s.trace);
  {
    const float sc = (float)(1.0 / s.trace);     // normalise: eigenvectors unchanged
#pragma unroll
    for (int i = 0; i < kEigPer; ++i) a[i] *= sc;
  }

  // --- Householder tridiagonalisation (registers) ----------------------------
  // a[i] holds column kGroup*(i + base) + q4; every kGroup steps the row
  // shifts left by one (the finished columns drop out), so the column being
  // reduced is always a[0], every register index is a compile-time constant
  // and the loops stop at the last live column (a CTA-uniform bound).
  // Step j works with x = column j below the diagonal, zero-filled up to
  // index j in shared memory; the Householder vector v equals x except
  // v[j+1] = x[j+1] + delta, which enters as one correction term. Each step
  // has two barriers: every warp recomputes the step's scalars from the
  // shared vectors (identical bits in every warp), and the vectors are
  // double-buffered by step parity. Warps whose rows are all finished skip.
  constexpr int kRowsPerWarp = 32 / kGroup;
  int base = 0;
  for (int j = 0; j < n - 2; ++j) {
    float* xj = s.x[j & 1];
    float* pj = s.pv[j & 1];
    if (q4 == j % kGroup) {
      xj[row] = row > j ? a[0] : 0.f;             // column j below the diagonal, zeros above
      if (row == j) s.d[j] = a[0];                // diagonal element j
    }
    __syncthreads();
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) ss = fmaf(xj[32 * k + lane], xj[32 * k + lane], ss);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float x0 = xj[j + 1];
    const float tail = ss - x0 * x0;
    float beta = 0.f, alpha = x0, delta = 0.f;
    if (tail > 0.f) {
      const float sigma = sqrtf(ss);
      alpha = x0 >= 0.f ? -sigma : sigma;
      delta = -alpha;                             // v[j+1] = x0 - alpha
      beta = 1.f / (sigma * (sigma + fabsf(x0)));
    }
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 32 * k + lane;
        const float xv = xj[c];
        s.hv[j][c] = beta == 0.f ? 0.f : (c == j + 1 ? xv + delta : xv);
      }
      if (lane == 0) {
        s.beta[j] = beta;
        s.e[j] = alpha;
      }
    }
    const bool live_rows = warp * kRowsPerWarp + kRowsPerWarp - 1 > j;   // some row of this warp is > j
    // index of column j+1 in this thread's registers, if this thread owns it
    const bool owns_next = q4 == (j + 1) % kGroup;
    const int next_idx = (j + 1) / kGroup - base;      // 0 or 1
    if (beta != 0.f) {
      // p = beta * A v = beta * (A x + A[:, j+1] * delta)
      float acc = 0.f;
      if (live_rows) {
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int i = 0; i < kEigPer; ++i) {
          if (i + base >= kEigPer) break;
          const float xc = xj[kGroup * (i + base) + q4];
          if (i & 1) acc1 = fmaf(a[i], xc, acc1); else acc0 = fmaf(a[i], xc, acc0);
        }
        acc = acc0 + acc1;
        if (owns_next) acc = fmaf(next_idx == 0 ? a[0] : a[1], delta, acc);
#pragma unroll
        for (int o = 1; o < kGroup; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      }
      if (q4 == 0) pj[row] = row > j ? beta * acc : 0.f;
      __syncthreads();
      // K = beta/2 * v.p, recomputed by every warp (p is zero up to index j)
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) dot = fmaf(xj[32 * k + lane], pj[32 * k + lane], dot);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      dot = fmaf(delta, pj[j + 1], dot);
      const float K = 0.5f * beta * dot;
      if (live_rows) {
        // A -= v w^T + w v^T, w = p - K v; computed with x for v, then the
        // column j+1 term corrected by delta * (w_r - K v_r)
        const float vr = row > j ? xj[row] + (row == j + 1 ? delta : 0.f) : 0.f;
        const float wr = pj[row] - K * vr;
#pragma unroll
        for (int i = 0; i < kEigPer; ++i) {
          if (i + base >= kEigPer) break;
          const int c = kGroup * (i + base) + q4;
          const float xc = xj[c];
          a[i] -= vr * fmaf(-K, xc, pj[c]) + wr * xc;
        }
        if (owns_next) {
          const float corr = delta * (wr - K * vr);
          if (next_idx == 0) a[0] -= corr; else a[1] -= corr;
        }
      }
    }
    if (j % kGroup == kGroup - 1) {
#pragma unroll
      for (int i = 0; i < kEigPer - 1; ++i) a[i] = a[i + 1];
      a[kEigPer - 1] = 0.f;
      ++base;
    }
  }
  // last 2 x 2 block: after (n-2)/kGroup shifts a[0] holds column n-2-(n-2)%kGroup + q4
  static_assert((kHeadDim - 2) % kGroup + 1 < kGroup, "columns n-2 and n-1 share a[0]");
  if (row == n - 2 && q4 == (n - 2) % kGroup) s.d[n - 2] = a[0];
  if (row == n - 1 && q4 == (n - 2) % kGroup) s.e[n - 2] = a[0];
  if (row == n - 1 && q4 == (n - 1) % kGroup) s.d[n - 1] = a[0];
  __syncthreads();
  if (tid == 0) {
    s.e[n - 1] = 0.f;
    float tn = 0.f;
    for (int i = 0; i < n; ++i) {
      const float rad = fabsf(s.d[i]) + fabsf(s.e[i]) + (i > 0 ? fabsf(s.e[i - 1]) : 0.f);
      tn = fmaxf(tn, rad);
    }
    s.tnorm = fmaxf(tn, FLT_MIN);
  }
  __syncthreads();
  if (tid < n) s.e2[tid] = s.e[tid] * s.e[tid];
  __syncthreads();

  // --- top r eigenvalues by multisection (one warp per eigenvalue) ----------
  const float tnorm = s.tnorm;
  const float pivmin = FLT_MIN * 1e4f;
  for (int jj = warp; jj < r; jj += kWarps) {
    const int target = n - 1 - jj;                   // ascending index
    float lo = -tnorm * 1.01f - pivmin, hi = tnorm * 1.01f + pivmin;
    for (int round = 0; round < 8; ++round) {
      const float step = (hi - lo) / 33.f;
      const float xv = lo + step * (float)(lane + 1);
      const int cnt = sturm_count(s, xv, pivmin);
      const unsigned above = __ballot_sync(0xffffffffu, cnt >= target + 1);
      const int first = above ? __ffs(above) - 1 : 32;
      const float nlo = first == 0 ? lo : lo + step * (float)first;
      const float nhi = first == 32 ? hi : lo + step * (float)(first + 1);
      lo = nlo;
      hi = nhi;
      if (hi - lo <= 2.f * FLT_EPSILON * fmaxf(fabsf(lo), fabsf(hi)) + pivmin) break;
    }
    if (lane == 0) s.lam[jj] = 0.5f * (lo + hi);
  }
  __syncthreads();

  // --- inverse iteration (lane 0 of one warp per eigenvalue) -----------------
  const float guard = FLT_EPSILON * tnorm;
  for (int jj = warp; jj < r; jj += kWarps) {
    float* rd = s.lu[jj][0];
    float* u1 = s.lu[jj][1];
    float* u2 = s.lu[jj][2];
    float* ml = s.lu[jj][3];
    float* pf = s.lu[jj][4];
    float* zz = s.z[jj];
    for (int i = lane; i < n; i += 32) zz[i] = hash_unit(i, jj) + 0.75f;
    __syncwarp();
    if (lane == 0) {
      const float lam = s.lam[jj];
      // LU with partial pivoting of T - lam I (rows: sub e[i-1], diag d[i]-lam, super e[i]);
      // rd holds the reciprocals of U's (guarded) diagonal
      float cd = s.d[0] - lam, cs = s.e[0];
      for (int i = 0; i < n - 1; ++i) {
        const float sub = s.e[i], nd = s.d[i + 1] - lam, ns = s.e[i + 1];
        if (fabsf(cd) >= fabsf(sub)) {
          if (fabsf(cd) < guard) cd = cd < 0.f ? -guard : guard;
          const float inv = 1.f / cd;
          const float l = sub * inv;
          rd[i] = inv; u1[i] = cs; u2[i] = 0.f; ml[i] = l; pf[i] = 0.f;
          cd = nd - l * cs;
          cs = ns;
        } else {
          const float l = cd / sub;
          const float dg = fabsf(sub) < guard ? (sub < 0.f ? -guard : guard) : sub;
          rd[i] = 1.f / dg; u1[i] = nd; u2[i] = ns; ml[i] = l; pf[i] = 1.f;
          cd = cs - l * nd;
          cs = -l * ns;
        }
      }
      if (fabsf(cd) < guard) cd = cd < 0.f ? -guard : guard;
      rd[n - 1] = 1.f / cd; u1[n - 1] = 0.f; u2[n - 1] = 0.f;
      for (int it = 0; it < 2; ++it) {
        for (int i = 0; i < n - 1; ++i) {
          if (pf[i] != 0.f) {
            const float t = zz[i];
            zz[i] = zz[i + 1];
            zz[i + 1] = t - ml[i] * zz[i + 1];
          } else {
            zz[i + 1] -= ml[i] * zz[i];
          }
        }
        zz[n - 1] = zz[n - 1] * rd[n - 1];
        zz[n - 2] = (zz[n - 2] - u1[n - 2] * zz[n - 1]) * rd[n - 2];
        float mx = fmaxf(fabsf(zz[n - 1]), fabsf(zz[n - 2]));
        for (int i = n - 3; i >= 0; --i) {
          zz[i] = (zz[i] - u1[i] * zz[i + 1] - u2[i] * zz[i + 2]) * rd[i];
          mx = fmaxf(mx, fabsf(zz[i]));
        }
        const float inv = mx > 0.f ? 1.f / mx : 0.f;
        for (int i = 0; i < n; ++i) zz[i] *= inv;
      }
    }
    __syncwarp();
  }
  __syncthreads();

  // --- orthonormalise the r vectors: Cholesky-QR, two passes ---------------
  // M = Z Z^T = L L^T, Z <- L^{-1} Z. A non-positive pivot (a dependent
  // vector) drops that vector.
  for (int pass = 0; pass < 2; ++pass) {
    for (int pr = warp; pr < r * r; pr += kWarps) {
      const int ia = pr / r, ib = pr % r;
      if (ib > ia) continue;
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) dot = fmaf(s.z[ia][32 * k + lane], s.z[ib][32 * k + lane], dot);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (lane == 0) s.gram[ia][ib] = dot;
    }
    __syncthreads();
    if (warp == 0) {                                   // in-place lower Cholesky factor, lane = row
      for (int k = 0; k < r; ++k) {
        // row k's entries left of the diagonal are final: finish column k
        float dkk = 0.f;
        if (lane == k) {
          float acc = s.gram[k][k];
          for (int m = 0; m < k; ++m) acc -= s.gram[k][m] * s.gram[k][m];
          dkk = acc > 1e-20f ? sqrtf(acc) : 0.f;
          s.gram[k][k] = dkk;
        }
        dkk = __shfl_sync(0xffffffffu, dkk, k);
        if (lane > k && lane < r) {
          float acc = s.gram[lane][k];
          for (int m = 0; m < k; ++m) acc -= s.gram[lane][m] * s.gram[k][m];
          s.gram[lane][k] = dkk > 0.f ? acc / dkk : 0.f;
        }
        __syncwarp();
      }
    }
    __syncthreads();
    if (tid < n) {                                     // forward substitution in place, one column per thread
      for (int ia = 0; ia < r; ++ia) {
        float acc = s.z[ia][tid];
        for (int ib = 0; ib < ia; ++ib) acc -= s.gram[ia][ib] * s.z[ib][tid];
        s.z[ia][tid] = s.gram[ia][ia] > 0.f ? acc / s.gram[ia][ia] : 0.f;
      }
    }
    __syncthreads();
  }

  // --- back-transform: y = H_0 H_1 ... H_{n-3} z  (one warp per vector) -----
  for (int jj = warp; jj < r; jj += kWarps) {
    float* y = s.z[jj];
    float yl[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) yl[c] = y[lane + 32 * c];
    for (int j = n - 3; j >= 0; --j) {
      const float beta = s.beta[j];
      if (beta == 0.f) continue;
      const float* hv = s.hv[j];
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) dot = fmaf(hv[lane + 32 * c], yl[c], dot);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      const float f = beta * dot;
#pragma unroll
      for (int c = 0; c < 4; ++c) yl[c] -= f * hv[lane + 32 * c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) y[lane + 32 * c] = yl[c];
  }
  __syncthreads();
  for (int el = tid; el < kCurdkvMaxRank * n; el += kEigThreads) {
    const int jj = el / n;
    evec_out[el] = jj < r ? s.z[jj][el % n] : 0.f;
  }
}

// ---------------------------------------------------------------------------
// Leverage and cumulative score on the tensor cores. One CTA per 128 rows of
// one (b, h): the projections P = V_tile E^T (E = the top-r eigenvectors,
// split into bf16 hi + lo, zero rows past r) come from one M=128, N=32 MMA
// chain with the value tile in its natural K-major layout; then
// l_i = a_i^2 * |P_i|^2 / E, accumulated into kept rows' scores and seeding
// incoming rows'. grid = (ceil(n / 128), B*H), block = 128.
// ---------------------------------------------------------------------------
constexpr int kEvecTileBytes = kCurdkvMaxRank * kHeadDim * 2;
constexpr int kLevSmem = kTileBytes + 2 * kEvecTileBytes + 1024;
static_assert(kCurdkvMaxRank == 32, "the leverage MMA uses N = 32");

__global__ void __launch_bounds__(kAttnThreads) curdkv_leverage_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int bh = blockIdx.y, i0 = blockIdx.x * kTile, tid = threadIdx.x, warp = tid >> 5;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t v_tile = tc::smem_u32(smem), ehi = v_tile + kTileBytes, elo = ehi + kEvecTileBytes;
  const int row_end = min(p.n, i0 + kTile);
  if (tid == 0) tc::mbar_init(&bar, 1);
  if (warp == 0) tc::tmem_alloc(&tmem_base, kCurdkvMaxRank);
  for (int c = tid; c < kTile * 16; c += kAttnThreads) {
    const int r = c >> 4, j = c & 15;
    const int row = i0 + r;
    const bool ok = row < row_end;
    tc::cp_async16(v_tile + tc::sw128_offset(r, j, kTile), value_row(p, bh, ok ? row : i0) + j * 16, ok ? 16u : 0u);
  }
  // eigenvectors -> bf16 hi and lo tiles (32 rows, K-major, swizzled)
  const float* ev = p.evec + (size_t)bh * kCurdkvMaxRank * kHeadDim;
  for (int item = tid; item < kCurdkvMaxRank * 16; item += kAttnThreads) {
    const int jr = item >> 4, ch = item & 15;
    const float4 x0 = *reinterpret_cast<const float4*>(ev + jr * kHeadDim + 8 * ch);
    const float4 x1 = *reinterpret_cast<const float4*>(ev + jr * kHeadDim + 8 * ch + 4);
    const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hw[q] = pack_bf16x2(x[2 * q], x[2 * q + 1]);
      lw[q] = pack_bf16x2(x[2 * q] - __uint_as_float(hw[q] << 16), x[2 * q + 1] - __uint_as_float(hw[q] & 0xffff0000u));
    }
    const uint32_t off = tc::sw128_offset(jr, ch, kCurdkvMaxRank);
    *reinterpret_cast<uint4*>(smem + kTileBytes + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(smem + kTileBytes + kEvecTileBytes + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
  tc::cp_async_wait_all();
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kTile, kCurdkvMaxRank);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      const uint32_t a_off = (uint32_t)((st >> 2) * kTile * 128 + (st & 3) * 32);
      const uint32_t b_off = (uint32_t)((st >> 2) * kCurdkvMaxRank * 128 + (st & 3) * 32);
      const uint64_t ad = tc::sw128_desc(v_tile + a_off);
      tc::mma_bf16(tmem, ad, tc::sw128_desc(ehi + b_off), idesc, st > 0 ? 1u : 0u);
      tc::mma_bf16(tmem, ad, tc::sw128_desc(elo + b_off), idesc, 1u);
    }
    tc::mma_commit(&bar);
  }
  bool ok = false;
  for (int spin = 0; spin < kMbarSpin && !ok; ++spin) ok = tc::mbar_try_wait(&bar, 0);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (tid & 31) == 0) raise_device_error(p.err, kDevWaitTimeout);
  tc::fence_after_sync();
  const int i = i0 + tid;
  if (ok) {
    float proj[32];
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), proj);
    float e4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) e4[jj & 3] = fmaf(proj[jj], proj[jj], e4[jj & 3]);
    if (i < p.n) {
      const float a = p.attn[(size_t)bh * p.rows + i];
      const float l = a * a * ((e4[0] + e4[1]) + (e4[2] + e4[3])) * p.inv_e[bh];
      p.lev[(size_t)bh * p.rows + i] = l;
      if (i < p.k) p.score_st[(size_t)bh * p.cap + i] += l;
      else p.new_score[(size_t)bh * p.new_stride + (i - p.k)] = l;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kCurdkvMaxRank);
}

// Append the block (cache stays within budget): grid = (ceil(m / 64), B*H), block = 256.
__global__ void __launch_bounds__(256) curdkv_append_kernel(const __grid_constant__ CurdkvParams p) {
  const int bh = blockIdx.y, b = bh / p.heads;
  const int c = threadIdx.x & 15, hw = threadIdx.x >> 4;
  constexpr int kRowBytes = kHeadDim * 2;
  for (int j = 0; j < 4; ++j) {
    const int t = blockIdx.x * 64 + hw + 16 * j;
    if (t >= p.m) break;
    const size_t dst = (size_t)bh * p.cap + p.k + t;
    const size_t src = (size_t)bh * p.m + t;
    reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.kst)) + dst * kRowBytes)[c] =
        reinterpret_cast<const uint4*>(static_cast<const char*>(p.k_in) + src * kRowBytes)[c];
    reinterpret_cast<uint4*>(static_cast<char*>(const_cast<void*>(p.vst)) + dst * kRowBytes)[c] =
        reinterpret_cast<const uint4*>(static_cast<const char*>(p.v_in) + src * kRowBytes)[c];
    if (c == 0) {
      p.score_st[dst] = p.new_score[(size_t)bh * p.new_stride + t];
      p.pos_st[dst] = p.pos_in ? p.pos_in[(size_t)b * p.m + t] : (int32_t)(p.offset + t);
    }
  }
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

void curdkv_layout(evict_handle* h, size_t* off, char* base) {
  if (!h->curdkv) h->curdkv = new CurdkvState();
  CurdkvState& st = *h->curdkv;
  const size_t bh = (size_t)h->cfg.batch * h->cfg.n_kv_heads;
  st.rows = h->cap + h->cfg.max_block;
  st.splits = (st.rows + kGramRows - 1) / kGramRows;
  auto take = [&](size_t bytes) {
    *off = round256(*off);
    char* p = base ? base + *off : nullptr;
    *off += bytes;
    return p;
  };
  st.lse_stride = (h->cfg.max_block + 3) / 4 * 4;
  st.lse = reinterpret_cast<float*>(take(bh * st.lse_stride * 4));
  st.lse_part = reinterpret_cast<float2*>(take(bh * kMaxLseSplit * st.lse_stride * sizeof(float2)));
  st.attn = reinterpret_cast<float*>(take(bh * st.rows * 4));
  st.lev = reinterpret_cast<float*>(take(bh * st.rows * 4));
  st.gram_part = reinterpret_cast<float*>(take(bh * st.splits * kHeadDim * kHeadDim * 4));
  st.evec = reinterpret_cast<float*>(take(bh * kCurdkvMaxRank * kHeadDim * 4));
  st.inv_e = reinterpret_cast<float*>(take(bh * 4));
}

void curdkv_release(evict_handle* h) {
  delete h->curdkv;
  h->curdkv = nullptr;
}

int curdkv_prepare(evict_handle* h) {
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&h->curdkv->sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPipeSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPipeSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGramTcSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_leverage_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLevSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(EigSmem))) != cudaSuccess)
    return cuda_fail(e, "CurDKV kernel attributes");
  return EVICT_OK;
}

int curdkv_update(evict_handle* h, const void* k, const void* v, const int32_t* pos, int m) {
  CurdkvState& st = *h->curdkv;
  const evict_config& c = h->cfg;
  const int bh = c.batch * c.n_kv_heads;
  const int n = h->n_kept + m;
  CurdkvParams p;
  memset(&p, 0, sizeof(p));
  p.k_in = k;
  p.v_in = v;
  p.kst = h->kst;
  p.vst = h->vst;
  p.k = h->n_kept;
  p.m = m;
  p.n = n;
  p.cap = h->cap;
  p.heads = c.n_kv_heads;
  p.rank = std::min(std::min(c.rank_cap, n), kHeadDim);
  p.scale2 = kLog2e / sqrtf((float)kHeadDim);
  p.lse = st.lse;
  p.lse_part = st.lse_part;
  p.lse_stride = st.lse_stride;
  p.attn = st.attn;
  p.lev = st.lev;
  p.rows = st.rows;
  p.gram_part = st.gram_part;
  p.splits = st.splits;
  p.evec = st.evec;
  p.inv_e = st.inv_e;
  p.score_st = h->score_st;
  p.new_score = h->new_score;
  p.new_stride = h->new_stride;
  p.pos_st = h->pos_st;
  p.pos_in = pos;
  p.offset = h->offset;
  p.err = h->err;
  const cudaStream_t sm = h->stream;
  cudaError_t e;
  const int k_tiles = (n + kTile - 1) / kTile;
  // key splits for pass 1: enough CTAs to fill the GPU a few times over,
  // each split keeping at least 4 key tiles
  const int q_pairs = (m + 2 * kTile - 1) / (2 * kTile), k_pairs = (n + 2 * kTile - 1) / (2 * kTile);
  int n_split = (4 * std::max(st.sm_count, 1) + q_pairs * bh - 1) / (q_pairs * bh);
  n_split = std::max(1, std::min({n_split, kMaxLseSplit, std::max(1, k_tiles / 4)}));
  e = timed_launch(h, kKidCurdkvLse, [&] {
    curdkv_lse_kernel<<<dim3(q_pairs, n_split, bh), kPipeThreads, kPipeSmem, sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 1 launch");
  e = timed_launch(h, kKidCurdkvLseMerge, [&] {
    curdkv_lse_merge_kernel<<<dim3((m + 255) / 256, bh), 256, 0, sm>>>(p, n_split);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention merge launch");
  e = timed_launch(h, kKidCurdkvColsum, [&] {
    curdkv_colsum_kernel<<<dim3(k_pairs, bh), kPipeThreads, kPipeSmem, sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 2 launch");
  e = timed_launch(h, kKidCurdkvGram, [&] {
    curdkv_gram_kernel<<<dim3((n + kGramRows - 1) / kGramRows, bh), kAttnThreads, kGramTcSmem, sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV Gram launch");
  e = timed_launch(h, kKidCurdkvEig, [&] {
    curdkv_eig_kernel<<<bh, kEigThreads, sizeof(EigSmem), sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV eigensolver launch");
  e = timed_launch(h, kKidCurdkvLeverage, [&] {
    curdkv_leverage_kernel<<<dim3(k_tiles, bh), kAttnThreads, kLevSmem, sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV leverage launch");
  if (n <= c.budget) {
    e = timed_launch(h, kKidAppend, [&] {
      curdkv_append_kernel<<<dim3((m + 63) / 64, bh), 256, 0, sm>>>(p);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV append launch");
    h->n_kept = n;
    h->last_evicted = false;
  } else {
    GroupParams P = make_group_params(h, m, 1);
    P.L[0] = make_layer_ptrs(h, k, v, pos);
    e = timed_launch(h, kKidSelect, [&] { return launch_select(P, sm); });
    if (e != cudaSuccess) return cuda_fail(e, "select kernel launch");
    e = timed_launch(h, kKidCompact, [&] { return launch_compact(P, 2, sm); });
    if (e != cudaSuccess) return cuda_fail(e, "compact kernel launch");
    h->n_kept = c.budget;
    h->last_evicted = true;
  }
  h->offset += m;
  st.last_n = n;
  return EVICT_OK;
}

int curdkv_last_scores(const evict_handle* h, float* attn, float* lev, int* n_out) {
  const CurdkvState& st = *h->curdkv;
  *n_out = st.last_n;
  if (st.last_n == 0) return EVICT_OK;
  const size_t bh = (size_t)h->cfg.batch * h->cfg.n_kv_heads;
  const size_t w = (size_t)st.last_n * sizeof(float);
  cudaError_t e = cudaSuccess;
  if (attn) e = cudaMemcpy2DAsync(attn, w, st.attn, st.rows * sizeof(float), w, bh, cudaMemcpyDeviceToDevice, h->stream);
  if (e == cudaSuccess && lev)
    e = cudaMemcpy2DAsync(lev, w, st.lev, st.rows * sizeof(float), w, bh, cudaMemcpyDeviceToDevice, h->stream);
  if (e != cudaSuccess) return cuda_fail(e, "copying CurDKV scores");
  return EVICT_OK;
}

}  // namespace evict
