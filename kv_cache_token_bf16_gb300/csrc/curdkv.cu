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
//   curdkv_lse_kernel      pass 1: per query, running max and sum of 2^logit over
//                          this CTA's key tiles (TMA-fed tcgen05 MMA, 512 queries x
//                          128 keys per step, warp-specialised, persistent grid)
//   curdkv_lse_merge_kernel  log2-sum-exp per query from the per-CTA partials
//   curdkv_colsum_kernel   pass 2: per key, sum over queries of 2^(logit - lse)
//                          (same pipeline, 128 keys x 512 queries per step)
//   curdkv_colsum_merge_kernel  sum of the per-quad column sums (blocks > 512 rows)
//   curdkv_gram_kernel     partial G over a slice of rows (tcgen05, split bf16)
//   curdkv_eig_kernel      sum of partials (fp64), Householder tridiagonalisation,
//                          multisection bisection for the top r eigenvalues,
//                          inverse iteration, orthonormalisation, back-transform
//   curdkv_leverage_kernel l_i (projections on tcgen05) and the cumulative-score update
//   curdkv_append_kernel   copy of the block when the cache stays within budget
#include <cuda.h>
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
  float* colpart = nullptr;    // [quads, BH, rows] per-quad column sums (blocks > 512 rows)
  int quads = 0;               // ceil(max_block / 512)
};

namespace {

constexpr int kTile = 128;                  // rows of a query or key tile
constexpr int kAttnThreads = 128;           // 4 warps: one TMEM lane per thread
constexpr int kTileBytes = kTile * kHeadDim * 2;
constexpr int kGramRows = 2048;             // rows per Gram partial
constexpr int kEigThreads = 1024;
constexpr int kMbarSpin = 1 << 22;          // bounded MMA wait (well above a tile's time)
constexpr float kLog2e = 1.4426950408889634f;

// Static split of the attention passes' key tiles over a persistent grid.
struct AttnSched {
  int C;            // kept-row key tiles, ceil(k / 128)
  int Q;            // query quads, ceil(m / 512)
  int per_bh;       // key tiles of all quads of one (b, h)
  int bh_count;
  int ctas;
  long long total;  // per_bh * bh_count
  // first key tile of CTA c; CTA c takes [begin(c), begin(c + 1))
  __host__ __device__ long long begin(int c) const { return total * c / ctas; }
  // the CTA whose share holds key tile g
  __host__ __device__ int cta_of(long long g) const { return (int)(((g + 1) * ctas + total - 1) / total) - 1; }
};

struct CurdkvParams {
  CUtensorMap tm_kin;    // incoming keys [BH][m][128] bf16, boxes of 128 rows x 64 elements, 128-byte swizzle
  CUtensorMap tm_kst;    // kept keys [BH][k][128] (row pitch cap), same boxes; unused when k = 0
  AttnSched sched1, sched2;
  float* colpart;        // [Q, BH, rows] per-quad column sums (= attn when Q = 1)
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
// Proxy-softmax attention passes: tensor cores, TMA, warp specialisation and
// a persistent grid.
//
// Work unit = (b, h, query quad): up to four 128-row tiles of incoming rows
// (512 proxy queries), held fixed in shared memory while the key tiles they
// can see stream through a ring. Key tiles are aligned to the end of the kept
// rows: kept tile c covers rows k - 128 (C - c) .. +127 (the first may start
// below zero; TMA fills those rows with zeros), incoming tile u covers rows
// k + 128 u .. +127. No tile mixes the two buffers, so each is one pair of
// TMA boxes. The key tiles of all units are laid end to end and every CTA
// takes an equal contiguous share: one wave of CTAs with equal work; a unit
// may be shared by neighbouring CTAs (pass 1 then leaves one partial per CTA).
//
// Roles (576 threads): warps 0-15 read the accumulators (warp w: TMEM lanes
// 32 (w % 4) .. +31, accumulator w / 4 = query tile w / 4 of the quad);
// warp 16 issues the TMA loads; warp 17 issues the MMAs. Each query tile has
// its own 128-column fp32 accumulator (512 TMEM columns), so the MMAs of one
// accumulator run while the other three are read. mbarriers connect the
// roles; every wait is bounded and a timeout stops the CTA cleanly.
// ---------------------------------------------------------------------------
constexpr int kQuad = 4;                          // fixed query tiles per unit
constexpr int kSoftWarps = 16;
constexpr int kAttnCtaThreads = (kSoftWarps + 2) * 32;
constexpr int kMaxLseSplit = 8;                   // CTAs that may share one unit in pass 1
constexpr int kLseStages = 3, kColStages = 2;
constexpr int attn_smem_bytes(int stages) { return (kQuad + stages) * kTileBytes + 1024; }

// Key tiles seen by quad q: every kept tile and the incoming tiles up to the quad's last query.
__host__ __device__ __forceinline__ int quad_tiles(int C, int m, int q) {
  const int last = (m < kQuad * kTile * (q + 1) ? m : kQuad * kTile * (q + 1)) - 1;
  return C + last / kTile + 1;
}
// Key tiles of quads 0 .. q-1 (all full: quad j sees C + 4 j + 4 tiles).
__host__ __device__ __forceinline__ int quad_prefix(int C, int q) { return q * C + 2 * q * (q + 1); }
// Query tiles of quad q that hold at least one incoming row.
__host__ __device__ __forceinline__ int quad_rows(int m, int q) {
  const int left = (m - kQuad * kTile * q + kTile - 1) / kTile;
  return left < kQuad ? left : kQuad;
}

// Cursor over the flattened key tiles (b, h) -> quad -> key tile.
struct UnitCursor {
  int bh, q, kt, tiles;
  __device__ void init(const AttnSched& s, int m, long long g) {
    bh = (int)(g / s.per_bh);
    int rem = (int)(g - (long long)bh * s.per_bh);
    q = 0;
    while (rem >= quad_tiles(s.C, m, q)) rem -= quad_tiles(s.C, m, q++);
    kt = rem;
    tiles = quad_tiles(s.C, m, q);
  }
  __device__ void next(const AttnSched& s, int m) {
    if (++kt == tiles) {
      kt = 0;
      if (++q == s.Q) {
        q = 0;
        ++bh;
      }
      tiles = quad_tiles(s.C, m, q);
    }
  }
};

// Bounded wait on an mbarrier phase. Gives up early once the CTA's failure
// flag is set; after kMbarSpin polls it sets the flag and the error word.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* fail, int* err) {
  for (int spin = 0; spin < kMbarSpin; ++spin) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((spin & 63) == 63 && *fail) return false;
  }
  *fail = 1;
  raise_device_error(err, kDevWaitTimeout);
  return false;
}
// The same wait ignoring the failure flag: used to let copies and MMAs already
// issued finish before the CTA releases its shared and tensor memory.
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity, int* err) {
  for (int spin = 0; spin < kMbarSpin; ++spin)
    if (tc::mbar_try_wait(bar, parity)) return;
  raise_device_error(err, kDevWaitTimeout);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Shared state of one attention CTA (static shared memory).
struct AttnBars {
  uint64_t stage_full[kLseStages], stage_empty[kLseStages];
  uint64_t fixed_full, fixed_empty;
  uint64_t acc_full[kQuad], acc_empty[kQuad];
  uint32_t tmem_base;
  int fail;
};

// The two data-movement roles, shared by both passes.
// kColsum = false: pass 1, accumulator a = fixed query tile a x streamed keys.
// kColsum = true:  pass 2, accumulator a = streamed keys x fixed query tile a.
template <int kStagesT>
__device__ void attn_producer(const CurdkvParams& p, const AttnSched& s, AttnBars& b, uint32_t fixed,
                              uint32_t stage0, long long g0, long long g1) {
  UnitCursor u;
  u.init(s, p.m, g0);
  int units = 0, issued[kStagesT];
#pragma unroll
  for (int i = 0; i < kStagesT; ++i) issued[i] = 0;
  tc::tma_prefetch_desc(&p.tm_kin);
  if (s.C > 0) tc::tma_prefetch_desc(&p.tm_kst);
  for (long long g = g0; g < g1; ++g) {
    const int j = (int)(g - g0);
    if (g == g0 || u.kt == 0) {                   // a new unit: its query tiles
      if (!wait_phase(&b.fixed_empty, (uint32_t)((units & 1) ^ 1), &b.fail, p.err)) break;
      const int nq = quad_rows(p.m, u.q);
      tc::mbar_arrive_expect_tx(&b.fixed_full, (uint32_t)(nq * kTileBytes));
      for (int a = 0; a < nq; ++a)
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(fixed + a * kTileBytes + hf * (kTileBytes / 2), &p.tm_kin, 64 * hf,
                          kQuad * kTile * u.q + kTile * a, u.bh, &b.fixed_full);
      ++units;
    }
    const int st = j % kStagesT;
    if (!wait_phase(&b.stage_empty[st], (uint32_t)(((j / kStagesT) & 1) ^ 1), &b.fail, p.err)) break;
    tc::mbar_arrive_expect_tx(&b.stage_full[st], (uint32_t)kTileBytes);
    const bool kept = u.kt < s.C;
    const void* map = kept ? (const void*)&p.tm_kst : (const void*)&p.tm_kin;
    const int y = kept ? p.k - kTile * (s.C - u.kt) : kTile * (u.kt - s.C);
    for (int hf = 0; hf < 2; ++hf)
      tc::tma_load_3d(stage0 + st * kTileBytes + hf * (kTileBytes / 2), map, 64 * hf, y, u.bh, &b.stage_full[st]);
    ++issued[st];
    u.next(s, p.m);
  }
  // every copy issued must land before the CTA may release its shared memory
  for (int i = 0; i < kStagesT; ++i)
    if (issued[i] > 0) drain_phase(&b.stage_full[i], (uint32_t)((issued[i] - 1) & 1), p.err);
  if (units > 0) drain_phase(&b.fixed_full, (uint32_t)((units - 1) & 1), p.err);
}

template <int kStagesT, bool kColsum>
__device__ void attn_mma(const CurdkvParams& p, const AttnSched& s, AttnBars& b, uint32_t tmem, uint32_t fixed,
                         uint32_t stage0, long long g0, long long g1) {
  UnitCursor u;
  u.init(s, p.m, g0);
  int units = 0, uses[kQuad] = {0, 0, 0, 0};
  bool ok = true;
  for (long long g = g0; g < g1 && ok; ++g) {
    const int j = (int)(g - g0);
    const int nq = quad_rows(p.m, u.q);
    if (g == g0 || u.kt == 0) {
      if (!wait_phase(&b.fixed_full, (uint32_t)(units & 1), &b.fail, p.err)) break;
      ++units;
    }
    const int st = j % kStagesT;
    if (!wait_phase(&b.stage_full[st], (uint32_t)((j / kStagesT) & 1), &b.fail, p.err)) break;
    const uint32_t keys = stage0 + st * kTileBytes;
    for (int a = 0; a < nq; ++a) {
      if (!wait_phase(&b.acc_empty[a], (uint32_t)((uses[a] & 1) ^ 1), &b.fail, p.err)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t q_tile = fixed + a * kTileBytes;
      if (kColsum) issue_tile_mma(tmem + (uint32_t)(a * kTile), keys, q_tile);
      else issue_tile_mma(tmem + (uint32_t)(a * kTile), q_tile, keys);
      tc::mma_commit(&b.acc_full[a]);
      ++uses[a];
    }
    if (!ok) break;
    tc::mma_commit(&b.stage_empty[st]);
    if (u.kt == u.tiles - 1) tc::mma_commit(&b.fixed_empty);
    u.next(s, p.m);
  }
  // the accumulators' last MMAs must finish before TMEM is released
  for (int a = 0; a < kQuad; ++a)
    if (uses[a] > 0) drain_phase(&b.acc_full[a], (uint32_t)((uses[a] - 1) & 1), p.err);
}

// Bounded, warp-uniform wait of an accumulator-reading warp.
__device__ __forceinline__ bool warp_wait_acc(uint64_t* bar, uint32_t parity, AttnBars& b, int* err) {
  bool ok = wait_phase(bar, parity, &b.fail, err);
  return __all_sync(0xffffffffu, ok);
}

// 64 accumulator columns of this thread's row (two 32-column loads, one wait).
__device__ __forceinline__ void load64(uint32_t taddr, float (&v)[64]) {
  uint32_t r0[32], r1[32];
  tc::tmem_ld32_nowait(taddr, r0);
  tc::tmem_ld32_nowait(taddr + 32, r1);
  tc::tmem_wait_ld32x2(r0, r1);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    v[c] = __uint_as_float(r0[c]);
    v[c + 32] = __uint_as_float(r1[c]);
  }
}

// Setup shared by both passes: barriers, TMEM, this CTA's share of the tiles.
template <int kStagesT>
__device__ __forceinline__ void attn_setup(AttnBars& b) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesT; ++i) {
      tc::mbar_init(&b.stage_full[i], 1);
      tc::mbar_init(&b.stage_empty[i], 1);
    }
    tc::mbar_init(&b.fixed_full, 1);
    tc::mbar_init(&b.fixed_empty, 1);
    for (int a = 0; a < kQuad; ++a) {
      tc::mbar_init(&b.acc_full[a], 1);
      tc::mbar_init(&b.acc_empty[a], 4);         // the four warps reading accumulator a
    }
    b.fail = 0;
  }
  if (warp == 0) tc::tmem_alloc(&b.tmem_base, kQuad * kTile);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__device__ __forceinline__ void attn_teardown(AttnBars& b) {
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if ((threadIdx.x >> 5) == 0) tc::tmem_dealloc(b.tmem_base, kQuad * kTile);
}

// ---------------------------------------------------------------------------
// Pass 1: for each proxy query t, (max, sum) of 2^x over the keys i <= k + t
// that this CTA streams, x = scale2 * q_t . k_i (base 2). A unit shared by
// several CTAs leaves one partial per CTA (slot = CTA - first CTA of the unit).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAttnCtaThreads, 1) curdkv_lse_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ AttnBars b;
  const AttnSched& s = p.sched1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t fixed = tc::smem_u32(smem), stage0 = fixed + kQuad * kTileBytes;
  const long long g0 = s.begin(blockIdx.x), g1 = s.begin(blockIdx.x + 1);
  attn_setup<kLseStages>(b);
  const uint32_t tmem = b.tmem_base;
  if (warp == kSoftWarps) {
    if (lane == 0) attn_producer<kLseStages>(p, s, b, fixed, stage0, g0, g1);
    __syncwarp();
  } else if (warp == kSoftWarps + 1) {
    if (lane == 0) attn_mma<kLseStages, false>(p, s, b, tmem, fixed, stage0, g0, g1);
    __syncwarp();
  } else {
    const int a = warp >> 2, row = 32 * (warp & 3) + lane;
    const uint32_t acc = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(a * kTile);
    UnitCursor u;
    u.init(s, p.m, g0);
    int uses = 0;
    bool dead = false;
    float run_max = -INFINITY, run_sum = 0.f;
    for (long long g = g0; g < g1; ++g) {
      const int nq = quad_rows(p.m, u.q);
      const int t = kQuad * kTile * u.q + kTile * a + row;        // this thread's query
      if (a < nq && !dead) {
        if (!warp_wait_acc(&b.acc_full[a], (uint32_t)(uses & 1), b, p.err)) dead = true;
        ++uses;
      }
      if (a < nq && !dead) {
        tc::fence_after_sync();
        const bool kept = u.kt < s.C;
        const int base = kept ? p.k - kTile * (s.C - u.kt) : p.k + kTile * (u.kt - s.C);
        // every key of the tile is a real row visible to every query of the accumulator
        const bool full = kept ? base >= 0 : kTile * (u.kt - s.C) + kTile - 1 <= kQuad * kTile * u.q + kTile * a;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float v[64];
          load64(acc + (uint32_t)(64 * hf), v);
          if (!full) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int i = base + 64 * hf + c;
              if (i < 0 || i > p.k + t) v[c] = -INFINITY;
            }
          }
          float mx[22];
#pragma unroll
          for (int c = 0; c < 21; ++c) mx[c] = fmax3(v[3 * c], v[3 * c + 1], v[3 * c + 2]);
          mx[21] = v[63];
#pragma unroll
          for (int c = 0; c < 7; ++c) mx[c] = fmax3(mx[3 * c], mx[3 * c + 1], mx[3 * c + 2]);
          mx[7] = mx[21];
          const float m8 = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
          if (m8 > -INFINITY) {
            const float nm = fmaxf(run_max, m8 * p.scale2);
            float sm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 64; ++c) sm[c & 7] += ex2(fmaf(v[c], p.scale2, -nm));
            const float tot = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
            run_sum = run_sum * ex2(run_max - nm) + tot;         // ex2(-inf) = 0 on the first visible tile
            run_max = nm;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&b.acc_empty[a]);
      }
      if (u.kt == u.tiles - 1 || g == g1 - 1) {                   // this CTA's part of the unit ends
        if (a < nq && !dead && t < p.m) {
          const long long first = (long long)u.bh * s.per_bh + quad_prefix(s.C, u.q);
          const int slot = (int)blockIdx.x - s.cta_of(first);
          p.lse_part[((size_t)u.bh * kMaxLseSplit + slot) * p.lse_stride + t] = make_float2(run_max, run_sum);
        }
        run_max = -INFINITY;
        run_sum = 0.f;
      }
      u.next(s, p.m);
    }
  }
  attn_teardown(b);
}

// Merge the per-CTA partials: lse2[t] = log2 sum_s s_s 2^(m_s). grid = (ceil(m / 256), B*H).
__global__ void __launch_bounds__(256) curdkv_lse_merge_kernel(const __grid_constant__ CurdkvParams p) {
  const AttnSched& s = p.sched1;
  const int bh = blockIdx.y, t = blockIdx.x * 256 + threadIdx.x;
  if (t >= p.m) return;
  const int q = t / (kQuad * kTile);
  const long long first = (long long)bh * s.per_bh + quad_prefix(s.C, q);
  const int n_seg = s.cta_of(first + quad_tiles(s.C, p.m, q) - 1) - s.cta_of(first) + 1;
  const float2* part = p.lse_part + (size_t)bh * kMaxLseSplit * p.lse_stride + t;
  float mm = -INFINITY;
  for (int i = 0; i < n_seg; ++i) mm = fmaxf(mm, part[(size_t)i * p.lse_stride].x);
  float ss = 0.f;
  for (int i = 0; i < n_seg; ++i) {
    const float2 v = part[(size_t)i * p.lse_stride];
    if (v.x > -INFINITY) ss += v.y * ex2(v.x - mm);
  }
  p.lse[(size_t)bh * p.lse_stride + t] = mm + log2f(ss);
}

// ---------------------------------------------------------------------------
// Pass 2: for each key i and query quad q,
//   part_q[i] = sum over the quad's queries t with i <= k + t of 2^(x - lse2[t]).
// Accumulator a holds keys x query tile a; the four warps of one TMEM lane
// quarter each sum one query tile and combine their sums in shared memory
// in a fixed order. With one quad the sums are the column sums themselves.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kAttnCtaThreads, 1) curdkv_colsum_kernel(const __grid_constant__ CurdkvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ AttnBars b;
  __shared__ __align__(16) float s_lse[2][kQuad * kTile];
  __shared__ float s_part[2][kQuad][kTile];
  const AttnSched& s = p.sched2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t fixed = tc::smem_u32(smem), stage0 = fixed + kQuad * kTileBytes;
  const long long g0 = s.begin(blockIdx.x), g1 = s.begin(blockIdx.x + 1);
  attn_setup<kColStages>(b);
  const uint32_t tmem = b.tmem_base;
  if (warp == kSoftWarps) {
    if (lane == 0) attn_producer<kColStages>(p, s, b, fixed, stage0, g0, g1);
    __syncwarp();
  } else if (warp == kSoftWarps + 1) {
    if (lane == 0) attn_mma<kColStages, true>(p, s, b, tmem, fixed, stage0, g0, g1);
    __syncwarp();
  } else {
    const int a = warp >> 2, row = 32 * (warp & 3) + lane, tid = threadIdx.x;
    const uint32_t acc = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(a * kTile);
    const float* lse = p.lse;
    UnitCursor u;
    u.init(s, p.m, g0);
    int uses = 0, units = 0;
    bool dead = false;
    for (long long g = g0; g < g1; ++g) {
      const int j = (int)(g - g0);
      const int nq = quad_rows(p.m, u.q);
      if (g == g0 || u.kt == 0) {                  // the quad's lse2, +inf past the last query
        const int t = kQuad * kTile * u.q + tid;
        s_lse[units & 1][tid] = t < p.m ? lse[(size_t)u.bh * p.lse_stride + t] : INFINITY;
        ++units;
        tc::named_sync(1, kSoftWarps * 32);
      }
      const float* l = s_lse[(units - 1) & 1] + kTile * a;
      float part = 0.f;
      if (a < nq && !dead) {
        if (!warp_wait_acc(&b.acc_full[a], (uint32_t)(uses & 1), b, p.err)) dead = true;
        ++uses;
      }
      const bool kept = u.kt < s.C;
      const int base = kept ? p.k - kTile * (s.C - u.kt) : p.k + kTile * (u.kt - s.C);
      const int i = base + row;                    // this thread's key
      if (a < nq && !dead) {
        tc::fence_after_sync();
        const int tq = kQuad * kTile * u.q + kTile * a;            // first query of the accumulator
        const bool full = kept || kTile * (u.kt - s.C) + kTile - 1 <= tq;
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float v[64];
          load64(acc + (uint32_t)(64 * hf), v);
          const float* lh = l + 64 * hf;
          if (full) {
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lh + c);
              sm[0] += ex2(fmaf(v[c], p.scale2, -l4.x));
              sm[1] += ex2(fmaf(v[c + 1], p.scale2, -l4.y));
              sm[2] += ex2(fmaf(v[c + 2], p.scale2, -l4.z));
              sm[3] += ex2(fmaf(v[c + 3], p.scale2, -l4.w));
            }
          } else {
            const int first_t = i - p.k - tq - 64 * hf;              // columns c >= first_t see key i
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= first_t) sm[c & 3] += ex2(fmaf(v[c], p.scale2, -lh[c]));
          }
        }
        part = (sm[0] + sm[1]) + (sm[2] + sm[3]);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&b.acc_empty[a]);
      }
      s_part[j & 1][a][row] = part;
      tc::named_sync(1, kSoftWarps * 32);
      if (a == 0 && !b.fail && i >= 0 && i < p.n) {
        const float* sp = &s_part[j & 1][0][row];
        p.colpart[((size_t)u.q * s.bh_count + u.bh) * p.rows + i] =
            (sp[0] + sp[kTile]) + (sp[2 * kTile] + sp[3 * kTile]);
      }
      u.next(s, p.m);
    }
  }
  attn_teardown(b);
}

// attn[i] = sum of the quads' partial column sums, over the quads whose key
// tiles include row i. grid = (ceil(n / 256), B*H); only launched with two
// or more quads.
__global__ void __launch_bounds__(256) curdkv_colsum_merge_kernel(const __grid_constant__ CurdkvParams p) {
  const AttnSched& s = p.sched2;
  const int bh = blockIdx.y, i = blockIdx.x * 256 + threadIdx.x;
  if (i >= p.n) return;
  float sum = 0.f;
  for (int q = 0; q < s.Q; ++q) {
    if (i >= p.k && (i - p.k) / kTile > quad_tiles(s.C, p.m, q) - s.C - 1) continue;   // not seen by quad q
    sum += p.colpart[((size_t)q * s.bh_count + bh) * p.rows + i];
  }
  p.attn[(size_t)bh * p.rows + i] = sum;
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

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Map of `rows` bf16 rows of 128 elements per (b, h), planes `pitch` rows
// apart; boxes of 64 elements x 128 rows land in the K-major 128-byte-swizzled
// tile layout (one box per 64-element half).
bool encode_rows(CUtensorMap* tm, const void* base, int rows, int pitch, int bh) {
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows, (cuuint64_t)bh};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)pitch * kHeadDim * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tiled()(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Equal contiguous shares of the key tiles for at most `sm_count` CTAs. With
// `bounded_split`, every share holds at least a sixth of the largest unit, so
// a unit spans at most 7 CTAs (the pass-1 partial slots).
AttnSched make_sched(int k, int m, int bh, int sm_count, bool bounded_split) {
  AttnSched s;
  s.C = (k + kTile - 1) / kTile;
  s.Q = (m + kQuad * kTile - 1) / (kQuad * kTile);
  const int largest = quad_tiles(s.C, m, s.Q - 1);
  s.per_bh = quad_prefix(s.C, s.Q - 1) + largest;
  s.bh_count = bh;
  s.total = (long long)s.per_bh * bh;
  long long ctas = std::max(sm_count, 1);
  if (bounded_split) ctas = std::min(ctas, std::max(1LL, s.total / ((largest + 5) / 6)));
  s.ctas = (int)std::min(ctas, s.total);
  return s;
}

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
  st.quads = (h->cfg.max_block + kQuad * kTile - 1) / (kQuad * kTile);
  st.colpart = st.quads > 1 ? reinterpret_cast<float*>(take((size_t)st.quads * bh * st.rows * 4)) : nullptr;
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
  if (!encode_tiled()) return fail(EVICT_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&h->curdkv->sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_lse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn_smem_bytes(kLseStages))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_colsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn_smem_bytes(kColStages))) != cudaSuccess ||
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
  // attention passes: TMA maps of the incoming and kept keys, tile shares
  if (!encode_rows(&p.tm_kin, k, m, m, bh) || (p.k > 0 && !encode_rows(&p.tm_kst, h->kst, p.k, h->cap, bh)))
    return fail(EVICT_EINVAL, "cannot describe the key buffers for TMA (k must be 16-byte aligned)");
  p.sched1 = make_sched(p.k, m, bh, st.sm_count, true);
  p.sched2 = make_sched(p.k, m, bh, st.sm_count, false);
  p.colpart = p.sched2.Q > 1 ? st.colpart : st.attn;
  e = timed_launch(h, kKidCurdkvLse, [&] {
    curdkv_lse_kernel<<<p.sched1.ctas, kAttnCtaThreads, attn_smem_bytes(kLseStages), sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 1 launch");
  e = timed_launch(h, kKidCurdkvLseMerge, [&] {
    curdkv_lse_merge_kernel<<<dim3((m + 255) / 256, bh), 256, 0, sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention merge launch");
  e = timed_launch(h, kKidCurdkvColsum, [&] {
    curdkv_colsum_kernel<<<p.sched2.ctas, kAttnCtaThreads, attn_smem_bytes(kColStages), sm>>>(p);
    return cudaGetLastError();
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 2 launch");
  if (p.sched2.Q > 1) {
    e = timed_launch(h, kKidCurdkvColsumMerge, [&] {
      curdkv_colsum_merge_kernel<<<dim3((n + 255) / 256, bh), 256, 0, sm>>>(p);
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV column-sum merge launch");
  }
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
