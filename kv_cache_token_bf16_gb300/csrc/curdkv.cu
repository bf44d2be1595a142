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
#include <type_traits>

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
  float* gram = nullptr;       // [BH, 128*128]
  float* evec = nullptr;       // [BH, kCurdkvMaxRank, 128]
  float* inv_e = nullptr;      // [BH]
  int rows = 0;                // cap + max_block
  int last_n = 0;              // rows of the last update
  float* colpart = nullptr;    // [quads, BH, rows] per-quad column sums (blocks > 512 rows)
  int quads = 0;               // ceil(max_block / 512)
};

namespace {

constexpr int kTile = 128;                  // rows of a query or key tile
constexpr int kTileBytes = kTile * kHeadDim * 2;
constexpr int kEigThreads = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // bound of every pipeline wait (2 s, far above a tile's time)
constexpr uint32_t kWaitSleepNs = 20000;             // longest hardware sleep per poll
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
  CUtensorMap tm_vin;    // incoming values, as tm_kin
  CUtensorMap tm_vst;    // kept values, as tm_kst
  AttnSched sched1, sched2;
  float* colpart;        // [Q, BH, rows] per-quad column sums (= attn when Q = 1)
  const void* k_in;      // [BH, m, D] bf16
  const void* v_in;
  const void* kst;       // [BH, cap, D] bf16
  const void* vst;
  int k, m, n, cap, heads, rank;
  int units;             // B * H
  float scale2;          // log2(e) / sqrt(D)
  int self_excluded;      // H2O: a new row's column sum leaves out its own query (t > i - k)
  float* lse;
  float2* lse_part;       // [BH, kMaxLseSplit, lse_stride] per-split (max, sum)
  int lse_stride;         // max_block rounded up to 4
  float* attn;
  float* lev;
  int rows;
  float* gram;            // [BH, 128, 128] G of the call
  int gram_cluster;       // CTAs per (b, h) in the Gram kernel
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


__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs: one instruction for two lanes of arithmetic, each lane rounded to nearest
// exactly as the scalar operation would be.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ void split_f32x2(uint64_t x, float& lo, float& hi) {
  lo = __uint_as_float((uint32_t)x);
  hi = __uint_as_float((uint32_t)(x >> 32));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// ex2 of both lanes (the special-function unit takes one value at a time)
__device__ __forceinline__ uint64_t ex2_f32x2(uint64_t x) {
  float lo, hi;
  split_f32x2(x, lo, hi);
  return pack_f32x2(ex2(lo), ex2(hi));
}

// 8 MMAs (K = 128 in steps of 16): D[128 x 128] = A[128 x 128] * B[128 x 128]^T.
// The steps' descriptors differ from the tile's only in the start-address field
// (bits 0-13, byte address / 16): a step adds its offset / 16 to the low word;
// tiles lie below 256 KB of shared memory, so the field never carries over.
__device__ __forceinline__ void issue_tile_mma(uint32_t tmem, uint32_t a, uint32_t b) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kTile, kTile);
  const uint64_t da = tc::sw128_desc(a), db = tc::sw128_desc(b);
  const uint32_t a_lo = (uint32_t)da, b_lo = (uint32_t)db, a_hi = (uint32_t)(da >> 32), b_hi = (uint32_t)(db >> 32);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t off16 = (uint32_t)(((s >> 2) * kTile * 128 + (s & 3) * 32) >> 4);
    tc::mma_bf16(tmem, ((uint64_t)a_hi << 32) | (uint64_t)(a_lo + off16), ((uint64_t)b_hi << 32) | (uint64_t)(b_lo + off16),
                 idesc, s > 0 ? 1u : 0u);
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
// Roles (608 threads): warps 0-15 read the accumulators (warp w: TMEM lanes
// 32 (w % 4) .. +31, accumulator w / 4 = query tile w / 4 of the quad);
// warp 16 issues the TMA loads; warps 17 and 18 issue the MMAs of
// accumulators {0, 2} and {1, 3}. Each query tile has
// its own 128-column fp32 accumulator (512 TMEM columns), so the MMAs of one
// accumulator run while the other three are read. mbarriers connect the
// roles; every wait is bounded and a timeout stops the CTA cleanly.
// ---------------------------------------------------------------------------
constexpr int kQuad = 4;                          // fixed query tiles per unit
constexpr int kSoftWarps = 16;
constexpr int kAttnCtaThreads = (kSoftWarps + 3) * 32;   // + the TMA warp and two MMA warps
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

// Bounded wait on an mbarrier phase. The waiting thread sleeps in hardware
// between polls (no issue slots spent while it waits); it gives up early once
// the CTA's failure flag is set, and after kWaitLimitNs it sets the flag and
// the error word.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* fail, int* err) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tc::global_ns();
  for (;;) {
    if (tc::mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*fail) return false;
    if (tc::global_ns() - t0 > kWaitLimitNs) break;
  }
  *fail = 1;
  raise_device_error(err, kDevWaitTimeout);
  return false;
}
// The same wait ignoring the failure flag: used to let copies and MMAs already
// issued finish before the CTA releases its shared and tensor memory.
__device__ __forceinline__ void drain_phase(uint64_t* bar, uint32_t parity, int* err) {
  if (tc::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = tc::global_ns();
  for (;;) {
    if (tc::mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return;
    if (tc::global_ns() - t0 > kWaitLimitNs) break;
  }
  raise_device_error(err, kDevWaitTimeout);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Shared state of one attention CTA (static shared memory).
constexpr int kPartSlots = 4;                     // pass 2: ring of key tiles' partial column sums
struct AttnBars {
  uint64_t stage_full[kLseStages], stage_empty[kLseStages];
  uint64_t fixed_full, fixed_empty;
  uint64_t acc_full[kQuad], acc_empty[kQuad];
  uint64_t part_full[kPartSlots], part_empty[kPartSlots];
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

// Two MMA-issuing threads, one for accumulators {0, 2} and one for {1, 3}: the
// softmax warps hand the accumulators back one after another, and each thread
// issues its next tile's MMAs as soon as its own accumulators are free, not
// behind the other pair's. Both release the key stage and the fixed tiles
// (those barriers count kMmaThreads arrivals).
constexpr int kMmaThreads = 2;
template <int kStagesT, bool kColsum>
__device__ void attn_mma(const CurdkvParams& p, const AttnSched& s, AttnBars& b, uint32_t tmem, uint32_t fixed,
                         uint32_t stage0, long long g0, long long g1, int first) {
  UnitCursor u;
  u.init(s, p.m, g0);
  int units = 0, uses[2] = {0, 0};
  bool ok = true;
  for (long long g = g0; g < g1 && ok; ++g) {
    const int j = (int)(g - g0);
    if (g == g0 || u.kt == 0) {
      if (!wait_phase(&b.fixed_full, (uint32_t)(units & 1), &b.fail, p.err)) break;
      ++units;
    }
    const int st = j % kStagesT;
    if (!wait_phase(&b.stage_full[st], (uint32_t)((j / kStagesT) & 1), &b.fail, p.err)) break;
    const uint32_t keys = stage0 + st * kTileBytes;
    const int nq = quad_rows(p.m, u.q);
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int a = first + kMmaThreads * x;
      if (a >= nq) continue;
      if (!wait_phase(&b.acc_empty[a], (uint32_t)((uses[x] & 1) ^ 1), &b.fail, p.err)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t q_tile = fixed + a * kTileBytes, d = tmem + (uint32_t)(a * kTile);
      if (kColsum) issue_tile_mma(d, keys, q_tile);
      else issue_tile_mma(d, q_tile, keys);
      tc::mma_commit(&b.acc_full[a]);
      ++uses[x];
    }
    if (!ok) break;
    tc::mma_commit(&b.stage_empty[st]);
    if (u.kt == u.tiles - 1) tc::mma_commit(&b.fixed_empty);
    u.next(s, p.m);
  }
  // the accumulators' last MMAs must finish before TMEM is released
#pragma unroll
  for (int x = 0; x < 2; ++x)
    if (uses[x] > 0) drain_phase(&b.acc_full[first + kMmaThreads * x], (uint32_t)((uses[x] - 1) & 1), p.err);
}

// Bounded, warp-uniform wait of an accumulator-reading warp.
__device__ __forceinline__ bool warp_wait_acc(uint64_t* bar, uint32_t parity, AttnBars& b, int* err) {
  bool ok = wait_phase(bar, parity, &b.fail, err);
  return __all_sync(0xffffffffu, ok);
}

// 64 accumulator columns of this thread's row: one load and its wait in one asm statement, so
// no use of the registers can be scheduled before the data is there.
__device__ __forceinline__ void load64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int c = 0; c < 64; ++c) v[c] = __uint_as_float(r[c]);
}

// Setup shared by both passes: barriers, TMEM, this CTA's share of the tiles.
template <int kStagesT>
__device__ __forceinline__ void attn_setup(AttnBars& b) {
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesT; ++i) {
      tc::mbar_init(&b.stage_full[i], 1);
      tc::mbar_init(&b.stage_empty[i], 2);         // released by both MMA threads
    }
    tc::mbar_init(&b.fixed_full, 1);
    tc::mbar_init(&b.fixed_empty, 2);
    for (int a = 0; a < kQuad; ++a) {
      tc::mbar_init(&b.acc_full[a], 1);
      tc::mbar_init(&b.acc_empty[a], 4);         // the four warps reading accumulator a
    }
    for (int i = 0; i < kPartSlots; ++i) {
      tc::mbar_init(&b.part_full[i], 4 * (kQuad - 1));   // the warps of accumulators 0 .. 2
      tc::mbar_init(&b.part_empty[i], 4);                // the warps of the last accumulator
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
  pdl_wait();
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
  } else if (warp > kSoftWarps) {
    if (lane == 0) attn_mma<kLseStages, false>(p, s, b, tmem, fixed, stage0, g0, g1, warp - kSoftWarps - 1);
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
          if (hf == 1) {                                  // the accumulator is in registers: release it
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&b.acc_empty[a]);
          }
          if (!full) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int i = base + 64 * hf + c;
              if (i < 0 || i > p.k + t) v[c] = -INFINITY;
            }
          }
          // Sum of 2^(x - ref) over the half, x = scale2 * logit: eight running sums (element c
          // into sum c & 7), two per packed register.
          auto half_sum = [&](float ref) {
            uint64_t sm2[4] = {0ull, 0ull, 0ull, 0ull};
            const uint64_t sc2 = pack_f32x2(p.scale2, p.scale2), nr2 = pack_f32x2(-ref, -ref);
#pragma unroll
            for (int c = 0; c < 64; c += 2)
              sm2[(c & 7) >> 1] = add_f32x2(sm2[(c & 7) >> 1], ex2_f32x2(fma_f32x2(pack_f32x2(v[c], v[c + 1]), sc2, nr2)));
            float sm[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) split_f32x2(sm2[j], sm[2 * j], sm[2 * j + 1]);
            return ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
          };
          // The reference is the exact maximum of the query's first visible half. Later halves
          // are summed against it without a maximum of their own while the half's sum stays
          // below 2^64 (no term can then overflow, and terms far below it are negligible next
          // to the reference's own term, 1); otherwise (a much larger logit, +inf, NaN) the
          // half takes its exact maximum and the running sum is rescaled, as lse2 = ref +
          // log2(sum) holds for any reference.
          bool exact = true;
          if (run_max > -INFINITY) {
            const float tot = half_sum(run_max);
            if (tot < 0x1p64f) {
              run_sum += tot;
              exact = false;
            }
          }
          if (exact) {
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
              const float tot = half_sum(nm);
              run_sum = run_sum * ex2(run_max - nm) + tot;         // ex2(-inf) = 0 on the first visible half
              run_max = nm;
            }
          }
        }
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
  pdl_wait();
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
// quarter each sum one query tile. The warps of accumulators 0-2 leave their
// sums in a four-slot shared-memory ring and the warps of accumulator 3 (the
// last one the MMAs fill for a key tile) add them in a fixed order and write
// the result, so the accumulators never wait for each other within a unit.
// With one quad the sums are the column sums themselves.
__global__ void __launch_bounds__(kAttnCtaThreads, 1) curdkv_colsum_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ AttnBars b;
  __shared__ __align__(16) float s_lse[2][kQuad * kTile];
  __shared__ float s_part[kPartSlots][kQuad - 1][kTile];
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
  } else if (warp > kSoftWarps) {
    if (lane == 0) attn_mma<kColStages, true>(p, s, b, tmem, fixed, stage0, g0, g1, warp - kSoftWarps - 1);
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
        s_lse[units & 1][tid] = t < p.m ? -lse[(size_t)u.bh * p.lse_stride + t] : -INFINITY;   // negated
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
        const bool full = kept || kTile * (u.kt - s.C) + kTile - 1 + p.self_excluded <= tq;
        uint64_t s01 = 0ull, s23 = 0ull;                  // sums of columns c & 3 = 0, 1 and 2, 3
        const uint64_t sc2 = pack_f32x2(p.scale2, p.scale2);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          float v[64];
          load64(acc + (uint32_t)(64 * hf), v);
          if (hf == 1) {                                  // the accumulator is in registers: release it
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&b.acc_empty[a]);
          }
          const float* lh = l + 64 * hf;                  // negated lse2 of the columns
          if (full) {
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lh + c);
              s01 = add_f32x2(s01, ex2_f32x2(fma_f32x2(pack_f32x2(v[c], v[c + 1]), sc2, pack_f32x2(l4.x, l4.y))));
              s23 = add_f32x2(s23, ex2_f32x2(fma_f32x2(pack_f32x2(v[c + 2], v[c + 3]), sc2, pack_f32x2(l4.z, l4.w))));
            }
          } else {
            // columns c >= first_t see key i (H2O: from the query after its own)
            const int first_t = i - p.k - tq - 64 * hf + p.self_excluded;
            float sm[4];
            split_f32x2(s01, sm[0], sm[1]);
            split_f32x2(s23, sm[2], sm[3]);
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c >= first_t) sm[c & 3] += ex2(fmaf(v[c], p.scale2, lh[c]));
            s01 = pack_f32x2(sm[0], sm[1]);
            s23 = pack_f32x2(sm[2], sm[3]);
          }
        }
        float sm[4];
        split_f32x2(s01, sm[0], sm[1]);
        split_f32x2(s23, sm[2], sm[3]);
        part = (sm[0] + sm[1]) + (sm[2] + sm[3]);
      }
      const int slot = j % kPartSlots, round = j / kPartSlots;
      if (a < kQuad - 1) {
        // the slot was last used four key tiles ago: wait until the last accumulator read it
        if (round == 0 || wait_phase(&b.part_empty[slot], (uint32_t)((round - 1) & 1), &b.fail, p.err))
          s_part[slot][a][row] = part;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&b.part_full[slot]);
      } else {
        if (wait_phase(&b.part_full[slot], (uint32_t)(round & 1), &b.fail, p.err) && !b.fail && i >= 0 &&
            i < p.n) {
          const float* sp = &s_part[slot][0][row];
          p.colpart[((size_t)u.q * s.bh_count + u.bh) * p.rows + i] = (sp[0] + sp[kTile]) + (sp[2 * kTile] + part);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&b.part_empty[slot]);
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
  pdl_wait();
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

// H2O-adapted cumulative mass ("CurDKV-adapted", §How it works step 1: the
// proxy softmax H2O uses; §The honesty crux item 4: a new token starts from
// 0): kept rows add their column sum to the stored score, new rows start
// from theirs (their own query already left out by the column-sum pass).
// grid = (ceil(n / 256), B*H).
__global__ void __launch_bounds__(256) h2o_mass_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  const int bh = blockIdx.y, i = blockIdx.x * 256 + threadIdx.x;
  if (i >= p.n) return;
  const float a = p.attn[(size_t)bh * p.rows + i];
  p.lev[(size_t)bh * p.rows + i] = a;
  if (i < p.k) p.score_st[(size_t)bh * p.cap + i] += a;
  else p.new_score[(size_t)bh * p.new_stride + (i - p.k)] = a;
}

// ---------------------------------------------------------------------------
// Proxy attention of a short block, one CTA per (b, h): the quantities of the
// three tensor-core passes (logits k_i . q_t / sqrt(D) in base 2, each
// query's softmax over its rows i <= k + t, column sums a_i) computed with
// fp32 FMAs in one kernel. A decode step has one query per unit, which would
// fill one row of a 128-row MMA tile; here the work is one dot product per
// key. Used when m <= kSmallAttnMaxM and the m x n logits fit shared memory;
// kM (1, 2, 4 or 8) is m rounded up, so a decode step holds one query in
// registers and keeps eight rows per half-warp in flight (a unit's keys are
// read at the rate its loads in flight allow). For H2O (self_excluded) it
// also applies the mass update of h2o_mass_kernel.
//   1. a half-warp per key row: lane c holds elements 8c .. 8c+7 of the row
//      and of every query, and xor shuffles sum the 16 partial products; the
//      logits go to shared memory, [t][i].
//   2. per query: the maximum over its rows, then the sum of 2^(l - max),
//      the terms overwriting the logits (block reductions of all m queries at
//      once, in a fixed order).
//   3. per row: a_i = sum over the queries that see row i of term / sum
//      (H2O: a new row's own query left out).
// ---------------------------------------------------------------------------
constexpr int kSmallAttnMaxM = 8;
constexpr int kSmallAttnMaxLogits = 16384;       // 64 KB of fp32 logits
constexpr int kSmallAttnThreads = 512;
constexpr int kSmallAttnWarps = kSmallAttnThreads / 32;
constexpr int kSmallAttnHalfWarps = kSmallAttnThreads / 16;

__host__ __device__ constexpr bool small_attn_fits(int m, int n) {
  return m >= 1 && m <= kSmallAttnMaxM && (long long)m * n <= kSmallAttnMaxLogits;
}

template <int kM>
__global__ void __launch_bounds__(kSmallAttnThreads) curdkv_attn_small_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  static_assert(kM >= 1 && kM <= kSmallAttnMaxM, "queries per CTA");
  extern __shared__ __align__(16) float s_term[];            // [m][n]: logits, then 2^(l - max)
  __shared__ float s_red[kSmallAttnWarps][kSmallAttnMaxM];
  __shared__ float s_max[kSmallAttnMaxM], s_inv[kSmallAttnMaxM];
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = tid & 15, hw = tid >> 4;
  const int m = p.m, k = p.k, n = p.n;
  const uint4* qin = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.k_in) + (size_t)bh * m * kHeadDim);
  const uint4* kept = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.kst) + (size_t)bh * p.cap * kHeadDim);
  constexpr int kRowVecs = kHeadDim / 8;                    // 16-byte pieces per row
  float q[kM][8];
#pragma unroll
  for (int t = 0; t < kM; ++t) {
    if (t < m) {
      bf16x8_to_f32(__ldg(qin + (size_t)t * kRowVecs + c), q[t]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[t][e] = 0.f;
    }
  }
  // 1. logits, kRowsInFlight rows of the half-warp in flight; the trip count follows the warp's
  // first row (2 warp), so both half-warps run every shuffle together
  constexpr int kRowsInFlight = kM <= 2 ? 8 : 4;
  constexpr int kStep = kSmallAttnHalfWarps * kRowsInFlight;
  for (int i0 = hw, w0 = 2 * warp; w0 < n; i0 += kStep, w0 += kStep) {
    uint4 r[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int i = i0 + kSmallAttnHalfWarps * u;
      r[u] = make_uint4(0, 0, 0, 0);
      if (i < n) r[u] = __ldg((i < k ? kept + (size_t)i * kRowVecs : qin + (size_t)(i - k) * kRowVecs) + c);
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int i = i0 + kSmallAttnHalfWarps * u;
      float x[8];
      bf16x8_to_f32(r[u], x);
#pragma unroll
      for (int t = 0; t < kM; ++t) {
        if (t < m) {
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) d = fmaf(x[e], q[t][e], d);
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          if (c == t && i < n) s_term[t * n + i] = d * p.scale2;
        }
      }
    }
  }
  __syncthreads();
  // 2. per query: maximum, then the sum of the terms
  float acc[kM];
#pragma unroll
  for (int t = 0; t < kM; ++t) acc[t] = -INFINITY;
  for (int i = tid; i < n; i += kSmallAttnThreads)
#pragma unroll
    for (int t = 0; t < kM; ++t)
      if (t < m && i <= k + t) acc[t] = fmaxf(acc[t], s_term[t * n + i]);
#pragma unroll
  for (int t = 0; t < kM; ++t) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[t] = fmaxf(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], o));
    if (lane == 0) s_red[warp][t] = acc[t];
  }
  __syncthreads();
  if (tid < m) {
    float mx = s_red[0][tid];
    for (int w = 1; w < kSmallAttnWarps; ++w) mx = fmaxf(mx, s_red[w][tid]);
    s_max[tid] = mx;                                         // finite: row 0 is seen by every query
  }
  __syncthreads();
#pragma unroll
  for (int t = 0; t < kM; ++t) acc[t] = 0.f;
  for (int i = tid; i < n; i += kSmallAttnThreads)
#pragma unroll
    for (int t = 0; t < kM; ++t)
      if (t < m) {
        const float e = i <= k + t ? exp2f(s_term[t * n + i] - s_max[t]) : 0.f;
        s_term[t * n + i] = e;
        acc[t] += e;
      }
#pragma unroll
  for (int t = 0; t < kM; ++t) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
    if (lane == 0) s_red[warp][t] = acc[t];
  }
  __syncthreads();
  if (tid < m) {
    float sum = s_red[0][tid];
    for (int w = 1; w < kSmallAttnWarps; ++w) sum += s_red[w][tid];
    s_inv[tid] = 1.f / sum;                                  // >= 1: the maximum's own term
  }
  __syncthreads();
  // 3. column sums (each thread reads back only the terms it wrote)
  for (int i = tid; i < n; i += kSmallAttnThreads) {
    float a = 0.f;
#pragma unroll
    for (int t = 0; t < kM; ++t)
      if (t < m && !(p.self_excluded && i == k + t)) a = fmaf(s_term[t * n + i], s_inv[t], a);
    p.attn[(size_t)bh * p.rows + i] = a;
    if (p.self_excluded) {
      p.lev[(size_t)bh * p.rows + i] = a;
      if (i < k) p.score_st[(size_t)bh * p.cap + i] += a;
      else p.new_score[(size_t)bh * p.new_stride + (i - k)] = a;
    }
  }
}

// ---------------------------------------------------------------------------
// Gram of the weighted values on the tensor cores: G = sum_i a_i^2 v_i v_i^T.
//
// A cluster of S CTAs per (b, h). The unit's value rows are cut into 128-row
// tiles (kept rows from row 0, then incoming rows from row k) and CTA c of the
// cluster takes a contiguous share of them. TMA streams each tile in its
// natural layout (tokens x features), which makes tokens the contraction
// dimension and features the M and N dimensions: both MMA operands are
// MN-major, so nothing is transposed. A = the value tile (exact in bf16);
// B = a^2 v split into bf16 hi + lo (~16 significant bits; the remainder is
// below 2^-17 of each term), two MMAs per 16-token step, fp32 accumulation
// in TMEM. The cluster then sums its S partials through distributed shared
// memory in a fixed order (CTA c writes rows [c R, (c+1) R) of G), so the
// result does not depend on timing.
//
// Roles (320 threads): warp 0 issues the TMA loads, warp 1 the MMAs, warps
// 2-9 write the hi / lo tiles (packed fp32x2 arithmetic) and read the
// accumulator. Rows past the valid range of a tile are zero (TMA fill), so
// they add nothing.
// ---------------------------------------------------------------------------
constexpr int kGramVStages = 3, kGramHStages = 2;
constexpr int kGramConvWarps = 8;
constexpr int kGramThreads = (2 + kGramConvWarps) * 32;
constexpr int kGramMaxCluster = 8;
constexpr int kGramRedPitch = kHeadDim + 4;         // floats per row of the reduction buffer
constexpr int kGramSmem = (kGramVStages + 2 * kGramHStages) * kTileBytes + 1024;
static_assert(kHeadDim * kGramRedPitch * 4 <= kGramVStages * kTileBytes, "reduction buffer fits the value ring");

struct GramBars {
  uint64_t v_full[kGramVStages], v_empty[kGramVStages];
  uint64_t h_full[kGramHStages], h_empty[kGramHStages];
  uint64_t done;
  uint32_t tmem_base;
  int fail;
};


__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo_elem, hi_elem);   // .x (low half) = lo_elem
  return *reinterpret_cast<const uint32_t*>(&b);
}

__global__ void __launch_bounds__(kGramThreads, 1) curdkv_gram_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ GramBars b;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.gram_cluster;
  const int rank = (int)tc::cluster_rank();
  const int bh = blockIdx.x / S;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t vring = tc::smem_u32(smem);
  const uint32_t hring = vring + kGramVStages * kTileBytes;   // stage s: hi at 2s, lo at 2s+1
  const int Ck = (p.k + kTile - 1) / kTile, Cm = (p.m + kTile - 1) / kTile;
  const int T = Ck + Cm;
  const int t0 = (int)((long long)T * rank / S), t1 = (int)((long long)T * (rank + 1) / S);
  if (tid == 0) {
    for (int i = 0; i < kGramVStages; ++i) {
      tc::mbar_init(&b.v_full[i], 1);
      tc::mbar_init(&b.v_empty[i], 1);
    }
    for (int i = 0; i < kGramHStages; ++i) {
      tc::mbar_init(&b.h_full[i], kGramConvWarps);     // one arrival per converting warp
      tc::mbar_init(&b.h_empty[i], 1);
    }
    tc::mbar_init(&b.done, 1);
    b.fail = 0;
  }
  if (warp == 2) tc::tmem_alloc(&b.tmem_base, kTile);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0) {
    if (lane == 0 && t1 > t0) {                         // TMA producer
      tc::tma_prefetch_desc(&p.tm_vin);
      if (Ck > 0) tc::tma_prefetch_desc(&p.tm_vst);
      int issued[kGramVStages] = {0, 0, 0};
      for (int i = t0; i < t1; ++i) {
        const int j = i - t0, st = j % kGramVStages;
        if (!wait_phase(&b.v_empty[st], (uint32_t)(((j / kGramVStages) & 1) ^ 1), &b.fail, p.err)) break;
        tc::mbar_arrive_expect_tx(&b.v_full[st], (uint32_t)kTileBytes);
        const bool kept = i < Ck;
        const void* map = kept ? (const void*)&p.tm_vst : (const void*)&p.tm_vin;
        const int y = kept ? kTile * i : kTile * (i - Ck);
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(vring + st * kTileBytes + hf * (kTileBytes / 2), map, 64 * hf, y, bh, &b.v_full[st]);
        ++issued[st];
      }
      for (int i = 0; i < kGramVStages; ++i)
        if (issued[i] > 0) drain_phase(&b.v_full[i], (uint32_t)((issued[i] - 1) & 1), p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && t1 > t0) {                         // MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16_f32_mn(kTile, kTile);
      for (int i = t0; i < t1; ++i) {
        const int j = i - t0, vs = j % kGramVStages, hs = j % kGramHStages;
        if (!wait_phase(&b.v_full[vs], (uint32_t)((j / kGramVStages) & 1), &b.fail, p.err)) break;
        if (!wait_phase(&b.h_full[hs], (uint32_t)((j / kGramHStages) & 1), &b.fail, p.err)) break;
        tc::fence_after_sync();
        const uint32_t va = vring + vs * kTileBytes, hi = hring + 2 * hs * kTileBytes, lo = hi + kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint32_t off = (uint32_t)ks * 2048u;   // 16 tokens = two 8-token groups of 1024 bytes
          const uint64_t ad = tc::sw128_desc_mn(va + off, kTileBytes / 2, 1024);
          tc::mma_bf16(tmem, ad, tc::sw128_desc_mn(hi + off, kTileBytes / 2, 1024), idesc, (j > 0 || ks > 0) ? 1u : 0u);
          tc::mma_bf16(tmem, ad, tc::sw128_desc_mn(lo + off, kTileBytes / 2, 1024), idesc, 1u);
        }
        tc::mma_commit(&b.v_empty[vs]);
        tc::mma_commit(&b.h_empty[hs]);
      }
      tc::mma_commit(&b.done);                          // after every MMA issued (also on a failure)
      drain_phase(&b.done, 0, p.err);                   // none may run once TMEM is released
    }
    __syncwarp();
  } else {                                              // converters: a^2 v -> bf16 hi + lo
    const int ct = tid - 64;                            // 0 .. 255
    const int p16 = ct & 7;                             // 16-byte chunk position inside a row
    const float* attn = p.attn + (size_t)bh * p.rows;
    // this thread's four tokens' weights a^2, loaded one tile ahead
    float asq_next[4];
    auto load_asq = [&](int i, float (&dst)[4]) {
      const bool kept = i < Ck;
      const int base = kept ? kTile * i : p.k + kTile * (i - Ck);
      const int lim = kept ? p.k : p.k + p.m;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int gi = base + (ct >> 3) + 32 * rr;
        const float av = (i < t1 && gi < lim) ? attn[gi] : 0.f;
        dst[rr] = av * av;
      }
    };
    load_asq(t0, asq_next);
    for (int i = t0; i < t1; ++i) {
      const int j = i - t0, vs = j % kGramVStages, hs = j % kGramHStages;
      float asq_cur[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) asq_cur[rr] = asq_next[rr];
      load_asq(i + 1, asq_next);
      bool ok = wait_phase(&b.v_full[vs], (uint32_t)((j / kGramVStages) & 1), &b.fail, p.err);
      ok = ok && wait_phase(&b.h_empty[hs], (uint32_t)(((j / kGramHStages) & 1) ^ 1), &b.fail, p.err);
      if (!__all_sync(0xffffffffu, ok)) break;
      const unsigned char* vt = smem + vs * kTileBytes;
      unsigned char* ht = smem + (kGramVStages + 2 * hs) * kTileBytes;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int row = (ct >> 3) + 32 * rr;            // token of this thread's chunks
        const uint64_t asq2 = pack_f32x2(asq_cur[rr], asq_cur[rr]);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int off = hf * (kTileBytes / 2) + row * 128 + p16 * 16;
          const uint4 raw = *reinterpret_cast<const uint4*>(vt + off);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t y = mul_f32x2(pack_f32x2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u)), asq2);
            const float y0 = __uint_as_float((uint32_t)y), y1 = __uint_as_float((uint32_t)(y >> 32));
            hw[q] = pack_bf16x2(y0, y1);
            const uint64_t r = sub_f32x2(y, pack_f32x2(__uint_as_float(hw[q] << 16), __uint_as_float(hw[q] & 0xffff0000u)));
            lw[q] = pack_bf16x2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
          }
          *reinterpret_cast<uint4*>(ht + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(ht + kTileBytes + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b.h_full[hs]);
    }
    // accumulator -> reduction buffer (row f = feature, padded rows); the two
    // warps of a TMEM lane quarter take 64 columns each
    const bool have = t1 > t0;
    bool ok = !have || wait_phase(&b.done, 0, &b.fail, p.err);
    ok = __all_sync(0xffffffffu, ok);
    tc::fence_after_sync();
    const int f = 32 * (warp & 3) + lane;               // TMEM lane quarter of this warp
    const int cbase = ((warp - 2) >> 2) * 64;
    float* red = reinterpret_cast<float*>(smem) + (size_t)f * kGramRedPitch;
#pragma unroll 1
    for (int c0 = cbase; c0 < cbase + 64; c0 += 32) {
      float v[32];
      if (have && ok) {
        tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0, v);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) v[c] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4*>(red + c0 + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
    }
  }
  tc::fence_before_sync();
  tc::cluster_sync();                                   // every partial is in its CTA's shared memory
  tc::fence_after_sync();
  {
    const int rows_per = (kHeadDim + S - 1) / S;
    const int f0 = rank * rows_per, f1 = min(kHeadDim, f0 + rows_per);
    float* out = p.gram + (size_t)bh * kHeadDim * kHeadDim;
    const uint32_t red0 = tc::smem_u32(smem);
    for (int item = tid; item < (f1 - f0) * (kHeadDim / 4); item += kGramThreads) {
      const int f = f0 + item / (kHeadDim / 4), c = 4 * (item % (kHeadDim / 4));
      const uint32_t off = (uint32_t)((f * kGramRedPitch + c) * 4);
      float4 acc = tc::ld_cluster_f4(tc::map_to_rank(red0 + off, 0));
      for (int sr = 1; sr < S; ++sr) {
        const float4 v = tc::ld_cluster_f4(tc::map_to_rank(red0 + off, (uint32_t)sr));
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      *reinterpret_cast<float4*>(out + (size_t)f * kHeadDim + c) = acc;
    }
  }
  tc::cluster_sync();                                   // no CTA leaves while others read its memory
  if (warp == 2) tc::tmem_dealloc(tmem, kTile);
}

// ---------------------------------------------------------------------------
// Top-r eigenvectors of G (symmetric, 128 x 128), one CTA of 128 threads per
// (b, h). G is normalised by its trace and held in registers: warp w owns
// rows 32 w .. +31 (whole rows, so A v needs no reduction across warps);
// lane (lr, lc) = (lane / 8, lane % 8) owns rows R0 = 32 w + 8 lr .. +7 and
// the columns 64 h + 8 lc .. +7 for h = 0, 1 (a[h][i][c]).
//
// Phases:
//   1. Householder tridiagonalisation, one CTA barrier per step (below).
//   2. Multisection (Sturm counts) for the top r eigenvalues of T.
//   3. Inverse iteration on T (one lane per eigenvalue).
//   4. Cholesky QR, two passes, to re-orthonormalise the r vectors.
//   5. Back-transformation through the Householder reflections in blocks of
//      eight (one reduction per block).
// ---------------------------------------------------------------------------
constexpr int kEigSteps = kHeadDim - 2;            // Householder steps
// |x|^2 below which a column of the unit-trace matrix counts as already
// reduced and its reflection is skipped: its entries (< 1e-8) lie under the
// fp32 rounding of the matrix (1.2e-7 of its norm, which is at most 1), and
// beta = 1 / (sigma (sigma + |x0|)) stays below 1e16, so that the 0.5 beta^2
// of the next update stays in range. Nearly rank-deficient G (a proxy query
// that attends almost only to itself) leave columns of rounding noise that
// shrink step by step and would otherwise overflow beta^2 into inf and NaN.
constexpr float kEigTinyColumn = 1e-16f;
constexpr int kZPad = kHeadDim + 4;                // padded vector rows
constexpr int kBtBlock = 8;                        // reflections per back-transform block
constexpr int kBtBlocks = (kEigSteps + kBtBlock - 1) / kBtBlock;
constexpr int kEigWarps = kEigThreads / 32;
static_assert(kEigWarps == 4, "the eigensolver layout assumes four warps of 32 rows");

// The Householder vectors are stored as packed rows: v_j is exactly zero at
// indices <= j, so row j keeps only its float4 chunks from (j + 1) / 4 on
// (16-byte aligned, about half of the square array). Chunk c of row j sits at
// hv_row_base(j) + 4 (c - hv_first_chunk(j)); the chunks before it read as 0.
__host__ __device__ constexpr int hv_first_chunk(int j) { return (j + 1) >> 2; }
__host__ __device__ constexpr int hv_row_base(int j) {
  // 4 * sum_{t < j} (32 - hv_first_chunk(t)), with sum_{u=1..j} floor(u / 4) in closed form
  return 4 * (32 * j - (2 * (j >> 2) * ((j >> 2) - 1) + (j >> 2) * ((j & 3) + 1)));
}
constexpr int kHvFloats = hv_row_base(kEigSteps);
static_assert(hv_row_base(1) == 128 && hv_row_base(4) == 4 * (4 * 32 - 1) && kHvFloats == 8316,
              "packed Householder rows");

__device__ __forceinline__ float4 hv_chunk(const float* hv, int j, int c) {
  const int c0 = hv_first_chunk(j);
  return c < c0 ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(hv + hv_row_base(j) + 4 * (c - c0));
}

// Shared memory of the eigensolver for up to kR eigenvectors: 106 KB for
// kR = 16 (two CTAs per SM), 166 KB for kR = 32.
template <int kR>
struct EigSmem {
  float hv[kHvFloats];                             // Householder vectors v_j, packed rows
  float lu[5][kHeadDim][kR];                       // inverse-iteration LU factors, [factor][row][vector]
  float z[kR][kZPad];                              // eigenvectors (tridiagonal basis)
  float zt[kHeadDim][kR];                          // the same during inverse iteration, [row][vector]
  float vs[2][kHeadDim];                           // v of the step (by step parity)
  float cb[2][kHeadDim];                           // the next column before the step's update
  float pp[2][kHeadDim];                           // A v of the step
  float kp[2][kEigWarps];                          // per-warp partials of v . A v
  float wv[kEigWarps][3][kHeadDim];                // warp-private: v_{j-1}, w_{j-1}, x_j of every row
  float vtv[kBtBlocks][kBtBlock][kBtBlock];        // v_k . v_m within a back-transform block
  float beta[kHeadDim], d[kHeadDim], e[kHeadDim];
  float2 de2[kHeadDim];                            // {d[i], e[i-1]^2} for the Sturm counts
  float gram[kR][kR + 1];
  float lam[kR];
  double diag[kHeadDim];
  double trace;
  float tnorm;
};

__device__ __forceinline__ float hash_unit(int i, int j) {
  uint32_t h = (uint32_t)i * 2654435761u ^ (uint32_t)(j + 1) * 2246822519u;
  h ^= h >> 15;
  h *= 2654435761u;
  h ^= h >> 13;
  return (float)(h & 0xFFFFu) * (1.f / 65536.f) - 0.5f;
}

// Number of eigenvalues of the tridiagonal T that are <= x, for two shifts at
// once: the sign changes of the leading principal minors of T - x I,
//   p_0 = 1, p_1 = d_0 - x, p_{i+1} = (d_i - x) p_i - e_{i-1}^2 p_{i-1}.
// This is the pivot recurrence q_i = p_i / p_{i-1} without its division
// (the same rounding behaviour up to scaling); a minor smaller than 2^-24 of
// its predecessor counts as a negative pivot, and every fourth step both
// minors are scaled by the exact power of two that brings the larger into
// [1, 2). T is similar to a unit-trace positive semi-definite matrix, so
// |d|, |e| <= 1 and |x| <= 1.01 tnorm <= 3.03: a step multiplies the larger
// minor by at most 5.03, the guard keeps each minor at least 2^-24 of its
// predecessor, and a minor is at most 4.03 + 2^24 times its predecessor. So
// after a scaling both minors are at least about 2^-24, and four steps later
// every minor lies in [2^-121, 2^11]: none becomes subnormal or overflows,
// and exact power-of-two scaling changes no count.
__device__ __forceinline__ void sturm_count2(const float2* de2, const float (&x)[2], int (&cnt)[2]) {
  constexpr float kTiny = 5.9604645e-08f;          // 2^-24
  float u[2], v[2];
  const float d0 = de2[0].x;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    u[k] = 1.f;
    v[k] = d0 - x[k];
    if (fabsf(v[k]) < kTiny) v[k] = -kTiny;
    cnt[k] = v[k] < 0.f ? 1 : 0;
  }
  float2 tn = de2[1];
#pragma unroll 4
  for (int i = 1; i < kHeadDim; ++i) {
    const float2 t = tn;
    if (i + 1 < kHeadDim) tn = de2[i + 1];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float g = kTiny * v[k];
      float w = fmaf(t.x - x[k], v[k], -t.y * u[k]);
      if (fabsf(w) < fabsf(g)) w = -g;
      cnt[k] += (int)((__float_as_uint(w) ^ __float_as_uint(v[k])) >> 31);
      u[k] = v[k];
      v[k] = w;
    }
    if ((i & 3) == 3) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int ex = (int)((__float_as_uint(fmaxf(fabsf(u[k]), fabsf(v[k]))) >> 23) & 0xff) - 127;
        const float sc = __uint_as_float((uint32_t)(127 - ex) << 23);
        u[k] *= sc;
        v[k] *= sc;
      }
    }
  }
}

__device__ __forceinline__ float eig_xval(float cbq, float vq, float wq, float omega, float nu) {
  return fmaf(-vq, omega, fmaf(-wq, nu, cbq));
}

template <bool kBoth>
struct EigHalves {
  static constexpr int kFirst = kBoth ? 0 : 1;     // first live column half
  static constexpr int kOwnHalf = kBoth ? 0 : 1;   // half holding column j + 1
};

template <int kR>
__global__ void __launch_bounds__(kEigThreads, kR <= 16 ? 2 : 1)
    curdkv_eig_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  extern __shared__ __align__(16) unsigned char eig_raw[];
  EigSmem<kR>& s = *reinterpret_cast<EigSmem<kR>*>(eig_raw);
  const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int n = kHeadDim;
  const int r = p.rank;
  float* evec_out = p.evec + (size_t)bh * kCurdkvMaxRank * n;
  const int lr = lane >> 3, lc = lane & 7;
  const int R0 = 32 * warp + 8 * lr;

  // --- G (summed by the Gram kernel's cluster); E = trace G in fp64 --------
  float a[2][8][8];
  {
    const float* src = p.gram + (size_t)bh * n * n + (size_t)R0 * n + 8 * lc;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(src + i * n + 64 * h));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(src + i * n + 64 * h + 4));
        a[h][i][0] = u0.x; a[h][i][1] = u0.y; a[h][i][2] = u0.z; a[h][i][3] = u0.w;
        a[h][i][4] = u1.x; a[h][i][5] = u1.y; a[h][i][6] = u1.z; a[h][i][7] = u1.w;
      }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (R0 == 64 * h + 8 * lc) {
#pragma unroll
      for (int i = 0; i < 8; ++i) s.diag[R0 + i] = (double)a[h][i][i];
    }
  __syncthreads();
  if (warp == 0) {
    double t = ((s.diag[4 * lane] + s.diag[4 * lane + 1]) + s.diag[4 * lane + 2]) + s.diag[4 * lane + 3];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s.trace = t;
  }
  __syncthreads();
  if (!(s.trace > 0.0)) {
    for (int el = tid; el < kCurdkvMaxRank * n; el += kEigThreads) evec_out[el] = 0.f;
    if (tid == 0) p.inv_e[bh] = 0.f;
    return;
  }
  if (tid == 0) p.inv_e[bh] = (float)(1.0 / s.trace);
  {
    const float sc = (float)(1.0 / s.trace);         // normalise: eigenvectors unchanged
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) a[h][i][c] *= sc;
  }

  // --- 1. Householder tridiagonalisation -------------------------------------
  // Step j: x = column j below the diagonal (zeros at rows <= j), sigma = |x|,
  // v = x + delta e_{j+1}, beta = 2 / |v|^2, p = beta A v, K = beta/2 v.p,
  // w = p - K v, A -= v w^T + w v^T (rows and columns > j only).
  //
  // One CTA barrier per step. Before the barrier of step j-1 the owners of
  // column j publish it as it stands before step j-1's update (cb), and A v,
  // the per-warp partials of v.A v and v itself are published. After it each
  // warp forms, four rows per lane, w_{j-1} = beta A v - K v and
  //   x_j = cb - v_{j-1} w_{j-1}[j] - w_{j-1} v_{j-1}[j]
  // with |x_j|^2 (the same bits in every warp), keeps them in a warp-private
  // buffer, and every thread applies step j-1's update fused with A x_j; the
  // owners of column j+1 then add delta A[:, j+1] (v = x + delta e_{j+1}).
  // The fused pass has no branch, so its multiply-adds overlap the scalar
  // chain of the step; a warp whose rows are all finished computes values
  // that nobody reads. After step 62 the first column half is finished and a
  // second copy of the loop skips it.
  if (lc == 0) {
    *reinterpret_cast<float4*>(&s.cb[1][R0]) = make_float4(a[0][0][0], a[0][1][0], a[0][2][0], a[0][3][0]);
    *reinterpret_cast<float4*>(&s.cb[1][R0 + 4]) = make_float4(a[0][4][0], a[0][5][0], a[0][6][0], a[0][7][0]);
  }
  s.vs[1][tid] = 0.f;
  s.pp[1][tid] = 0.f;
  if (tid < kEigWarps) s.kp[1][tid] = 0.f;
  __syncthreads();

  float beta_prev = 0.f;
  float* wv = &s.wv[warp][0][0];
  auto step = [&](auto both_tag, int j) {
    constexpr bool kBoth = decltype(both_tag)::value;
    constexpr int kFirst = EigHalves<kBoth>::kFirst, kOwnHalf = EigHalves<kBoth>::kOwnHalf;
    const int b = j & 1, bp = b ^ 1;
    float Kp;
    {
      const float4 k4 = *reinterpret_cast<const float4*>(&s.kp[bp][0]);
      Kp = 0.5f * beta_prev * beta_prev * ((k4.x + k4.y) + (k4.z + k4.w));
    }
    const float nu = s.vs[bp][j];
    const float omega = fmaf(-Kp, nu, beta_prev * s.pp[bp][j]);
    // v_{j-1}, w_{j-1}, x_j of rows 4 lane .. +3 (warp-private), |x_j|^2; x_j stays in xq
    float ss = 0.f;
    float xq[4];
    {
      const int q0 = 4 * lane;
      const float4 c4 = *reinterpret_cast<const float4*>(&s.cb[bp][q0]);
      const float4 v4 = *reinterpret_cast<const float4*>(&s.vs[bp][q0]);
      const float4 p4 = *reinterpret_cast<const float4*>(&s.pp[bp][q0]);
      const float cq[4] = {c4.x, c4.y, c4.z, c4.w}, vq[4] = {v4.x, v4.y, v4.z, v4.w};
      const float pq[4] = {p4.x, p4.y, p4.z, p4.w};
      float wq[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int q = q0 + k;
        wq[k] = fmaf(-Kp, vq[k], q > j - 1 ? beta_prev * pq[k] : 0.f);
        const float val = eig_xval(cq[k], vq[k], wq[k], omega, nu);
        if (warp == 0 && q == j) s.d[j] = val;
        xq[k] = q > j ? val : 0.f;
        ss = fmaf(xq[k], xq[k], ss);
      }
      *reinterpret_cast<float4*>(wv + q0) = v4;
      *reinterpret_cast<float4*>(wv + n + q0) = make_float4(wq[0], wq[1], wq[2], wq[3]);
      *reinterpret_cast<float4*>(wv + 2 * n + q0) = make_float4(xq[0], xq[1], xq[2], xq[3]);
    }
    __syncwarp();
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float x0 = wv[2 * n + j + 1];
    const float tail = ss - x0 * x0;
    // branch-free (selects), so that this chain and the update below share one basic block
    const bool reflect = tail > 0.f && ss > kEigTinyColumn;
    const float ssr = reflect ? ss : 1.f;
    const float sigma = ssr * rsqrtf(ssr);
    const float alpha = reflect ? (x0 >= 0.f ? -sigma : sigma) : x0;
    const float delta = reflect ? -alpha : 0.f;         // v[j+1] = x0 - alpha
    const float beta = reflect ? __fdividef(1.f, sigma * (sigma + fabsf(x0))) : 0.f;
    // this thread's rows: v_{j-1}, w_{j-1}, x_j
    float pvr[8], pwr[8], xr[8];
    {
      const float4 v0 = *reinterpret_cast<const float4*>(wv + R0), v1 = *reinterpret_cast<const float4*>(wv + R0 + 4);
      const float4 w0 = *reinterpret_cast<const float4*>(wv + n + R0);
      const float4 w1 = *reinterpret_cast<const float4*>(wv + n + R0 + 4);
      const float4 x0v = *reinterpret_cast<const float4*>(wv + 2 * n + R0);
      const float4 x1v = *reinterpret_cast<const float4*>(wv + 2 * n + R0 + 4);
      pvr[0] = v0.x; pvr[1] = v0.y; pvr[2] = v0.z; pvr[3] = v0.w; pvr[4] = v1.x; pvr[5] = v1.y; pvr[6] = v1.z; pvr[7] = v1.w;
      pwr[0] = w0.x; pwr[1] = w0.y; pwr[2] = w0.z; pwr[3] = w0.w; pwr[4] = w1.x; pwr[5] = w1.y; pwr[6] = w1.z; pwr[7] = w1.w;
      xr[0] = x0v.x; xr[1] = x0v.y; xr[2] = x0v.z; xr[3] = x0v.w; xr[4] = x1v.x; xr[5] = x1v.y; xr[6] = x1v.z; xr[7] = x1v.w;
    }
    // step j-1's update fused with A x_j (column halves from kFirst)
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
    for (int h = kFirst; h < 2; ++h) {
      const int cb0 = 64 * h + 8 * lc;
      float pvc[8], pwc[8], xc[8];
      {
        const float4 v0 = *reinterpret_cast<const float4*>(wv + cb0);
        const float4 v1 = *reinterpret_cast<const float4*>(wv + cb0 + 4);
        const float4 w0 = *reinterpret_cast<const float4*>(wv + n + cb0);
        const float4 w1 = *reinterpret_cast<const float4*>(wv + n + cb0 + 4);
        const float4 x0v = *reinterpret_cast<const float4*>(wv + 2 * n + cb0);
        const float4 x1v = *reinterpret_cast<const float4*>(wv + 2 * n + cb0 + 4);
        pvc[0] = v0.x; pvc[1] = v0.y; pvc[2] = v0.z; pvc[3] = v0.w; pvc[4] = v1.x; pvc[5] = v1.y; pvc[6] = v1.z; pvc[7] = v1.w;
        pwc[0] = w0.x; pwc[1] = w0.y; pwc[2] = w0.z; pwc[3] = w0.w; pwc[4] = w1.x; pwc[5] = w1.y; pwc[6] = w1.z; pwc[7] = w1.w;
        xc[0] = x0v.x; xc[1] = x0v.y; xc[2] = x0v.z; xc[3] = x0v.w; xc[4] = x1v.x; xc[5] = x1v.y; xc[6] = x1v.z; xc[7] = x1v.w;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float val = fmaf(-pvr[i], pwc[c], fmaf(-pwr[i], pvc[c], a[h][i][c]));
          a[h][i][c] = val;
          acc[i] = fmaf(val, xc[c], acc[i]);
        }
    }
    // column j+1 (updated through step j-1): delta A[:, j+1] completes A v_j;
    // its owners publish it for the next step
    const int j1 = j + 1;
    const bool own1 = 64 * kOwnHalf + 8 * lc == (j1 & ~7);
    float col[8];
    switch (j1 & 7) {
#define EIG_COL_CASE(c)                                                 \
  case c:                                                               \
    for (int i = 0; i < 8; ++i) col[i] = a[kOwnHalf][i][c];             \
    break;
      EIG_COL_CASE(0) EIG_COL_CASE(1) EIG_COL_CASE(2) EIG_COL_CASE(3)
      EIG_COL_CASE(4) EIG_COL_CASE(5) EIG_COL_CASE(6) EIG_COL_CASE(7)
#undef EIG_COL_CASE
    }
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      acc[i] = own1 ? fmaf(delta, col[i], acc[i]) : acc[i];
      const float vr = xr[i] + (R0 + i == j1 ? delta : 0.f);
      t = fmaf(vr, acc[i], t);
    }
    // reduce-scatter over the 8 column lanes: lane lc ends with row R0 + lc
    const bool h4 = lc & 4, h2 = lc & 2, h1 = lc & 1;
    float s4[4], s2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float keep = h4 ? acc[4 + i] : acc[i];
      const float send = h4 ? acc[i] : acc[4 + i];
      s4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float keep = h2 ? s4[2 + i] : s4[i];
      const float send = h2 ? s4[i] : s4[2 + i];
      s2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float s1 = (h1 ? s2[1] : s2[0]) + __shfl_xor_sync(0xffffffffu, h1 ? s2[0] : s2[1], 1);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    s.pp[b][R0 + lc] = s1;
    if (lane == 0) s.kp[b][warp] = 32 * warp + 31 > j ? t : 0.f;   // finished rows: v is zero there
    if (own1) {
      *reinterpret_cast<float4*>(&s.cb[b][R0]) = make_float4(col[0], col[1], col[2], col[3]);
      *reinterpret_cast<float4*>(&s.cb[b][R0 + 4]) = make_float4(col[4], col[5], col[6], col[7]);
    }
    if (warp == 0) {                                    // v_j for the next step and the back-transform
      const int q0 = 4 * lane;
      float4 v4;
      v4.x = xq[0] + (q0 == j1 ? delta : 0.f);
      v4.y = xq[1] + (q0 + 1 == j1 ? delta : 0.f);
      v4.z = xq[2] + (q0 + 2 == j1 ? delta : 0.f);
      v4.w = xq[3] + (q0 + 3 == j1 ? delta : 0.f);
      *reinterpret_cast<float4*>(&s.vs[b][q0]) = v4;
      if (lane >= hv_first_chunk(j))                    // the chunks before are exactly zero
        *reinterpret_cast<float4*>(&s.hv[hv_row_base(j) + 4 * (lane - hv_first_chunk(j))]) = v4;
      if (lane == 0) {
        s.beta[j] = beta;
        s.e[j] = alpha;
      }
    }
    beta_prev = beta;
    __syncthreads();
  };
#pragma unroll 1
  for (int j = 0; j < 63; ++j) step(std::true_type{}, j);
#pragma unroll 1
  for (int j = 63; j < kEigSteps; ++j) step(std::false_type{}, j);

  // the trailing 2 x 2 block after the last step's update
  {
    constexpr int bp = (kEigSteps & 1) ^ 1;            // the last step's buffers
    float Kp;
    {
      const float4 k4 = *reinterpret_cast<const float4*>(&s.kp[bp][0]);
      Kp = 0.5f * beta_prev * beta_prev * ((k4.x + k4.y) + (k4.z + k4.w));
    }
    auto w_at = [&](int q) { return fmaf(-Kp, s.vs[bp][q], beta_prev * s.pp[bp][q]); };
    if (tid == 0) {
      const float nu = s.vs[bp][n - 2], omega = w_at(n - 2);
      s.d[n - 2] = eig_xval(s.cb[bp][n - 2], nu, omega, omega, nu);
      s.e[n - 2] = eig_xval(s.cb[bp][n - 1], s.vs[bp][n - 1], w_at(n - 1), omega, nu);
      s.e[n - 1] = 0.f;
    }
    if (R0 == n - 8 && lc == 7) {
      const float v7 = s.vs[bp][n - 1], w7 = w_at(n - 1);
      s.d[n - 1] = fmaf(-v7, w7, fmaf(-w7, v7, a[1][7][7]));
    }
  }
  __syncthreads();
  if (warp == 0) {
    float tn = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = 4 * lane + k;
      const float em = i > 0 ? s.e[i - 1] : 0.f;
      tn = fmaxf(tn, fabsf(s.d[i]) + fabsf(s.e[i]) + fabsf(em));
      s.de2[i] = make_float2(s.d[i], em * em);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) tn = fmaxf(tn, __shfl_xor_sync(0xffffffffu, tn, o));
    if (lane == 0) s.tnorm = fmaxf(tn, FLT_MIN);
  }
  __syncthreads();

  // --- 2. top r eigenvalues by multisection (8 threads x 2 shifts each) -------
  const float tnorm = s.tnorm;
  {
    const int grp = tid >> 3, sub = tid & 7;          // eigenvalue grp, 16 shifts per round
    const unsigned gmask = 0xffu << (lane & 24);
    for (int jj = grp; jj < r; jj += kEigThreads / 8) {
      const int target = n - 1 - jj;                  // ascending index
      float lo = -tnorm * 1.01f, hi = tnorm * 1.01f;
      for (int round = 0; round < 6; ++round) {       // 17^6: width below 1e-7 tnorm
        const float step = (hi - lo) / 17.f;
        float xv[2];
        int cnt[2];
        xv[0] = lo + step * (float)(2 * sub + 1);
        xv[1] = lo + step * (float)(2 * sub + 2);
        sturm_count2(s.de2, xv, cnt);
        int first = 16;                               // first shift with count > target
        if (cnt[1] >= target + 1) first = 2 * sub + 1;
        if (cnt[0] >= target + 1) first = 2 * sub;
        first = (int)__reduce_min_sync(gmask, (unsigned)first);
        const float nlo = first == 0 ? lo : lo + step * (float)first;
        const float nhi = first == 16 ? hi : lo + step * (float)(first + 1);
        lo = nlo;
        hi = nhi;
        if (hi - lo <= 2.f * FLT_EPSILON * fmaxf(fabsf(lo), fabsf(hi))) break;
      }
      if (sub == 0) s.lam[jj] = 0.5f * (lo + hi);
    }
  }
  __syncthreads();

  // --- 3. inverse iteration: lane jj of warp 0, vector in registers ----------
  if (warp == 0 && lane < r) {
    const int jj = lane;
    const float lam = s.lam[jj];
    const float guard = FLT_EPSILON * tnorm;
    // LU with partial pivoting of T - lam I (rows: sub e[i-1], diag d[i]-lam, super e[i])
    float cd = s.d[0] - lam, cs = s.e[0];
#pragma unroll 2
    for (int i = 0; i < n - 1; ++i) {
      const float sub = s.e[i], nd = s.d[i + 1] - lam, ns = s.e[i + 1];
      const bool piv = fabsf(cd) < fabsf(sub);
      float ud = piv ? sub : cd;
      if (fabsf(ud) < guard) ud = ud < 0.f ? -guard : guard;
      const float rinv = __fdividef(1.f, ud);
      const float l = (piv ? cd : sub) * rinv;
      s.lu[0][i][jj] = rinv;
      s.lu[1][i][jj] = piv ? nd : cs;
      s.lu[2][i][jj] = piv ? ns : 0.f;
      s.lu[3][i][jj] = l;
      s.lu[4][i][jj] = piv ? 1.f : 0.f;
      const float ncd = piv ? fmaf(-l, nd, cs) : fmaf(-l, cs, nd);
      cs = piv ? -l * ns : ns;
      cd = ncd;
    }
    if (fabsf(cd) < guard) cd = cd < 0.f ? -guard : guard;
    s.lu[0][n - 1][jj] = __fdividef(1.f, cd);
    // the vector lives in shared memory ([row][vector]: conflict-free); each
    // recurrence keeps its running values in registers, so the dependency
    // chains never pass through memory
    for (int i = 0; i < n; ++i) s.zt[i][jj] = hash_unit(i, jj) + 0.75f;
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
      float cur = s.zt[0][jj];
#pragma unroll 4
      for (int i = 0; i < n - 1; ++i) {               // row interchanges and L
        const bool pv = s.lu[4][i][jj] != 0.f;
        const float ml = s.lu[3][i][jj];
        const float nxt = s.zt[i + 1][jj];
        s.zt[i][jj] = pv ? nxt : cur;
        cur = pv ? fmaf(-ml, nxt, cur) : fmaf(-ml, cur, nxt);
      }
      float z2 = cur * s.lu[0][n - 1][jj];            // back substitution with U
      float z1 = fmaf(-s.lu[1][n - 2][jj], z2, s.zt[n - 2][jj]) * s.lu[0][n - 2][jj];
      s.zt[n - 1][jj] = z2;
      s.zt[n - 2][jj] = z1;
      float mx = fmaxf(fabsf(z1), fabsf(z2));
#pragma unroll 4
      for (int i = n - 3; i >= 0; --i) {
        const float z0 = fmaf(-s.lu[2][i][jj], z2, fmaf(-s.lu[1][i][jj], z1, s.zt[i][jj])) * s.lu[0][i][jj];
        s.zt[i][jj] = z0;
        mx = fmaxf(mx, fabsf(z0));
        z2 = z1;
        z1 = z0;
      }
      const float inv = mx > 0.f ? 1.f / mx : 0.f;
      for (int i = 0; i < n; ++i) s.zt[i][jj] *= inv;
    }
  }
  __syncthreads();
  for (int el = tid; el < r * n; el += kEigThreads) s.z[el / n][el % n] = s.zt[el % n][el / n];
  // v_k . v_m inside each back-transform block (independent of the eigenvectors):
  // eight threads per block, lane q of the eight holding elements 4q + 32i + 0..3
  {
    const int g = tid >> 3, q = tid & 7;
    const unsigned gmask = 0xffu << (lane & 24);
    for (int blk = g; blk < kBtBlocks; blk += kEigThreads / 8) {
      const int j0 = blk * kBtBlock;
      float hvq[kBtBlock][16];
#pragma unroll
      for (int k = 0; k < kBtBlock; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
          if (j0 + k < kEigSteps) u = hv_chunk(s.hv, j0 + k, q + 8 * i);
          hvq[k][4 * i] = u.x; hvq[k][4 * i + 1] = u.y; hvq[k][4 * i + 2] = u.z; hvq[k][4 * i + 3] = u.w;
        }
#pragma unroll
      for (int k = 0; k < kBtBlock; ++k)
#pragma unroll
        for (int m = k + 1; m < kBtBlock; ++m) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) dot = fmaf(hvq[k][e], hvq[m][e], dot);
#pragma unroll
          for (int o = 4; o >= 1; o >>= 1) dot += __shfl_xor_sync(gmask, dot, o);
          if (q == 0) s.vtv[blk][k][m] = dot;           // zero past the last reflection
        }
    }
  }
  __syncthreads();

  // --- 4. orthonormalise the r vectors: Cholesky QR, two passes ---------------
  // M = Z Z^T = L L^T, Z <- L^{-1} Z; a non-positive pivot (a dependent
  // vector) drops that vector.
  for (int pass = 0; pass < 2; ++pass) {
    {                                                   // M = Z Z^T: eight threads per row ia, all ib <= ia
      const int g = tid >> 3, q = tid & 7;
      const unsigned gmask = 0xffu << (lane & 24);
      for (int ia = g; ia < r; ia += kEigThreads / 8) {
        float za[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 u = *reinterpret_cast<const float4*>(&s.z[ia][4 * q + 32 * i]);
          za[4 * i] = u.x; za[4 * i + 1] = u.y; za[4 * i + 2] = u.z; za[4 * i + 3] = u.w;
        }
#pragma unroll 4
        for (int ib = 0; ib <= ia; ++ib) {
          float dot = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 u = *reinterpret_cast<const float4*>(&s.z[ib][4 * q + 32 * i]);
            dot = fmaf(za[4 * i], u.x, fmaf(za[4 * i + 1], u.y, fmaf(za[4 * i + 2], u.z, fmaf(za[4 * i + 3], u.w, dot))));
          }
#pragma unroll
          for (int o = 4; o >= 1; o >>= 1) dot += __shfl_xor_sync(gmask, dot, o);
          if (q == 0) {
            s.gram[ia][ib] = dot;
            s.gram[ib][ia] = dot;
          }
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // right-looking Cholesky, lane = row: the row lives in registers and column k of L comes
      // from its rows' lanes by shuffles (the same multiply-adds in the same order as a
      // shared-memory update, without a shared-memory round trip per element)
      float g[kR];
#pragma unroll
      for (int m = 0; m < kR; ++m) g[m] = (lane < r && m < r) ? s.gram[lane][m] : 0.f;
#pragma unroll
      for (int k = 0; k < kR; ++k) {
        if (k < r) {
          const float dk = __shfl_sync(0xffffffffu, g[k], k);
          const float dinv = dk > 1e-20f ? rsqrtf(dk) : 0.f;
          if (lane >= k) g[k] *= dinv;                  // L[k][k] = sqrt(dk)
          if (lane == 0) s.lam[k] = dinv;               // reciprocal pivots
          const float lik = g[k];
#pragma unroll
          for (int m = k + 1; m < kR; ++m) {
            const float lmk = __shfl_sync(0xffffffffu, g[k], m);
            if (lane > k && m <= lane) g[m] = fmaf(-lik, lmk, g[m]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < kR; ++m)
        if (lane < r && m < r) s.gram[lane][m] = g[m];
    }
    __syncthreads();
    if (tid < n) {                                      // forward substitution, one column per thread, in registers
      float zc[kR];
#pragma unroll
      for (int ia = 0; ia < kR; ++ia) zc[ia] = ia < r ? s.z[ia][tid] : 0.f;
#pragma unroll
      for (int ia = 0; ia < kR; ++ia) {
        if (ia < r) {
          float acc = zc[ia];
#pragma unroll
          for (int ib = 0; ib < ia; ++ib) acc = fmaf(-s.gram[ia][ib], zc[ib], acc);
          zc[ia] = acc * s.lam[ia];
        }
      }
#pragma unroll
      for (int ia = 0; ia < kR; ++ia)
        if (ia < r) s.z[ia][tid] = zc[ia];
    }
    __syncthreads();
  }

  // --- 5. back-transform: y = H_0 H_1 ... H_{n-3} z, eight reflections a block --
  // Inside a block (reflections j0 .. j0+7, applied last first):
  //   s_k = v_k.y - sum_{m>k} beta_m s_m (v_k.v_m),  y -= sum_k beta_k s_k v_k.
  // Eight lanes per vector; lane q holds elements 4q + 32i + 0..3 (i < 4).
  {
    const int q = lane & 7;
    for (int vec = warp * 4 + (lane >> 3); vec < r; vec += kEigThreads / 8) {
      float y[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 t4 = *reinterpret_cast<const float4*>(&s.z[vec][4 * q + 32 * i]);
        y[4 * i] = t4.x; y[4 * i + 1] = t4.y; y[4 * i + 2] = t4.z; y[4 * i + 3] = t4.w;
      }
      const unsigned gmask = 0xffu << (lane & 24);
#pragma unroll 1
      for (int blk = kBtBlocks - 1; blk >= 0; --blk) {
        const int j0 = blk * kBtBlock;
        const int nb = min(kBtBlock, kEigSteps - j0);
        // the block's reflection vectors stay in registers for both the dots and the update
        float sdot[kBtBlock];
        float4 hvr[kBtBlock][4];
#pragma unroll
        for (int k = 0; k < kBtBlock; ++k) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 v = k < nb ? hv_chunk(s.hv, j0 + k, q + 8 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
            hvr[k][i] = v;
            if (k < nb)
              acc = fmaf(v.x, y[4 * i], fmaf(v.y, y[4 * i + 1], fmaf(v.z, y[4 * i + 2], fmaf(v.w, y[4 * i + 3], acc))));
          }
          sdot[k] = acc;
        }
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1)
#pragma unroll
          for (int k = 0; k < kBtBlock; ++k) sdot[k] += __shfl_xor_sync(gmask, sdot[k], o);
        float coef[kBtBlock];
#pragma unroll
        for (int k = kBtBlock - 1; k >= 0; --k) {
          float sk = sdot[k];
#pragma unroll
          for (int m = k + 1; m < kBtBlock; ++m) sk = fmaf(-coef[m], s.vtv[blk][k][m], sk);
          coef[k] = k < nb ? s.beta[j0 + k] * sk : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kBtBlock; ++k) {
          if (k < nb) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 v = hvr[k][i];
              y[4 * i] = fmaf(-coef[k], v.x, y[4 * i]);
              y[4 * i + 1] = fmaf(-coef[k], v.y, y[4 * i + 1]);
              y[4 * i + 2] = fmaf(-coef[k], v.z, y[4 * i + 2]);
              y[4 * i + 3] = fmaf(-coef[k], v.w, y[4 * i + 3]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(evec_out + (size_t)vec * n + 4 * q + 32 * i) =
            make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
    }
    for (int el = r * n + tid; el < kCurdkvMaxRank * n; el += kEigThreads) evec_out[el] = 0.f;
  }
}

// ---------------------------------------------------------------------------
// Leverage and cumulative score on the tensor cores, persistent and pipelined.
// The (b, h, 128-row tile) items of the call (kept rows from row 0, then
// incoming rows from row k, as in the Gram kernel) are laid end to end and
// every CTA takes an equal contiguous share. Per item, P = V_tile E^T (E = the
// unit's top-r eigenvectors split into bf16 hi + lo, zero rows past r) comes
// from one M = 128, N = 32 MMA chain with the value tile in its natural
// K-major layout; then l_i = a_i^2 |P_i|^2 / E, added to kept rows' scores
// and seeding incoming rows'.
// Roles (192 threads): warp 0 issues the TMA loads (a ring of value tiles),
// warp 1 the MMAs (two TMEM accumulators of 32 columns), warps 2-5 build each
// unit's eigenvector tiles and turn accumulators into leverage, one TMEM lane
// (one token) per thread.
// ---------------------------------------------------------------------------
constexpr int kEvecTileBytes = kCurdkvMaxRank * kHeadDim * 2;
constexpr int kLevStages = 4;
constexpr int kLevThreads = 192;
constexpr int kLevSmem = kLevStages * kTileBytes + 2 * 2 * kEvecTileBytes + 1024;
static_assert(kCurdkvMaxRank == 32, "the leverage MMA uses N = 32");

struct LevBars {
  uint64_t v_full[kLevStages], v_empty[kLevStages];
  uint64_t e_full[2], e_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int fail;
};

__global__ void __launch_bounds__(kLevThreads, 1) curdkv_leverage_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ LevBars b;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t vring = tc::smem_u32(smem);
  const uint32_t ering = vring + kLevStages * kTileBytes;   // unit parity u: hi at 2u, lo at 2u+1
  const int Ck = (p.k + kTile - 1) / kTile, Cm = (p.m + kTile - 1) / kTile;
  const int T = Ck + Cm;
  const long long total = (long long)T * p.units;
  const long long g0 = total * blockIdx.x / gridDim.x, g1 = total * (blockIdx.x + 1) / gridDim.x;
  if (tid == 0) {
    for (int i = 0; i < kLevStages; ++i) {
      tc::mbar_init(&b.v_full[i], 1);
      tc::mbar_init(&b.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&b.e_full[i], 4);                  // the four epilogue warps
      tc::mbar_init(&b.e_empty[i], 1);
      tc::mbar_init(&b.acc_full[i], 1);
      tc::mbar_init(&b.acc_empty[i], 4);
    }
    b.fail = 0;
  }
  if (warp == 2) tc::tmem_alloc(&b.tmem_base, 2 * kCurdkvMaxRank);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0) {
    if (lane == 0 && g1 > g0) {                         // TMA producer
      tc::tma_prefetch_desc(&p.tm_vin);
      if (Ck > 0) tc::tma_prefetch_desc(&p.tm_vst);
      int issued[kLevStages] = {0, 0, 0, 0};
      for (long long g = g0; g < g1; ++g) {
        const int j = (int)(g - g0), st = j % kLevStages;
        const int bh = (int)(g / T), i = (int)(g - (long long)bh * T);
        if (!wait_phase(&b.v_empty[st], (uint32_t)(((j / kLevStages) & 1) ^ 1), &b.fail, p.err)) break;
        tc::mbar_arrive_expect_tx(&b.v_full[st], (uint32_t)kTileBytes);
        const bool kept = i < Ck;
        const void* map = kept ? (const void*)&p.tm_vst : (const void*)&p.tm_vin;
        const int y = kept ? kTile * i : kTile * (i - Ck);
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(vring + st * kTileBytes + hf * (kTileBytes / 2), map, 64 * hf, y, bh, &b.v_full[st]);
        ++issued[st];
      }
      for (int i = 0; i < kLevStages; ++i)
        if (issued[i] > 0) drain_phase(&b.v_full[i], (uint32_t)((issued[i] - 1) & 1), p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && g1 > g0) {                         // MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTile, kCurdkvMaxRank);
      int units = 0, uses[2] = {0, 0};
      for (long long g = g0; g < g1; ++g) {
        const int j = (int)(g - g0), st = j % kLevStages, ab = j & 1;
        const int bh = (int)(g / T), i = (int)(g - (long long)bh * T);
        if (g == g0 || i == 0) {                        // a new unit: its eigenvector tiles
          if (!wait_phase(&b.e_full[units & 1], (uint32_t)((units >> 1) & 1), &b.fail, p.err)) break;
          ++units;
        }
        const int ub = (units - 1) & 1;
        if (!wait_phase(&b.v_full[st], (uint32_t)((j / kLevStages) & 1), &b.fail, p.err)) break;
        if (!wait_phase(&b.acc_empty[ab], (uint32_t)((uses[ab] & 1) ^ 1), &b.fail, p.err)) break;
        tc::fence_after_sync();
        const uint32_t va = vring + st * kTileBytes, ehi = ering + 2 * ub * kEvecTileBytes, elo = ehi + kEvecTileBytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a_off = (uint32_t)((ks >> 2) * kTile * 128 + (ks & 3) * 32);
          const uint32_t b_off = (uint32_t)((ks >> 2) * kCurdkvMaxRank * 128 + (ks & 3) * 32);
          const uint64_t ad = tc::sw128_desc(va + a_off);
          const uint32_t acc = tmem + (uint32_t)(ab * kCurdkvMaxRank);
          tc::mma_bf16(acc, ad, tc::sw128_desc(ehi + b_off), idesc, ks > 0 ? 1u : 0u);
          tc::mma_bf16(acc, ad, tc::sw128_desc(elo + b_off), idesc, 1u);
        }
        tc::mma_commit(&b.v_empty[st]);
        tc::mma_commit(&b.acc_full[ab]);
        ++uses[ab];
        if (g + 1 == g1 || i == T - 1) tc::mma_commit(&b.e_empty[ub]);
      }
      for (int a = 0; a < 2; ++a)                       // the last MMAs finish before TMEM is released
        if (uses[a] > 0) drain_phase(&b.acc_full[a], (uint32_t)((uses[a] - 1) & 1), p.err);
    }
    __syncwarp();
  } else {                                              // epilogue: one token per thread
    const int et = tid - 64;                            // 0 .. 127
    const int quarter = warp & 3, row_in_tile = 32 * quarter + lane;
    int units = 0, uses[2] = {0, 0};
    auto attn_of = [&](long long g) -> float {
      if (g >= g1) return 0.f;
      const int bh = (int)(g / T), i = (int)(g - (long long)bh * T);
      const int row = i < Ck ? kTile * i + row_in_tile : p.k + kTile * (i - Ck) + row_in_tile;
      const int lim = i < Ck ? p.k : p.k + p.m;
      return row < lim ? p.attn[(size_t)bh * p.rows + row] : 0.f;
    };
    float a_next = attn_of(g0);
    for (long long g = g0; g < g1; ++g) {
      const int j = (int)(g - g0), ab = j & 1;
      const int bh = (int)(g / T), i = (int)(g - (long long)bh * T);
      const float a_cur = a_next;
      a_next = attn_of(g + 1);
      if (g == g0 || i == 0) {                          // build this unit's eigenvector tiles
        const int ub = units & 1;
        bool ok = wait_phase(&b.e_empty[ub], (uint32_t)(((units >> 1) & 1) ^ 1), &b.fail, p.err);
        if (!__all_sync(0xffffffffu, ok)) break;
        const float* ev = p.evec + (size_t)bh * kCurdkvMaxRank * kHeadDim;
        unsigned char* eh = smem + kLevStages * kTileBytes + 2 * ub * kEvecTileBytes;
        for (int item = et; item < kCurdkvMaxRank * 16; item += 128) {
          const int jr = item >> 4, ch = item & 15;
          const float4 x0 = *reinterpret_cast<const float4*>(ev + jr * kHeadDim + 8 * ch);
          const float4 x1 = *reinterpret_cast<const float4*>(ev + jr * kHeadDim + 8 * ch + 4);
          const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            hw[q] = pack_bf16x2(x[2 * q], x[2 * q + 1]);
            lw[q] = pack_bf16x2(x[2 * q] - __uint_as_float(hw[q] << 16),
                                x[2 * q + 1] - __uint_as_float(hw[q] & 0xffff0000u));
          }
          const uint32_t off = tc::sw128_offset(jr, ch, kCurdkvMaxRank);
          *reinterpret_cast<uint4*>(eh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(eh + kEvecTileBytes + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&b.e_full[ub]);
        ++units;
      }
      bool ok = wait_phase(&b.acc_full[ab], (uint32_t)(uses[ab] & 1), &b.fail, p.err);
      if (!__all_sync(0xffffffffu, ok)) break;
      ++uses[ab];
      tc::fence_after_sync();
      float proj[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(ab * kCurdkvMaxRank), proj);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&b.acc_empty[ab]);
      float e4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) e4[jj & 3] = fmaf(proj[jj], proj[jj], e4[jj & 3]);
      const bool kept = i < Ck;
      const int row = kept ? kTile * i + row_in_tile : p.k + kTile * (i - Ck) + row_in_tile;
      const int lim = kept ? p.k : p.k + p.m;
      if (row < lim) {
        const float l = a_cur * a_cur * ((e4[0] + e4[1]) + (e4[2] + e4[3])) * p.inv_e[bh];
        p.lev[(size_t)bh * p.rows + row] = l;
        if (kept) p.score_st[(size_t)bh * p.cap + row] += l;
        else p.new_score[(size_t)bh * p.new_stride + (row - p.k)] = l;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) tc::tmem_dealloc(tmem, 2 * kCurdkvMaxRank);
}

// Append the block (cache stays within budget): grid = (ceil(m / 64), B*H), block = 256.
__global__ void __launch_bounds__(256) curdkv_append_kernel(const __grid_constant__ CurdkvParams p) {
  pdl_wait();
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
  st.gram = reinterpret_cast<float*>(take(bh * kHeadDim * kHeadDim * 4));
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
      (e = cudaFuncSetAttribute(curdkv_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGramSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_leverage_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLevSmem)) !=
          cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_attn_small_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmallAttnMaxLogits * (int)sizeof(float))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_attn_small_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmallAttnMaxLogits * (int)sizeof(float))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_attn_small_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmallAttnMaxLogits * (int)sizeof(float))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_attn_small_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmallAttnMaxLogits * (int)sizeof(float))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_eig_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(EigSmem<16>))) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_eig_kernel<16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(curdkv_eig_kernel<kCurdkvMaxRank>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(EigSmem<kCurdkvMaxRank>))) != cudaSuccess)
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
  p.units = bh;
  p.rank = std::min(std::min(c.rank_cap, n), kHeadDim);
  p.scale2 = kLog2e / sqrtf((float)kHeadDim);
  p.self_excluded = c.method == EVICT_H2O ? 1 : 0;
  p.lse = st.lse;
  p.lse_part = st.lse_part;
  p.lse_stride = st.lse_stride;
  p.attn = st.attn;
  p.lev = st.lev;
  p.rows = st.rows;
  p.gram = st.gram;
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
  // attention passes: TMA maps of the incoming and kept keys, tile shares
  if (!encode_rows(&p.tm_kin, k, m, m, bh) || (p.k > 0 && !encode_rows(&p.tm_kst, h->kst, p.k, h->cap, bh)))
    return fail(EVICT_EINVAL, "cannot describe the key buffers for TMA (k must be 16-byte aligned)");
  if (!encode_rows(&p.tm_vin, v, m, m, bh) || (p.k > 0 && !encode_rows(&p.tm_vst, h->vst, p.k, h->cap, bh)))
    return fail(EVICT_EINVAL, "cannot describe the value buffers for TMA (v must be 16-byte aligned)");
  {
    // Gram cluster: enough CTAs per (b, h) to cover the SMs, at most one per tile and 8
    const int tiles = (p.k + kTile - 1) / kTile + (m + kTile - 1) / kTile;
    p.gram_cluster = std::max(1, std::min({kGramMaxCluster, st.sm_count / std::max(bh, 1), tiles}));
  }
  p.sched1 = make_sched(p.k, m, bh, st.sm_count, true);
  p.sched2 = make_sched(p.k, m, bh, st.sm_count, false);
  p.colpart = p.sched2.Q > 1 ? st.colpart : st.attn;
  if (small_attn_fits(m, n)) {
    // short blocks (decode steps, the per-token mode): one fused pass per unit
    e = timed_launch(h, kKidCurdkvAttnSmall, [&] {
      const size_t smem = (size_t)m * n * sizeof(float);
      if (m == 1)
        return launch_pdl(curdkv_attn_small_kernel<1>, dim3(bh), dim3(kSmallAttnThreads), smem, sm, nullptr, p);
      else if (m == 2)
        return launch_pdl(curdkv_attn_small_kernel<2>, dim3(bh), dim3(kSmallAttnThreads), smem, sm, nullptr, p);
      else if (m <= 4)
        return launch_pdl(curdkv_attn_small_kernel<4>, dim3(bh), dim3(kSmallAttnThreads), smem, sm, nullptr, p);
      else
        return launch_pdl(curdkv_attn_small_kernel<8>, dim3(bh), dim3(kSmallAttnThreads), smem, sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV short-block attention launch");
  } else {
  e = timed_launch(h, kKidCurdkvLse, [&] {
    return launch_pdl(curdkv_lse_kernel, dim3(p.sched1.ctas), dim3(kAttnCtaThreads), attn_smem_bytes(kLseStages), sm,
                      nullptr, p);
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 1 launch");
  e = timed_launch(h, kKidCurdkvLseMerge, [&] {
    return launch_pdl(curdkv_lse_merge_kernel, dim3((m + 255) / 256, bh), dim3(256), 0, sm, nullptr, p);
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention merge launch");
  e = timed_launch(h, kKidCurdkvColsum, [&] {
    return launch_pdl(curdkv_colsum_kernel, dim3(p.sched2.ctas), dim3(kAttnCtaThreads), attn_smem_bytes(kColStages),
                      sm, nullptr, p);
  });
  if (e != cudaSuccess) return cuda_fail(e, "CurDKV attention pass 2 launch");
  if (p.sched2.Q > 1) {
    e = timed_launch(h, kKidCurdkvColsumMerge, [&] {
      return launch_pdl(curdkv_colsum_merge_kernel, dim3((n + 255) / 256, bh), dim3(256), 0, sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV column-sum merge launch");
  }
  if (p.self_excluded) {
    e = timed_launch(h, kKidH2oMass, [&] {
      return launch_pdl(h2o_mass_kernel, dim3((n + 255) / 256, bh), dim3(256), 0, sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "H2O mass launch");
  }
  }
  if (!p.self_excluded) {
    e = timed_launch(h, kKidCurdkvGram, [&] {
      cudaLaunchAttribute cluster;
      cluster.id = cudaLaunchAttributeClusterDimension;
      cluster.val.clusterDim.x = (unsigned)p.gram_cluster;
      cluster.val.clusterDim.y = 1;
      cluster.val.clusterDim.z = 1;
      return launch_pdl(curdkv_gram_kernel, dim3(p.gram_cluster * bh), dim3(kGramThreads), kGramSmem, sm, &cluster, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV Gram launch");
    e = timed_launch(h, kKidCurdkvEig, [&] {
      if (p.rank <= 16)
        return launch_pdl(curdkv_eig_kernel<16>, dim3(bh), dim3(kEigThreads), sizeof(EigSmem<16>), sm, nullptr, p);
      return launch_pdl(curdkv_eig_kernel<kCurdkvMaxRank>, dim3(bh), dim3(kEigThreads), sizeof(EigSmem<kCurdkvMaxRank>),
                        sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV eigensolver launch");
    e = timed_launch(h, kKidCurdkvLeverage, [&] {
      const long long items = (long long)bh * ((p.k + kTile - 1) / kTile + (m + kTile - 1) / kTile);
      return launch_pdl(curdkv_leverage_kernel, dim3((int)std::min<long long>(st.sm_count, items)), dim3(kLevThreads),
                        kLevSmem, sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV leverage launch");
  }
  if (n <= c.budget) {
    e = timed_launch(h, kKidAppend, [&] {
      return launch_pdl(curdkv_append_kernel, dim3((m + 63) / 64, bh), dim3(256), 0, sm, nullptr, p);
    });
    if (e != cudaSuccess) return cuda_fail(e, "CurDKV append launch");
    h->n_kept = n;
    h->last_evicted = false;
  } else if (n == c.budget + 1 && m <= evict1_max_block()) {
    // exactly one row leaves (decode steps): the fused single eviction on the pipeline's scores;
    // the per-token mode takes the argmin rule on ties, the block form keeps the lower index
    GroupParams P = make_group_params(h, m, 1);
    P.L[0] = make_layer_ptrs(h, k, v, pos);
    P.s.tie_low = c.per_token ? 1 : 0;
    e = timed_launch(h, kKidEvict1, [&] { return launch_evict1(P, 2, sm); });
    if (e != cudaSuccess) return cuda_fail(e, "single-eviction kernel launch");
    h->n_kept = c.budget;
    h->last_evicted = true;
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
