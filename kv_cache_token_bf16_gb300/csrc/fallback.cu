// Q-Filters key-SVD fallback: the one-time freeze of a per-(b, h) filter
// ("Q-Filters — Query-Agnostic Projection Eviction", §How it works step 2,
// §Key-SVD fallback, §Path dependence).
//
// Without calibrated filters the cache keeps every row until calib_tokens keys
// have been seen. The update whose block reaches that count runs this kernel
// once, before its usual score / select / compaction launches. A cluster of
// CTAs serves one (layer, b, h) unit, over the n = k + m keys present (the k
// kept rows, then the m incoming rows); each CTA takes a contiguous slice of
// the rows:
//   1. one pass over the rows, shifted by the unit's first key x_0: the slice
//      Gram G = sum (x - x_0)(x - x_0)^T in fp32 (x - x_0 rounded once per
//      element, 8 x 8 register blocks per thread) and the column sums
//      t = sum (x - x_0);
//   2. G and t added over the cluster in rank order (distributed shared
//      memory) into rank 0, which centres: C = G - n d d^T, d = t / n (fp64),
//      the Gram of the mean-centred keys;
//   3. rank 0: top eigenvector v of C, i.e. the top right singular vector of
//      the centred key matrix. C / tr C is squared eight times (each square
//      renormalised by its trace), so that power iteration (power.cuh) on
//      C^256, from its column of largest diagonal, converges at the rate
//      (lambda2 / lambda1)^256; a bounded power iteration on C itself then
//      polishes the result;
//   4. sign: the component of largest magnitude (first of equals) is made
//      positive. C = 0 (all keys equal) has no direction: v = e_0;
//   5. v becomes the unit's frozen filter, and the CTAs re-score the unit's k
//      kept rows with it (a slice each) in the canonical order of score.cuh;
//      the incoming rows are scored by the launches that follow.
// A non-finite entry of C (a non-finite key, or keys too large for an fp32
// Gram) raises kDevNonFinite and freezes the zero filter. When the top two
// eigenvalues are closer than fp32 rounding can separate, the bounded
// iterations return a unit vector of their span.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "params.h"
#include "power.cuh"
#include "score.cuh"
#include "tcgen05.cuh"

namespace evict {
namespace {

constexpr int kFzThreads = kPowerThreads;   // 256
constexpr int kFzTileRows = 32;
constexpr int kFzRowsPerHalfWarp = 4;       // kept rows re-scored per half-warp and round
constexpr int kFzPadded = kHeadDim * kPowerStride;   // floats of a padded 128 x 129 matrix
constexpr int kFzDense = kHeadDim * kHeadDim;        // floats of a dense 128 x 128 matrix
constexpr int kFzSquarings = 8;
constexpr int kFzSquaredIters = 128;        // power iterations on C^256
constexpr int kFzPolishIters = 64;          // power iterations on C
constexpr int kFzMaxCluster = 8;
constexpr int kFzMinSliceRows = 256;
// C (padded), S1 (padded capacity; holds the key tile during the Gram), S2 (dense)
constexpr size_t kFzSmem = (size_t)(2 * kFzPadded + kFzDense) * sizeof(float);
static_assert(kFzTileRows * kHeadDim <= kFzPadded, "key tile must fit in S1");

template <bool kBf16>
struct KeyRows {
  static constexpr int kRowBytes = kHeadDim * (kBf16 ? 2 : 4);
  const char* kst;    // this unit's kept rows
  const char* kin;    // this unit's incoming rows
  int k;
  __device__ __forceinline__ const char* row(int r) const {
    return r < k ? kst + (size_t)r * kRowBytes : kin + (size_t)(r - k) * kRowBytes;
  }
  __device__ __forceinline__ float elem(int r, int d) const {
    const char* p = row(r);
    if (kBf16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(p)[d] << 16);
    return reinterpret_cast<const float*>(p)[d];
  }
};

// acc[x][y] += sum over r < rows of src[r][i0 + x] * src[r][j0 + y] (dense rows of 128 floats)
__device__ __forceinline__ void rank_update(const float* src, int rows, int i0, int j0, float (&acc)[8][8]) {
#pragma unroll 4
  for (int r = 0; r < rows; ++r) {
    const float4* row = reinterpret_cast<const float4*>(src + r * kHeadDim);
    const float4 a0 = row[i0 / 4], a1 = row[i0 / 4 + 1], b0 = row[j0 / 4], b1 = row[j0 / 4 + 1];
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int x = 0; x < 8; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[8][8]) {
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
}

// Sum of the 128 diagonal entries of a matrix with row stride `ld` (all threads return it).
__device__ __forceinline__ float trace128(const float* m, int ld, float* red) {
  const int tid = threadIdx.x;
  float t = tid < kHeadDim ? m[tid * ld + tid] : 0.f;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if ((tid & 31) == 0 && tid < kHeadDim) red[tid >> 5] = t;
  __syncthreads();
  const float tr = (red[0] + red[1]) + (red[2] + red[3]);
  __syncthreads();
  return tr;
}

// grid = units * cluster (cluster dims (cluster, 1, 1)), block = 256, dynamic shared memory kFzSmem.
template <bool kBf16>
__global__ void __launch_bounds__(kFzThreads) freeze_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  extern __shared__ __align__(16) float fz_smem[];
  float* C = fz_smem;                            // padded: the unit's centred Gram (rank 0: the sum)
  float* S1 = fz_smem + kFzPadded;               // key tile, then the squarings (dense, the last padded)
  float* S2 = fz_smem + 2 * kFzPadded;           // squarings (dense)
  __shared__ double s_part[kHeadDim], s_d[kHeadDim];
  __shared__ float s_ref[kHeadDim], v[kHeadDim], w[kHeadDim], red[4];
  __shared__ float s_norm, s_delta;
  __shared__ int s_bad;
  const Shape& s = P.s;
  const int tid = threadIdx.x;
  const int cl = (int)(gridDim.x / (unsigned)(s.n_layers * s.batch * s.heads));
  const int rank = (int)tc::cluster_rank();
  const int u = blockIdx.x / cl;
  const int bhn = s.batch * s.heads;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  constexpr int kRowBytes = KeyRows<kBf16>::kRowBytes;
  KeyRows<kBf16> K{static_cast<const char*>(L.kst) + (size_t)bh * s.cap * kRowBytes,
                   static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes, s.k};
  const int n = s.k + s.m;
  const int per = (n + cl - 1) / cl;
  const int r_lo = min(n, rank * per), r_hi = min(n, r_lo + per);

  // 1-2. shifted slice Gram G = sum (x - x_0)(x - x_0)^T and column sums t = sum (x - x_0) over
  // this CTA's rows, shifted by the unit's first key x_0 (Chan, Golub & LeVeque, "Algorithms for
  // computing the sample variance", the shifted algorithm): C = G - n d d^T with d = t / n is
  // the centred Gram in one pass. Keys arrive as 16-byte vectors, the next tile's loads in
  // flight while the current one is multiplied.
  constexpr int kVpr = kRowBytes / 16;                        // 16-byte vectors per key row
  constexpr int kCols = 16 / (kBf16 ? 2 : 4);                 // columns per vector
  constexpr int kPer = kFzTileRows * kVpr / kFzThreads;       // vectors per thread and tile
  static_assert(kFzThreads % kVpr == 0 && kPer >= 1, "a thread keeps one vector column");
  if (tid < kHeadDim) s_ref[tid] = K.elem(0, tid);
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int cvec = tid % kVpr;                                // this thread's vector column
  float ref[kCols], csum[kCols];
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    ref[j] = s_ref[cvec * kCols + j];
    csum[j] = 0.f;
  }
  const int i0 = (tid >> 4) * 8, j0 = (tid & 15) * 8;
  float acc[8][8];
  zero_acc(acc);
  uint4 pre[kPer];
  auto fetch = [&](int r0) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int r = r0 + (tid + q * kFzThreads) / kVpr;
      pre[q] = r < r_hi ? ld_stream(K.row(r) + 16 * cvec) : make_uint4(0, 0, 0, 0);
    }
  };
  fetch(r_lo);
  for (int r0 = r_lo; r0 < r_hi; r0 += kFzTileRows) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int rr = (tid + q * kFzThreads) / kVpr;
      const bool live = r0 + rr < r_hi;
      float x[8];
      if (kBf16) {
        bf16x8_to_f32(pre[q], x);
      } else {
        x[0] = __uint_as_float(pre[q].x); x[1] = __uint_as_float(pre[q].y);
        x[2] = __uint_as_float(pre[q].z); x[3] = __uint_as_float(pre[q].w);
      }
      float* dst = S1 + rr * kHeadDim + cvec * kCols;
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const float y = live ? x[j] - ref[j] : 0.f;
        dst[j] = y;
        csum[j] += y;
      }
    }
    __syncthreads();
    if (r0 + kFzTileRows < r_hi) fetch(r0 + kFzTileRows);
    rank_update(S1, kFzTileRows, i0, j0, acc);
    __syncthreads();
  }
  // column sums: the threads of one vector column in order, then fp64
  {
    float* part = S2;                                         // [kFzThreads / kVpr][128] scratch
#pragma unroll
    for (int j = 0; j < kCols; ++j) part[(tid / kVpr) * kHeadDim + cvec * kCols + j] = csum[j];
    __syncthreads();
    if (tid < kHeadDim) {
      double t = 0.0;
      for (int g = 0; g < kFzThreads / kVpr; ++g) t += part[g * kHeadDim + tid];
      s_part[tid] = t;
    }
  }
#pragma unroll
  for (int x = 0; x < 8; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) C[(i0 + x) * kPowerStride + j0 + y] = acc[x][y];
  tc::cluster_sync();
  if (cl > 1) {
    // rows i with i % cl == rank are summed by this CTA (ranks in order) and stored into rank 0
    const uint32_t cbase = tc::smem_u32(C);
    for (int e = tid; e < kFzDense; e += kFzThreads) {
      const int i = e / kHeadDim, j = e % kHeadDim;
      if (i % cl != rank) continue;
      const uint32_t off = (uint32_t)((i * kPowerStride + j) * sizeof(float));
      float sum = 0.f;
      for (int q = 0; q < cl; ++q) sum += tc::ld_cluster_f32(tc::map_to_rank(cbase + off, (uint32_t)q));
      tc::st_cluster_f32(tc::map_to_rank(cbase + off, 0u), sum);
    }
    if (rank == 0 && tid < kHeadDim) {
      const uint32_t a = tc::smem_u32(&s_part[tid]);
      double t = 0.0;
      for (int q = 0; q < cl; ++q) t += tc::ld_cluster_f64(tc::map_to_rank(a, (uint32_t)q));
      s_d[tid] = t / (double)n;
    }
    tc::cluster_sync();
  } else if (tid < kHeadDim) {
    s_d[tid] = s_part[tid] / (double)n;
  }

  // 3. rank 0: top eigenvector
  if (rank == 0) {
    __syncthreads();                                      // s_d complete (single-CTA case)
    bool bad = false;
    for (int e = tid; e < kFzDense; e += kFzThreads) {
      const int i = e / kHeadDim, j = e % kHeadDim;
      float* cij = &C[i * kPowerStride + j];
      *cij = (float)((double)*cij - (double)n * s_d[i] * s_d[j]);   // centre: C = G - n d d^T
      bad |= !isfinite(*cij);
    }
    if (bad) s_bad = 1;
    __syncthreads();
    const bool bad_all = s_bad != 0;
    const float tr = bad_all ? 0.f : trace128(C, kPowerStride, red);
    const bool flat = !bad_all && !(tr > 0.f);           // C = 0: every key equal
    if (!bad_all && !flat) {
      // S2 = C / tr C (dense), then square: S <- S^2 / tr(S^2); the last square lands padded in S1
      const float inv = 1.f / tr;
      for (int e = tid; e < kFzDense; e += kFzThreads)
        S2[e] = C[(e / kHeadDim) * kPowerStride + e % kHeadDim] * inv;
      __syncthreads();
      float* src = S2;
      for (int q = 0; q < kFzSquarings; ++q) {
        const bool last = q == kFzSquarings - 1;
        float* dst = src == S2 ? S1 : S2;
        const int ld = last ? kPowerStride : kHeadDim;
        if (last && dst != S1) dst = S1;                  // S1 has the padded capacity
        zero_acc(acc);
        rank_update(src, kHeadDim, i0, j0, acc);          // S symmetric: (S^2)_ij = sum_r S_ri S_rj
        __syncthreads();                                  // every read of src done (dst may alias it)
#pragma unroll
        for (int x = 0; x < 8; ++x)
#pragma unroll
          for (int y = 0; y < 8; ++y) dst[(i0 + x) * ld + j0 + y] = acc[x][y];
        __syncthreads();
        const float t2 = trace128(dst, ld, red);
        const float inv2 = t2 > 0.f ? 1.f / t2 : 0.f;
        for (int e = tid; e < kFzDense; e += kFzThreads) dst[(e / kHeadDim) * ld + e % kHeadDim] *= inv2;
        __syncthreads();
        src = dst;
      }
      // start: the column of S1 = C^256 / tr with the largest diagonal entry
      if (tid == 0) {
        int best = 0;
        for (int j = 1; j < kHeadDim; ++j)
          if (S1[j * kPowerStride + j] > S1[best * kPowerStride + best]) best = j;
        double nrm = 0.0;
        for (int i = 0; i < kHeadDim; ++i) nrm += (double)S1[i * kPowerStride + best] * S1[i * kPowerStride + best];
        s_norm = (float)sqrt(nrm);
        s_delta = (float)best;
      }
      __syncthreads();
      const int best = (int)s_delta;
      const float nrm = s_norm;
      __syncthreads();
      if (tid < kHeadDim) v[tid] = nrm > 0.f ? S1[tid * kPowerStride + best] / nrm : (tid == best ? 1.f : 0.f);
      __syncthreads();
      power_iterate(S1, v, w, &s_norm, &s_delta, kFzSquaredIters);
      power_iterate(C, v, w, &s_norm, &s_delta, kFzPolishIters);
    } else if (tid < kHeadDim) {
      v[tid] = (!bad_all && tid == 0) ? 1.f : 0.f;
    }
    __syncthreads();
    // 4. sign: largest-magnitude component positive
    if (tid == 0) {
      int j = 0;
      for (int i = 1; i < kHeadDim; ++i)
        if (fabsf(v[i]) > fabsf(v[j])) j = i;
      s_norm = v[j] < 0.f ? -1.f : 1.f;
      if (bad_all) raise_device_error(P.err, kDevNonFinite);
    }
    __syncthreads();
    if (tid < kHeadDim) {
      const float fv = s_norm * v[tid];
      v[tid] = fv;
      L.filters[(size_t)bh * kHeadDim + tid] = fv;
    }
  }
  tc::cluster_sync();                                     // rank 0's v is final

  // 5. re-score this CTA's slice of the kept rows against the frozen filter
  const int c = tid & 15, hw = tid >> 4;
  float f[8];
  {
    const uint32_t vbase = tc::map_to_rank(tc::smem_u32(v), 0u);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = tc::ld_cluster_f32(vbase + (uint32_t)((8 * c + j) * sizeof(float)));
  }
  tc::cluster_sync();                                     // nobody reads rank 0 after this
  const int kper = (s.k + cl - 1) / cl;
  const int k_lo = min(s.k, rank * kper), k_hi = min(s.k, k_lo + kper);
  float* out = L.score_st + (size_t)bh * s.cap;
  constexpr int kRowsPerRound = (kFzThreads / 16) * kFzRowsPerHalfWarp;
  for (int base = k_lo; base < k_hi; base += kRowsPerRound) {
    RowLoad<kBf16> ld[kFzRowsPerHalfWarp];
#pragma unroll
    for (int j = 0; j < kFzRowsPerHalfWarp; ++j) {
      const int r = base + hw + 16 * j;
      if (r < k_hi) ld[j].load(K.row(r), c); else ld[j].zero();
    }
#pragma unroll
    for (int j = 0; j < kFzRowsPerHalfWarp; ++j) {
      float x[8];
      ld[j].widen(x);
      const float sigma = canonical_score<kQFilters>(x, f, s.sign);
      const int r = base + hw + 16 * j;
      if (c == 0 && r < k_hi) out[r] = sigma;
    }
  }
}

}  // namespace

cudaError_t prepare_freeze() {
  cudaError_t e = cudaFuncSetAttribute(freeze_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFzSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(freeze_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFzSmem);
}

cudaError_t launch_freeze(const GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const int units = P.s.n_layers * P.s.batch * P.s.heads;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int n = P.s.k + P.s.m;
  int cl = std::max(1, std::min({kFzMaxCluster, sms / units, n / kFzMinSliceRows}));
  cudaLaunchAttribute cluster;
  cluster.id = cudaLaunchAttributeClusterDimension;
  cluster.val.clusterDim.x = (unsigned)cl;
  cluster.val.clusterDim.y = 1;
  cluster.val.clusterDim.z = 1;
  const dim3 grid((unsigned)(units * cl)), block(kFzThreads);
  if (dtype_bytes == 2) return launch_pdl(freeze_kernel<true>, grid, block, kFzSmem, st, &cluster, P);
  return launch_pdl(freeze_kernel<false>, grid, block, kFzSmem, st, &cluster, P);
}

}  // namespace evict
