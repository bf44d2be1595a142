// Q-Filters key-SVD fallback: the one-time freeze of a per-(b, h) filter
// ("Q-Filters — Query-Agnostic Projection Eviction", §How it works step 2,
// §Key-SVD fallback, §Path dependence).
//
// Without calibrated filters the cache keeps every row until calib_tokens keys
// have been seen. The update whose block reaches that count runs this kernel
// once, before its usual score / select / compaction launches. One CTA per
// (layer, b, h) unit, over the n = k + m keys present (the k kept rows, then
// the m incoming rows):
//   1. column means mu of the keys, summed in fp64;
//   2. Gram C = sum (x - mu)(x - mu)^T of the centred keys, fp32 (x - mu
//      rounded to fp32 once per element, 8 x 8 register blocks per thread);
//   3. top eigenvector v of C, i.e. the top right singular vector of the
//      centred key matrix, by power iteration (power.cuh) from the column of C
//      with the largest diagonal entry (first of equals);
//   4. sign: the component of largest magnitude (first of equals) is made
//      positive. C = 0 (all keys equal) has no direction: v = e_0;
//   5. v becomes the unit's frozen filter, and the k kept rows are re-scored
//      with it in the canonical order of score.cuh (the incoming rows are
//      scored by the launches that follow).
// A non-finite entry of C (a non-finite key, or keys too large for an fp32
// Gram) raises kDevNonFinite and freezes the zero filter.
#include "common.cuh"
#include "launch.h"
#include "params.h"
#include "power.cuh"
#include "score.cuh"

namespace evict {
namespace {

constexpr int kFzThreads = kPowerThreads;   // 256
constexpr int kFzTileRows = 32;
constexpr int kFzRowsPerHalfWarp = 4;       // kept rows re-scored per half-warp and round
constexpr size_t kFzSmem = (size_t)(kHeadDim * kPowerStride + kFzTileRows * kHeadDim) * sizeof(float);

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

// grid = n_layers * B * H, block = 256, dynamic shared memory kFzSmem.
template <bool kBf16>
__global__ void __launch_bounds__(kFzThreads) freeze_kernel(const __grid_constant__ GroupParams P) {
  extern __shared__ float fz_smem[];
  float* C = fz_smem;                                   // [128][kPowerStride]
  float* tile = fz_smem + kHeadDim * kPowerStride;      // [kFzTileRows][128]
  __shared__ double s_sum[2][kHeadDim];
  __shared__ float s_mu[kHeadDim], v[kHeadDim], w[kHeadDim];
  __shared__ float s_norm, s_delta;
  __shared__ int s_col, s_bad;
  const Shape& s = P.s;
  const int tid = threadIdx.x;
  const int bhn = s.batch * s.heads;
  const int u = blockIdx.x;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn;
  constexpr int kRowBytes = KeyRows<kBf16>::kRowBytes;
  KeyRows<kBf16> K{static_cast<const char*>(L.kst) + (size_t)bh * s.cap * kRowBytes,
                   static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes, s.k};
  const int n = s.k + s.m;

  // 1. column means (fp64; two row-interleaved halves, four chains each)
  {
    const int col = tid & (kHeadDim - 1), half = tid >> 7;
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int r = half;
    for (; r + 6 < n; r += 8) {
      a0 += K.elem(r, col);
      a1 += K.elem(r + 2, col);
      a2 += K.elem(r + 4, col);
      a3 += K.elem(r + 6, col);
    }
    for (; r < n; r += 2) a0 += K.elem(r, col);
    s_sum[half][col] = (a0 + a1) + (a2 + a3);
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (tid < kHeadDim) s_mu[tid] = (float)((s_sum[0][tid] + s_sum[1][tid]) / (double)n);
  __syncthreads();

  // 2. Gram of the centred keys
  const int i0 = (tid >> 4) * 8, j0 = (tid & 15) * 8;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  for (int r0 = 0; r0 < n; r0 += kFzTileRows) {
    for (int e = tid; e < kFzTileRows * kHeadDim; e += kFzThreads) {
      const int rr = e / kHeadDim, d = e % kHeadDim;
      const int r = r0 + rr;
      tile[e] = r < n ? K.elem(r, d) - s_mu[d] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < kFzTileRows; ++rr) {
      float a[8], b[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        a[x] = tile[rr * kHeadDim + i0 + x];
        b[x] = tile[rr * kHeadDim + j0 + x];
      }
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
    }
    __syncthreads();
  }
  bool bad = false;
#pragma unroll
  for (int x = 0; x < 8; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      bad |= !isfinite(acc[x][y]);
      C[(i0 + x) * kPowerStride + j0 + y] = acc[x][y];
    }
  if (bad) s_bad = 1;
  __syncthreads();

  // 3. top eigenvector; start from the column of the largest diagonal entry
  if (tid == 0) {
    int best = 0;
    for (int j = 1; j < kHeadDim; ++j)
      if (C[j * kPowerStride + j] > C[best * kPowerStride + best]) best = j;
    s_col = best;
    double nrm = 0.0;
    for (int i = 0; i < kHeadDim; ++i) nrm += (double)C[i * kPowerStride + best] * C[i * kPowerStride + best];
    s_norm = (float)sqrt(nrm);
  }
  __syncthreads();
  const bool bad_all = s_bad != 0;
  const bool flat = !bad_all && !(s_norm > 0.f);         // C = 0: every key equal
  if (tid < kHeadDim) {
    if (bad_all) v[tid] = 0.f;
    else if (flat) v[tid] = tid == 0 ? 1.f : 0.f;
    else v[tid] = C[tid * kPowerStride + s_col] / s_norm;
  }
  __syncthreads();
  if (!bad_all && !flat) power_iterate(C, v, w, &s_norm, &s_delta);

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
  __syncthreads();

  // 5. re-score the kept rows against the frozen filter
  const int c = tid & 15, hw = tid >> 4;
  float f[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = v[8 * c + j];
  float* out = L.score_st + (size_t)bh * s.cap;
  constexpr int kRowsPerRound = (kFzThreads / 16) * kFzRowsPerHalfWarp;
  for (int base = 0; base < s.k; base += kRowsPerRound) {
    RowLoad<kBf16> ld[kFzRowsPerHalfWarp];
#pragma unroll
    for (int j = 0; j < kFzRowsPerHalfWarp; ++j) {
      const int r = base + hw + 16 * j;
      if (r < s.k) ld[j].load(K.row(r), c); else ld[j].zero();
    }
#pragma unroll
    for (int j = 0; j < kFzRowsPerHalfWarp; ++j) {
      float x[8];
      ld[j].widen(x);
      const float sigma = canonical_score<kQFilters>(x, f, s.sign);
      const int r = base + hw + 16 * j;
      if (c == 0 && r < s.k) out[r] = sigma;
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
  if (dtype_bytes == 2)
    freeze_kernel<true><<<units, kFzThreads, kFzSmem, st>>>(P);
  else
    freeze_kernel<false><<<units, kFzThreads, kFzSmem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace evict
