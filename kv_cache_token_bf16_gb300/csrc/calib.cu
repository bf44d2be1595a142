// One-time Q-Filters calibration ("Q-Filters — Query-Agnostic Projection
// Eviction", §Calibrated — the paper's actual mechanism): per query head the
// top right singular vector v1 of the UNCENTERED activations Q^h [N, D],
// sign-fixed as sgn(1^T u1) * v1, then averaged over each GQA group onto its
// KV head and renormalised (§Evidence: GQA averaging keeps filters unit-norm).
//
// v1 is the top eigenvector of C = Q^T Q, and 1^T u1 = (1^T Q v1) / s1, so the
// sign is that of (sum of the query rows) . v1.
//
// Kernels:
//   calib_gram   partial C and row sums over a slice of the samples (fp32)
//   calib_eig    sums the partials (fp64), power iteration on C (fp32) from
//                the column of the largest diagonal entry until the iterate
//                stops moving, then the sign fix
//   calib_gqa    group average and renormalisation; flags a degenerate group
#include <cuda_runtime.h>

#include <cmath>
#include <vector>

#include "api_internal.h"
#include "common.cuh"
#include "power.cuh"

namespace evict {
namespace {

constexpr int kGramThreads = 256;
constexpr int kGramTileRows = 32;
constexpr int kEigThreads = kPowerThreads;
constexpr int kCStride = kPowerStride;

enum CalibStatus : int { kCalibOk = 0, kCalibZeroHead = 1, kCalibDegenerateGroup = 2 };

template <bool kBf16>
__device__ __forceinline__ float load_q(const void* q, size_t idx) {
  if (kBf16) return __uint_as_float((uint32_t)static_cast<const uint16_t*>(q)[idx] << 16);
  return static_cast<const float*>(q)[idx];
}

// grid = (splits, n_q_heads). Partial Gram over rows [split*chunk, ...).
template <bool kBf16>
__global__ void __launch_bounds__(kGramThreads)
calib_gram_kernel(const void* q, int n_samples, int chunk, float* part_c, float* part_sum) {
  __shared__ float tile[kGramTileRows][kHeadDim];
  const int split = blockIdx.x, head = blockIdx.y, splits = gridDim.x;
  const int tid = threadIdx.x;
  const int i0 = (tid >> 4) * 8, j0 = (tid & 15) * 8;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
  float colsum = 0.f;
  const int r_begin = split * chunk, r_end = min(n_samples, r_begin + chunk);
  const size_t head_base = (size_t)head * n_samples * kHeadDim;
  for (int r0 = r_begin; r0 < r_end; r0 += kGramTileRows) {
    for (int e = tid; e < kGramTileRows * kHeadDim; e += kGramThreads) {
      const int rr = e / kHeadDim, d = e % kHeadDim;
      const int row = r0 + rr;
      tile[rr][d] = row < r_end ? load_q<kBf16>(q, head_base + (size_t)row * kHeadDim + d) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < kGramTileRows; ++rr) {
      float a[8], b[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) { a[x] = tile[rr][i0 + x]; b[x] = tile[rr][j0 + x]; }
#pragma unroll
      for (int x = 0; x < 8; ++x)
#pragma unroll
        for (int y = 0; y < 8; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
    }
    if (tid < kHeadDim)
      for (int rr = 0; rr < kGramTileRows; ++rr) colsum += tile[rr][tid];
    __syncthreads();
  }
  float* out = part_c + ((size_t)head * splits + split) * kHeadDim * kHeadDim;
#pragma unroll
  for (int x = 0; x < 8; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) out[(i0 + x) * kHeadDim + j0 + y] = acc[x][y];
  if (tid < kHeadDim) part_sum[((size_t)head * splits + split) * kHeadDim + tid] = colsum;
}

// grid = n_q_heads. Top eigenvector of C by power iteration, sign-fixed.
__global__ void __launch_bounds__(kEigThreads)
calib_eig_kernel(const float* part_c, const float* part_sum, int splits, float* head_filters, int* status) {
  extern __shared__ float c[];                 // [128][129]
  __shared__ float v[kHeadDim], w[kHeadDim];
  __shared__ double qsum[kHeadDim];
  __shared__ float s_norm, s_delta;
  __shared__ int s_col;
  const int head = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < kHeadDim * kHeadDim; e += kEigThreads) {
    double acc = 0.0;
    for (int s = 0; s < splits; ++s) acc += part_c[((size_t)head * splits + s) * kHeadDim * kHeadDim + e];
    c[(e / kHeadDim) * kCStride + e % kHeadDim] = (float)acc;
  }
  if (tid < kHeadDim) {
    double acc = 0.0;
    for (int s = 0; s < splits; ++s) acc += part_sum[((size_t)head * splits + s) * kHeadDim + tid];
    qsum[tid] = acc;
  }
  __syncthreads();
  if (tid == 0) {
    int best = 0;
    for (int j = 1; j < kHeadDim; ++j)
      if (c[j * kCStride + j] > c[best * kCStride + best]) best = j;
    s_col = best;
    double nrm = 0.0;
    for (int i = 0; i < kHeadDim; ++i) nrm += (double)c[i * kCStride + best] * c[i * kCStride + best];
    s_norm = (float)sqrt(nrm);
  }
  __syncthreads();
  if (!(s_norm > 0.f)) {                       // all-zero queries: no direction
    if (tid == 0) atomicMax(status, (int)kCalibZeroHead);
    if (tid < kHeadDim) head_filters[(size_t)head * kHeadDim + tid] = 0.f;
    return;
  }
  if (tid < kHeadDim) v[tid] = c[tid * kCStride + s_col] / s_norm;
  __syncthreads();
  power_iterate(c, v, w, &s_norm, &s_delta);
  // sign = sgn(qsum . v) (ties -> +1)
  if (tid < 32) {
    double dot = 0.0;
    for (int i = lane; i < kHeadDim; i += 32) dot += qsum[i] * (double)v[i];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) s_norm = dot >= 0.0 ? 1.f : -1.f;
  }
  __syncthreads();
  if (tid < kHeadDim) head_filters[(size_t)head * kHeadDim + tid] = s_norm * v[tid];
}

// grid = n_kv_heads, block = 128. Average a contiguous group of query-head filters.
__global__ void calib_gqa_kernel(const float* head_filters, int group, float* out, int* status) {
  __shared__ float red[4];
  const int g = blockIdx.x, d = threadIdx.x, lane = d & 31;
  float acc = 0.f;
  for (int j = 0; j < group; ++j) acc += head_filters[((size_t)g * group + j) * kHeadDim + d];
  acc /= (float)group;
  float ss = acc * acc;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[d >> 5] = ss;
  __syncthreads();
  const float nrm = sqrtf(red[0] + red[1] + red[2] + red[3]);
  if (nrm < 1e-6f) {
    if (d == 0) atomicMax(status, (int)kCalibDegenerateGroup);
    out[(size_t)g * kHeadDim + d] = 0.f;
    return;
  }
  out[(size_t)g * kHeadDim + d] = acc / nrm;
}

}  // namespace
}  // namespace evict

using namespace evict;

extern "C" int evict_qfilters_calibrate(const void* q, int dtype, int n_q_heads, int n_samples, int head_dim,
                                        int n_kv_heads, float* filters_out, void* stream_ptr) {
  if (!q || !filters_out) return fail(EVICT_EINVAL, "q and filters_out must not be NULL");
  if (dtype != EVICT_BF16 && dtype != EVICT_FP32) return fail(EVICT_EINVAL, "unknown dtype %d", dtype);
  if (head_dim != EVICT_HEAD_DIM) return fail(EVICT_EINVAL, "head_dim must be %d", EVICT_HEAD_DIM);
  if (n_q_heads < 1 || n_kv_heads < 1 || n_samples < 1) return fail(EVICT_EINVAL, "sizes must be >= 1");
  if (n_q_heads % n_kv_heads) return fail(EVICT_EINVAL, "n_q_heads must be a multiple of n_kv_heads");
  if (n_q_heads > 65535) return fail(EVICT_ELIMIT, "too many query heads");
  cudaStream_t st = static_cast<cudaStream_t>(stream_ptr);
  const int splits = std::max(1, std::min(64, n_samples / 256));
  const int chunk = (n_samples + splits - 1) / splits;
  const size_t c_bytes = (size_t)n_q_heads * splits * kHeadDim * kHeadDim * sizeof(float);
  const size_t s_bytes = (size_t)n_q_heads * splits * kHeadDim * sizeof(float);
  const size_t f_bytes = (size_t)n_q_heads * kHeadDim * sizeof(float);
  char* scratch = nullptr;
  cudaError_t e = cudaMalloc(&scratch, c_bytes + s_bytes + f_bytes + 256);
  if (e != cudaSuccess) return cuda_fail(e, "calibration scratch allocation");
  float* part_c = reinterpret_cast<float*>(scratch);
  float* part_s = reinterpret_cast<float*>(scratch + c_bytes);
  float* head_f = reinterpret_cast<float*>(scratch + c_bytes + s_bytes);
  int* status = reinterpret_cast<int*>(scratch + c_bytes + s_bytes + f_bytes);
  int rc = EVICT_OK;
  const size_t eig_smem = (size_t)kHeadDim * kCStride * sizeof(float);
  do {
    if ((e = cudaMemsetAsync(status, 0, sizeof(int), st)) != cudaSuccess) { rc = cuda_fail(e, "memset"); break; }
    const dim3 grid(splits, n_q_heads);
    if (dtype == EVICT_BF16)
      calib_gram_kernel<true><<<grid, kGramThreads, 0, st>>>(q, n_samples, chunk, part_c, part_s);
    else
      calib_gram_kernel<false><<<grid, kGramThreads, 0, st>>>(q, n_samples, chunk, part_c, part_s);
    g_launches.fetch_add(1);
    if ((e = cudaFuncSetAttribute(calib_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)eig_smem)) != cudaSuccess) { rc = cuda_fail(e, "eig attribute"); break; }
    calib_eig_kernel<<<n_q_heads, kEigThreads, eig_smem, st>>>(part_c, part_s, splits, head_f, status);
    g_launches.fetch_add(1);
    calib_gqa_kernel<<<n_kv_heads, kHeadDim, 0, st>>>(head_f, n_q_heads / n_kv_heads, filters_out, status);
    g_launches.fetch_add(1);
    if ((e = cudaGetLastError()) != cudaSuccess) { rc = cuda_fail(e, "calibration launch"); break; }
    int hs = 0;
    if ((e = cudaMemcpyAsync(&hs, status, sizeof(int), cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
        (e = cudaStreamSynchronize(st)) != cudaSuccess) { rc = cuda_fail(e, "calibration"); break; }
    if (hs == kCalibZeroHead) rc = fail(EVICT_ENUM, "a query head has all-zero activations");
    else if (hs == kCalibDegenerateGroup) rc = fail(EVICT_ENUM, "a GQA group average is shorter than 1e-6");
  } while (false);
  cudaFree(scratch);
  return rc;
}
