// Power iteration for the top eigenvector of a symmetric 128 x 128 matrix held
// in shared memory (Golub & Van Loan, "Matrix Computations", §7.3.1: repeated
// multiplication by C and renormalisation converge to the dominant
// eigenvector at the rate |lambda2 / lambda1|).
#pragma once

#include "common.cuh"

namespace evict {
namespace {

constexpr int kPowerThreads = 256;          // threads of the calling CTA
constexpr int kPowerStride = kHeadDim + 1;  // padded row stride of C in shared memory
constexpr int kMaxPowerIters = 20000;

// c: shared [128][kPowerStride]; v: shared [128], a unit start vector on
// entry and the unit iterate on exit; w: shared [128] scratch; s_norm,
// s_delta: shared scratch words. Every thread of the CTA calls it. Stops
// after max_iters iterations at most.
__device__ __forceinline__ void power_iterate(const float* c, float* v, float* w, float* s_norm, float* s_delta,
                                              int max_iters = kMaxPowerIters) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = tid >> 1, half = tid & 1;
  for (int it = 0; it < max_iters; ++it) {
    float acc = 0.f;
    const float* cr = c + row * kPowerStride + half * 64;
    const float* vv = v + half * 64;
#pragma unroll 8
    for (int j = 0; j < 64; ++j) acc = fmaf(cr[j], vv[j], acc);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (half == 0) w[row] = acc;
    __syncthreads();
    if (tid < 32) {
      float ss = 0.f;
      for (int i = lane; i < kHeadDim; i += 32) ss += w[i] * w[i];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) *s_norm = sqrtf(ss);
    }
    __syncthreads();
    float d = 0.f;
    if (tid < kHeadDim) {
      const float nv = w[tid] / *s_norm;
      d = (nv - v[tid]) * (nv - v[tid]);
      v[tid] = nv;
    }
    if ((it & 15) != 15) {
      __syncthreads();
      continue;
    }
    if (tid == 0) *s_delta = 0.f;
    __syncthreads();
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0 && tid < kHeadDim) atomicAdd(s_delta, d);
    __syncthreads();
    // Stop once the unit iterate moves by less than 3e-6 over one iteration:
    // a few times the fp32 rounding floor of a 128-long matvec.
    if (*s_delta < 1e-11f) break;
  }
}

}  // namespace
}  // namespace evict
