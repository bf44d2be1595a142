// Canonical per-key score shared by the kernels that score keys.
//
// Sources: "L2Norm — Intrinsic Key-Norm Eviction", §How it works step 1 (fp32
// L2 norm of each incoming key, computed once at insertion); "Q-Filters —
// Query-Agnostic Projection Eviction", §How it works step 3 (score =
// sign * (key . filter) in fp32, once).
//
// Evaluation order (fixed so that a key's score is a pure function of its
// bits, independent of block length or launch shape): a half-warp owns one
// key; lane c holds elements 8c..8c+7 and sums their products left to right
// with round-to-nearest multiplies and adds (no FMA contraction), then the 16
// lane sums are combined by an xor butterfly with strides 8, 4, 2, 1. The norm
// is the IEEE square root of that sum. Every lane of the warp must call
// canonical_score together (full-mask shuffles).
#pragma once

#include "common.cuh"
#include "params.h"

namespace evict {
namespace {

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

// Filter row `row` of [rows, D]: the KV head for calibrated filters, the
// (b, h) unit for filters frozen by the key-SVD fallback.
__device__ __forceinline__ int filter_row(const Shape& s, int bh) {
  return s.filter_per_unit ? bh : bh % s.heads;
}

template <int kMethod>
__device__ __forceinline__ void load_filter(const float* filters, int row, int c, float (&f)[8]) {
  if (kMethod == kQFilters) {
    const float4* fp = reinterpret_cast<const float4*>(filters + (size_t)row * kHeadDim + 8 * c);
    float4 a = fp[0], b = fp[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] = 0.f;
  }
}

}  // namespace
}  // namespace evict
