// Score kernels: fused per-key score (KNorm norm / Q-Filters projection) and
// the score + append path used while the cache stays within budget.
//
// Sources: "L2Norm — Intrinsic Key-Norm Eviction", §How it works step 1 (fp32
// L2 norm of each incoming key, computed once at insertion); "Q-Filters —
// Query-Agnostic Projection Eviction", §How it works step 3 (score =
// sign * (key . filter) in fp32, once) and §Metal kernels (fp32 accumulation
// over the stored keys).
//
// Evaluation order (fixed so that a key's score is a pure function of its
// bits, independent of block length or launch shape): a half-warp owns one
// key; lane c holds elements 8c..8c+7 and sums their products left to right
// with round-to-nearest multiplies and adds (no FMA contraction), then the 16
// lane sums are combined by an xor butterfly with strides 8, 4, 2, 1. The norm
// is the IEEE square root of that sum.
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

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  kernel<<<grid, block, smem, st>>>(P);
  return cudaGetLastError();
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
