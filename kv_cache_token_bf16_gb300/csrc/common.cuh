// Device helpers shared by the eviction kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace evict {

constexpr int kHeadDim = 128;
constexpr int kWarp = 32;

// Error codes written to the handle's device error word (first writer wins).
enum DeviceError : int {
  kDevOk = 0,
  kDevWaitTimeout = 1,   // a bounded inter-CTA wait gave up
  kDevBadIndex = 2,      // an index failed a bounds check
  kDevNonFinite = 3,     // the key-SVD fallback met a non-finite key Gram
};

// Spin limit of every inter-CTA wait (each spin sleeps ~100 ns; ~0.4 s total).
constexpr int kSpinLimit = 1 << 22;

// Programmatic dependent launch: every kernel of the eviction path is launched
// so that it may start while the previous kernel in the stream finishes, and
// waits here, before touching any memory, until that kernel has completed and
// its writes are visible. Without the launch attribute this is a no-op.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void raise_device_error(int* err, int code) {
  atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------------------
// Widening of 8 consecutive elements (one 16-byte bf16 load, or two fp32 loads)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bf16x8_to_f32(const uint4& r, float (&x)[8]) {
  x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xffff0000u);
  x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xffff0000u);
  x[4] = __uint_as_float(r.z << 16); x[5] = __uint_as_float(r.z & 0xffff0000u);
  x[6] = __uint_as_float(r.w << 16); x[7] = __uint_as_float(r.w & 0xffff0000u);
}

// Streaming 16-byte load that does not allocate in L1 (read-once data).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// Priority -> 32-bit order key. Higher key = higher priority (kept first).
// -0 is folded onto +0 and NaN onto -inf, so +-0 tie and NaN is evicted first.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(float p) {
  uint32_t b = __float_as_uint(p);
  if ((b & 0x7fffffffu) > 0x7f800000u) b = 0xff800000u;   // NaN -> -inf
  if ((b & 0x7fffffffu) == 0u) b = 0u;                     // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Release / acquire flag helpers for the ordered compaction.
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace evict
