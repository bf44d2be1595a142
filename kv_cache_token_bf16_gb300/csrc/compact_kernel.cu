// Order-preserving compaction ("Q-Filters — Query-Agnostic Projection
// Eviction", §Metal kernels: survivors are gathered preserving temporal
// order; §Adaptation notes: keys are copied bit-identically and positions are
// never renumbered).
#include "common.cuh"
#include "launch.h"
#include "params.h"

namespace evict {
namespace {

// ---------------------------------------------------------------------------
// Order-preserving in-place compaction.
//
// Destination rows are cut into chunks of kChunk rows; a CTA moves one chunk
// of one (layer, b, h). Every survivor moves to a destination at or below
// its source, so a chunk's writes can only clobber storage rows that LOWER
// chunks still have to read. With kept rows before the call (k > 0) each CTA
//   (1) takes the next chunk index of its (layer, b, h) from a per-unit
//       counter, so a lower chunk always belongs to a CTA that is already
//       running (every wait below ends);
//   (2) loads its sources into registers and proves the loads complete by
//       consuming them (an XOR into shared memory) before a barrier;
//   (3) publishes a read-done flag (release) and waits (acquire, bounded)
//       for the lower chunks whose kept-row sources lie in its destinations
//       (a range the select kernel recorded per chunk);
//   (4) stores.
// Rows below the first eviction never move and are not touched. Incoming
// survivors are read straight from the caller's K/V blocks, so with no kept
// rows (k = 0) nothing can be clobbered: the chunk is the CTA's own and no
// counter, flag or wait is used. The counter is the last slot of the unit's
// flag array; the select kernel zeroes both.
// ---------------------------------------------------------------------------
constexpr int kCompactThreads = 256;

template <int kRowBytes, int kChunk>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ GroupParams P) {
  constexpr int kVpr = kRowBytes / 16;                       // 16-byte vectors per row
  constexpr int kPer = kChunk * kVpr / kCompactThreads;      // vectors per thread (K and V each)
  static_assert(kChunk * kVpr % kCompactThreads == 0, "chunk must split evenly over the CTA");
  __shared__ int s_chunk, s_abort;
  __shared__ int2 s_wait;
  __shared__ volatile uint32_t s_sink[kCompactThreads];
  const Shape& s = P.s;
  const int tid = threadIdx.x;
  const int bhn = s.batch * s.heads;
  const int units = bhn * s.n_layers;
  const int u = blockIdx.x % units;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, b = bh / s.heads;
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  const int chunks = s.flag_stride - 1;
  const bool ordered = s.k > 0;                              // kept rows can be clobbered
  if (tid == 0) {
    s_chunk = ordered ? atomicAdd(&flags[chunks], 1) : (int)(blockIdx.x / units);   // per-unit chunk counter
    s_abort = 0;
  }
  __syncthreads();
  const int c = s_chunk;
  if (c >= chunks) {                                         // a stale counter: never index past the flags
    if (tid == 0) raise_device_error(P.err, kDevBadIndex);
    return;
  }
  if (tid == 0 && ordered) s_wait = L.waits[(size_t)bh * chunks + c];   // lower chunks to wait for
  int first = 0, old_kept = 0;
  if (ordered) {
    const int2 meta = L.meta[bh];
    first = meta.x;
    old_kept = meta.y;
  }
  const int d_lo = max(c * kChunk, first);
  const int d_hi = min(c * kChunk + kChunk, s.budget);
  if (d_lo >= d_hi) {
    if (tid == 0 && ordered) st_release(&flags[c], 1);
    return;
  }
  const int32_t* src = L.src_map + (size_t)bh * s.cap;
  const size_t plane = (size_t)bh * s.cap;
  const char* kst = static_cast<const char*>(L.kst);
  const char* vst = static_cast<const char*>(L.vst);
  const char* kin = static_cast<const char*>(L.k_in) + (size_t)bh * s.m * kRowBytes;
  const char* vin = static_cast<const char*>(L.v_in) + (size_t)bh * s.m * kRowBytes;
  const int rows = d_hi - d_lo;
  const int n_rows = s.k + s.m;

  // (2) loads into registers
  uint4 kr[kPer], vr[kPer];
  int32_t my_pos = 0;
  float my_score = 0.f;
  bool bad = false;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int idx = tid + q * kCompactThreads;
    const int r = idx / kVpr, vec = idx - r * kVpr;
    kr[q] = vr[q] = make_uint4(0, 0, 0, 0);
    if (r < rows) {
      const int sr = src[d_lo + r];
      if (sr < 0 || sr >= n_rows) {
        bad = true;
      } else if (sr < s.k) {
        kr[q] = reinterpret_cast<const uint4*>(kst + (plane + sr) * kRowBytes)[vec];
        vr[q] = reinterpret_cast<const uint4*>(vst + (plane + sr) * kRowBytes)[vec];
      } else {
        kr[q] = reinterpret_cast<const uint4*>(kin + (size_t)(sr - s.k) * kRowBytes)[vec];
        vr[q] = reinterpret_cast<const uint4*>(vin + (size_t)(sr - s.k) * kRowBytes)[vec];
      }
    }
  }
  if (tid < rows) {
    const int sr = src[d_lo + tid];
    if (sr < 0 || sr >= n_rows) {
      bad = true;
    } else if (sr < s.k) {
      my_pos = L.pos_st[plane + sr];
      my_score = L.score_st[plane + sr];
    } else {
      const int t = sr - s.k;
      my_pos = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      my_score = L.new_score[(size_t)bh * s.new_stride + t];
    }
  }
  uint32_t sink = (uint32_t)my_pos ^ __float_as_uint(my_score);
#pragma unroll
  for (int q = 0; q < kPer; ++q) sink ^= kr[q].x ^ kr[q].y ^ kr[q].z ^ kr[q].w ^ vr[q].x ^ vr[q].y ^ vr[q].z ^ vr[q].w;
  s_sink[tid] = sink;                                        // consumes every loaded value
  if (bad) s_abort = 1;
  __syncthreads();

  // (3) publish, then wait for the lower chunks that read our destinations
  if (tid == 0 && ordered) {
    st_release(&flags[c], 1);
    if (!s_abort) {
      const int2 w = s_wait;
      for (int j = w.x; j <= w.y && j < c; ++j) {
        int spins = 0;
        while (ld_acquire(&flags[j]) == 0) {
          if (++spins > kSpinLimit) {
            raise_device_error(P.err, kDevWaitTimeout);
            s_abort = 1;
            break;
          }
          __nanosleep(64);
        }
        if (s_abort) break;
      }
    } else {
      raise_device_error(P.err, kDevBadIndex);
    }
  } else if (tid == 0 && s_abort) {
    raise_device_error(P.err, kDevBadIndex);
  }
  __syncthreads();
  if (s_abort) return;

  // (4) stores
  char* kdst = static_cast<char*>(L.kst) + (plane + d_lo) * kRowBytes;
  char* vdst = static_cast<char*>(L.vst) + (plane + d_lo) * kRowBytes;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int idx = tid + q * kCompactThreads;
    if (idx / kVpr < rows) {
      reinterpret_cast<uint4*>(kdst)[idx] = kr[q];
      reinterpret_cast<uint4*>(vdst)[idx] = vr[q];
    }
  }
  if (tid < rows) {
    L.pos_st[plane + d_lo + tid] = my_pos;
    L.score_st[plane + d_lo + tid] = my_score;
  }
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  kernel<<<grid, block, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

int compact_chunk_rows(int dtype_bytes) { return dtype_bytes == 2 ? 64 : 32; }

int compact_flag_slots(int rows, int dtype_bytes) {
  const int chunk = compact_chunk_rows(dtype_bytes);
  return (rows + chunk - 1) / chunk + 1;          // one read-done flag per chunk + the chunk counter
}

cudaError_t launch_compact(GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const int chunk = compact_chunk_rows(dtype_bytes);
  const int chunks = (P.s.budget + chunk - 1) / chunk;
  P.total_ctas = chunks * P.s.n_layers * P.s.batch * P.s.heads;
  if (dtype_bytes == 2)
    return launch(compact_kernel<kHeadDim * 2, 64>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
  return launch(compact_kernel<kHeadDim * 4, 32>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
}

}  // namespace evict
