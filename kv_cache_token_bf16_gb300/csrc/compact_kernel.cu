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
// its source, so a chunk's writes can only clobber storage rows that lower
// chunks still have to read. Each CTA therefore (1) draws a ticket that
// orders chunks low-to-high (a lower ticket is already running), (2) reads
// its sources into shared memory and publishes a read-done flag (release),
// (3) waits (acquire, bounded) for the lower chunks whose storage sources
// overlap its destination range, and (4) writes. Rows below the first
// eviction never move and are not touched. Incoming survivors are read
// straight from the caller's K/V blocks.
// ---------------------------------------------------------------------------
constexpr int kCompactThreads = 256;

template <int kRowBytes, int kChunk>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ GroupParams P) {
  constexpr int kVpr = kRowBytes / 16;   // 16-byte vectors per row
  __shared__ uint4 sk[kChunk * kVpr];
  __shared__ uint4 sv[kChunk * kVpr];
  __shared__ int32_t spos[kChunk];
  __shared__ float sscore[kChunk];
  __shared__ int s_ticket, s_abort;
  const Shape& s = P.s;
  const int tid = threadIdx.x;
  if (tid == 0) {
    const int t = atomicAdd(P.ticket, 1);
    if (t == P.total_ctas - 1) atomicExch(P.ticket, 0);
    s_ticket = t;
    s_abort = 0;
  }
  __syncthreads();
  if (s_ticket >= P.total_ctas) {                // a stale counter: never index past the flags
    if (tid == 0) raise_device_error(P.err, kDevBadIndex);
    return;
  }
  const int bhn = s.batch * s.heads;
  const int units = bhn * s.n_layers;
  const int u = s_ticket % units;
  const int c = s_ticket / units;
  const LayerPtrs& L = P.L[u / bhn];
  const int bh = u % bhn, b = bh / s.heads;
  const int2 meta = L.meta[bh];
  const int first = meta.x, old_kept = meta.y;
  const int d_lo = max(c * kChunk, first);
  const int d_hi = min(c * kChunk + kChunk, s.budget);
  int* flags = L.flags + (size_t)bh * s.flag_stride;
  if (d_lo >= d_hi) {
    if (tid == 0) st_release(&flags[c], 1);
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
  for (int r = tid; r < rows; r += kCompactThreads) {
    const int sr = src[d_lo + r];
    if (sr < 0 || sr >= n_rows) s_abort = 1;
  }
  __syncthreads();
  if (s_abort) {                                  // corrupt map: record it, move nothing
    if (tid == 0) {
      raise_device_error(P.err, kDevBadIndex);
      st_release(&flags[c], 1);
    }
    return;
  }

  // (2) read phase
  for (int idx = tid; idx < rows * kVpr; idx += kCompactThreads) {
    const int r = idx / kVpr, vec = idx - r * kVpr;
    const int sr = src[d_lo + r];
    const char* kp;
    const char* vp;
    if (sr < s.k) {
      kp = kst + (plane + sr) * kRowBytes;
      vp = vst + (plane + sr) * kRowBytes;
    } else {
      kp = kin + (size_t)(sr - s.k) * kRowBytes;
      vp = vin + (size_t)(sr - s.k) * kRowBytes;
    }
    sk[idx] = reinterpret_cast<const uint4*>(kp)[vec];
    sv[idx] = reinterpret_cast<const uint4*>(vp)[vec];
  }
  for (int r = tid; r < rows; r += kCompactThreads) {
    const int sr = src[d_lo + r];
    if (sr < s.k) {
      spos[r] = L.pos_st[plane + sr];
      sscore[r] = L.score_st[plane + sr];
    } else {
      const int t = sr - s.k;
      spos[r] = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      sscore[r] = L.new_score[(size_t)bh * s.new_stride + t];
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    st_release(&flags[c], 1);
    // (3) wait for lower chunks whose storage sources overlap [d_lo, d_hi)
    for (int j = c - 1; j >= 0; --j) {
      if (j * kChunk + kChunk <= first) break;             // this and all lower chunks read nothing
      const int j_lo = max(j * kChunk, first);
      const int j_hi = min(j * kChunk + kChunk, old_kept); // storage-sourced destinations of chunk j
      if (j_lo >= j_hi) continue;                          // chunk j reads only incoming rows
      if (src[j_hi - 1] < d_lo) break;                     // chunk j (and lower) read below our range
      if (src[j_lo] >= d_hi) continue;                     // chunk j reads above our range
      int spins = 0;
      while (ld_acquire(&flags[j]) == 0) {
        if (++spins > kSpinLimit) {
          raise_device_error(P.err, kDevWaitTimeout);
          s_abort = 1;
          break;
        }
        __nanosleep(100);
      }
      if (s_abort) break;
    }
  }
  __syncthreads();
  if (s_abort) return;

  // (4) write phase
  char* kdst = static_cast<char*>(L.kst) + (plane + d_lo) * kRowBytes;
  char* vdst = static_cast<char*>(L.vst) + (plane + d_lo) * kRowBytes;
  for (int idx = tid; idx < rows * kVpr; idx += kCompactThreads) {
    reinterpret_cast<uint4*>(kdst)[idx] = sk[idx];
    reinterpret_cast<uint4*>(vdst)[idx] = sv[idx];
  }
  for (int r = tid; r < rows; r += kCompactThreads) {
    L.pos_st[plane + d_lo + r] = spos[r];
    L.score_st[plane + d_lo + r] = sscore[r];
  }
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  kernel<<<grid, block, smem, st>>>(P);
  return cudaGetLastError();
}

}  // namespace

int compact_chunk_rows(int dtype_bytes) { return dtype_bytes == 2 ? 32 : 16; }

cudaError_t launch_compact(GroupParams& P, int dtype_bytes, cudaStream_t st) {
  const int chunk = compact_chunk_rows(dtype_bytes);
  const int chunks = (P.s.budget + chunk - 1) / chunk;
  P.total_ctas = chunks * P.s.n_layers * P.s.batch * P.s.heads;
  if (dtype_bytes == 2)
    return launch(compact_kernel<kHeadDim * 2, 32>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
  return launch(compact_kernel<kHeadDim * 4, 16>, dim3(P.total_ctas), dim3(kCompactThreads), 0, st, P);
}

}  // namespace evict
