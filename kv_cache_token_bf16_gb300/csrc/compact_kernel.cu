// Order-preserving compaction ("Q-Filters — Query-Agnostic Projection
// Eviction", §Metal kernels: survivors are gathered preserving temporal
// order; §Adaptation notes: keys are copied bit-identically and positions are
// never renumbered).
#include "common.cuh"
#include "launch.h"
#include "params.h"
#include "tcgen05.cuh"

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
//   (2) gathers its source rows into shared memory with one bulk copy per
//       K / V row (all in flight at once, completing on one mbarrier) and
//       its positions / scores into registers, consumed into shared memory
//       before a barrier;
//   (3) publishes a read-done flag (release) and waits (acquire, bounded)
//       for the lower chunks whose kept-row sources lie in its destinations
//       (a range the select kernel recorded per chunk);
//   (4) writes the chunk's destination rows, which are contiguous, with one
//       bulk store for K and one for V.
// Rows below the first eviction never move and are not touched. Incoming
// survivors are read straight from the caller's K/V blocks, so with no kept
// rows (k = 0) nothing can be clobbered: the chunk is the CTA's own and no
// counter, flag or wait is used. The counter is the last slot of the unit's
// flag array; the select kernel zeroes both.
// ---------------------------------------------------------------------------
constexpr int kCompactThreads = 256;

// Bounded wait on the chunk's copy barrier (the thread sleeps between polls; 2 s at most);
// raises the device error on timeout.
__device__ __forceinline__ bool compact_wait(uint64_t* bar, int* err) {
  if (tc::mbar_try_wait(bar, 0)) return true;
  const uint64_t t0 = tc::global_ns();
  do {
    if (tc::mbar_try_wait_sleep(bar, 0, 20000)) return true;
  } while (tc::global_ns() - t0 < 2000000000ull);
  raise_device_error(err, kDevWaitTimeout);
  return false;
}

template <int kRowBytes, int kChunk>
__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const __grid_constant__ GroupParams P) {
  pdl_wait();
  static_assert(kChunk <= kCompactThreads, "one thread per destination row");
  extern __shared__ __align__(128) unsigned char c_smem[];   // the chunk's K rows, then its V rows
  __shared__ uint64_t s_bar;
  __shared__ int s_chunk, s_abort;
  __shared__ int2 s_wait;
  __shared__ volatile uint32_t s_sink[kChunk];
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
    tc::mbar_init(&s_bar, 1);
  }
  __syncthreads();
  const int c = s_chunk;
  if (c >= chunks) {                                         // a stale counter: never index past the flags
    if (tid == 0) raise_device_error(P.err, kDevBadIndex);
    return;
  }
  if (tid == 0 && ordered) s_wait = L.waits[(size_t)bh * chunks + c];   // lower chunks to wait for
  int first = 0;
  if (ordered) first = L.meta[bh].x;
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
  const uint32_t sk = tc::smem_u32(c_smem), sv = sk + kChunk * kRowBytes;

  // (2) sources: checked, then positions / scores into registers and K / V rows by bulk copies
  int sr = -1;
  int32_t my_pos = 0;
  float my_score = 0.f;
  if (tid < rows) {
    sr = src[d_lo + tid];
    if (sr < 0 || sr >= n_rows) {
      s_abort = 1;
    } else if (sr < s.k) {
      my_pos = L.pos_st[plane + sr];
      my_score = L.score_st[plane + sr];
    } else {
      const int t = sr - s.k;
      my_pos = L.pos_in ? L.pos_in[(size_t)b * s.m + t] : (int32_t)(s.offset + t);
      my_score = L.new_score[(size_t)bh * s.new_stride + t];
    }
  }
  if (tid == 0) tc::mbar_arrive_expect_tx(&s_bar, (uint32_t)(2 * rows * kRowBytes));
  __syncthreads();
  if (s_abort) {                                             // nothing issued yet: leave at once
    if (tid == 0) {
      raise_device_error(P.err, kDevBadIndex);
      if (ordered) st_release(&flags[c], 1);
    }
    return;
  }
  if (tid < rows) {
    const char* ks = sr < s.k ? kst + (plane + sr) * kRowBytes : kin + (size_t)(sr - s.k) * kRowBytes;
    const char* vs = sr < s.k ? vst + (plane + sr) * kRowBytes : vin + (size_t)(sr - s.k) * kRowBytes;
    tc::bulk_load(sk + (uint32_t)(tid * kRowBytes), ks, kRowBytes, &s_bar);
    tc::bulk_load(sv + (uint32_t)(tid * kRowBytes), vs, kRowBytes, &s_bar);
    s_sink[tid] = (uint32_t)my_pos ^ __float_as_uint(my_score);    // consumes the register loads
  }
  if (tid == 0 && !compact_wait(&s_bar, P.err)) {
    s_abort = 1;
    compact_wait(&s_bar, P.err);                             // the copies still in flight land first
  }
  __syncthreads();                                           // every source read has completed
  if (s_abort) {
    if (tid == 0 && ordered) st_release(&flags[c], 1);
    return;
  }

  // (3) publish, then wait for the lower chunks that read our destinations
  if (tid == 0 && ordered) {
    st_release(&flags[c], 1);
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
  }
  __syncthreads();
  if (s_abort) return;

  // (4) stores: the destination rows are contiguous
  if (tid == 0) {
    tc::bulk_store(static_cast<char*>(L.kst) + (plane + d_lo) * kRowBytes, sk, (uint32_t)(rows * kRowBytes));
    tc::bulk_store(static_cast<char*>(L.vst) + (plane + d_lo) * kRowBytes, sv, (uint32_t)(rows * kRowBytes));
    tc::bulk_commit();
  }
  if (tid < rows) {
    L.pos_st[plane + d_lo + tid] = my_pos;
    L.score_st[plane + d_lo + tid] = my_score;
  }
  if (tid == 0) tc::bulk_wait_all();
}

template <typename Kernel>
cudaError_t launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const GroupParams& P) {
  return launch_pdl(kernel, grid, block, smem, st, nullptr, P);
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
  // dynamic shared memory: the chunk's K and V rows (32 KB for either element size)
  if (dtype_bytes == 2)
    return launch(compact_kernel<kHeadDim * 2, 64>, dim3(P.total_ctas), dim3(kCompactThreads), 2 * 64 * kHeadDim * 2,
                  st, P);
  return launch(compact_kernel<kHeadDim * 4, 32>, dim3(P.total_ctas), dim3(kCompactThreads), 2 * 32 * kHeadDim * 4,
                st, P);
}

}  // namespace evict
