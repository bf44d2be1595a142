// evict_prefill_noalloc: one-shot KNorm / Q-Filters block eviction that
// allocates nothing.
//
// Why it exists: every other entry point works on a cache created by
// evict_init, which reserves device memory with cudaMalloc. Some callers
// cannot do that — code that runs while a CUDA graph is being captured,
// serving runtimes that hand out all device memory from their own pool at
// start-up and forbid later allocations, and plug-ins that live inside
// another framework's memory manager. This call takes the caller's input
// block and the caller's output buffers, and keeps its intermediate data
// (scores, the source map, per-(b,h) metadata and the compaction flags) in
// one file-scope device array of fixed size instead.
//
// The array (kNoallocScratchBytes, 8 MiB) is part of the library image: every
// GPU that loads the library holds it until the process exits. Its address
// is looked up once per device, with that device current, on the first call
// made on the device — make that first call before any stream capture.
// All calls on a device share the one array, so calls that overlap on the
// GPU (different streams, or different host threads without ordering) race.
// The array's first 256 bytes hold the device error word: kernels that give
// up a bounded wait or meet an index outside its bounds set it, nothing else
// clears it, and evict_noalloc_status reads and clears it.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/evict.h"
#include "api_internal.h"
#include "common.cuh"
#include "launch.h"
#include "params.h"

namespace evict {
namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The error word sits at the start of the array, at the same place for every call.
constexpr size_t kErrWordBytes = 256;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Device address of the scratch array on the current device (set-up on first use).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(EVICT_ELIMIT, "device ordinal %d above %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the no-allocation scratch");
    e = prepare_select();
    if (e != cudaSuccess) return cuda_fail(e, "select kernel attribute");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return EVICT_OK;
}

}  // namespace
}  // namespace evict

using namespace evict;

extern "C" int evict_prefill_noalloc(const evict_config* cfg, const void* k, const void* v, const int32_t* pos,
                                     int n, void* k_out, void* v_out, int32_t* pos_out, float* score_out) {
  if (!cfg) return fail(EVICT_EINVAL, "config is NULL");
  const evict_config& c = *cfg;
  if (c.method != EVICT_KNORM && c.method != EVICT_QFILTERS)
    return fail(EVICT_EINVAL, "evict_prefill_noalloc supports KNorm and Q-Filters");
  if (c.dtype != EVICT_BF16 && c.dtype != EVICT_FP32) return fail(EVICT_EINVAL, "unknown dtype %d", c.dtype);
  if (c.batch < 1 || c.n_kv_heads < 1) return fail(EVICT_EINVAL, "batch and n_kv_heads must be >= 1");
  if (c.head_dim != EVICT_HEAD_DIM) return fail(EVICT_EINVAL, "head_dim must be %d", EVICT_HEAD_DIM);
  if (c.budget < 1 || c.n_sink < 0 || c.recent < 0 || (long long)c.n_sink + c.recent >= c.budget)
    return fail(EVICT_EINVAL, "need budget >= 1 and 0 <= n_sink + recent < budget");
  if (c.method == EVICT_QFILTERS && (c.sign != 1 && c.sign != -1))
    return fail(EVICT_EINVAL, "sign must be +1 or -1");
  if (c.method == EVICT_QFILTERS && !c.filters) return fail(EVICT_EINVAL, "Q-Filters needs filters");
  if (c.method == EVICT_QFILTERS && c.n_filter_heads != 0 && c.n_filter_heads != c.n_kv_heads)
    return fail(EVICT_EINVAL, "filters hold %d heads but the layer has %d", c.n_filter_heads, c.n_kv_heads);
  if (c.method == EVICT_KNORM && c.keep_low != 0 && c.keep_low != 1)
    return fail(EVICT_EINVAL, "keep_low must be 0 or 1");
  if (n < 0) return fail(EVICT_EINVAL, "n must be >= 0");
  if (n == 0) return EVICT_OK;
  if (!k || !v || !k_out || !v_out || !pos_out || !score_out)
    return fail(EVICT_EINVAL, "input and output pointers must not be NULL");
  // 16-byte vector loads and bulk copies read k / v and write k_out / v_out; positions and scores
  // move as 4-byte words. A misaligned buffer is refused here, before anything is enqueued.
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_out, 16) || !aligned(v_out, 16))
    return fail(EVICT_EINVAL, "k, v, k_out and v_out must be 16-byte aligned");
  if (!aligned(pos, 4) || !aligned(pos_out, 4) || !aligned(score_out, 4))
    return fail(EVICT_EINVAL, "pos, pos_out and score_out must be 4-byte aligned");
  if (c.method == EVICT_QFILTERS && !aligned(c.filters, 4)) return fail(EVICT_EINVAL, "filters must be 4-byte aligned");
  if (n > EVICT_MAX_SELECT_ROWS) return fail(EVICT_ELIMIT, "n = %d above %d rows", n, EVICT_MAX_SELECT_ROWS);
  if ((long long)c.batch * c.n_kv_heads > 65535 / kMaxGroup) return fail(EVICT_ELIMIT, "batch * n_kv_heads too large");

  const int elem = c.dtype == EVICT_BF16 ? 2 : 4;
  const size_t bh = (size_t)c.batch * c.n_kv_heads;
  const int flag_stride = compact_flag_slots(c.budget, elem);
  const size_t off_score = kErrWordBytes;
  const size_t off_src = off_score + round256(bh * n * sizeof(float));
  const size_t off_meta = off_src + round256(bh * c.budget * sizeof(int32_t));
  const size_t off_flags = off_meta + round256(bh * sizeof(int2));
  const size_t need = off_flags + round256(bh * flag_stride * sizeof(int));
  if (need > kNoallocScratchBytes)
    return fail(EVICT_ELIMIT, "this call needs %zu bytes of scratch; the no-allocation path has %zu", need,
                kNoallocScratchBytes);

  void* base = nullptr;
  int rc = scratch_for_current_device(&base);
  if (rc) return rc;
  char* s = static_cast<char*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(c.stream);
  // Everything past the error word is written before it is read within this call (the select
  // kernel zeroes the compaction flags and counters). The error word starts at zero with the
  // library and is cleared only by evict_noalloc_status, so a failure is never lost.
  cudaError_t e = cudaSuccess;

  GroupParams P;
  memset(&P, 0, sizeof(P));
  P.s.batch = c.batch;
  P.s.heads = c.n_kv_heads;
  P.s.m = n;
  P.s.k = 0;
  P.s.cap = c.budget;
  P.s.budget = c.budget;
  P.s.n_sink = c.n_sink;
  P.s.recent = c.recent;
  P.s.new_stride = n;
  P.s.flag_stride = flag_stride;
  P.s.chunk = compact_chunk_rows(elem);
  P.s.n_layers = 1;
  P.s.keep_low = c.method == EVICT_KNORM ? c.keep_low : 0;
  P.s.sign = (float)(c.method == EVICT_QFILTERS ? c.sign : 1);
  P.s.method = c.method;
  P.s.offset = 0;
  P.err = reinterpret_cast<int*>(s);
  LayerPtrs& L = P.L[0];
  L.k_in = k;
  L.v_in = v;
  L.pos_in = pos;
  L.kst = k_out;
  L.vst = v_out;
  L.pos_st = pos_out;
  L.score_st = score_out;
  L.filters = const_cast<float*>(c.filters);   // read only: no fallback freeze here
  L.new_score = reinterpret_cast<float*>(s + off_score);
  L.src_map = reinterpret_cast<int32_t*>(s + off_src);
  L.meta = reinterpret_cast<int2*>(s + off_meta);
  L.flags = reinterpret_cast<int*>(s + off_flags);

  if (n <= c.budget) {
    e = launch_append(P, elem, st);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return cuda_fail(e, "append kernel launch");
    return EVICT_OK;
  }
  if ((e = launch_score(P, elem, st)) != cudaSuccess) return cuda_fail(e, "score kernel launch");
  if ((e = launch_select(P, st)) != cudaSuccess) return cuda_fail(e, "select kernel launch");
  if ((e = launch_compact(P, elem, st)) != cudaSuccess) return cuda_fail(e, "compact kernel launch");
  g_launches.fetch_add(3);
  return EVICT_OK;
}

extern "C" int evict_noalloc_status(void* stream) {
  void* base = nullptr;
  int rc = scratch_for_current_device(&base);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, base, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the no-allocation error word");
  if (word == kDevOk) return EVICT_OK;
  e = cudaMemsetAsync(base, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the no-allocation error word");
  return fail(EVICT_EDEVICE, "a no-allocation kernel reported %s",
              word == kDevWaitTimeout ? "a bounded wait that gave up" :
              word == kDevBadIndex ? "an index outside its bounds" : "an error");
}
