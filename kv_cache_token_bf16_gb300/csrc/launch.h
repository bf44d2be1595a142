// Host-side launchers of the eviction kernels (implemented in the .cu files).
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "params.h"

namespace evict {

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous kernel in the stream is still finishing (it waits for it
// in its first statement, pdl_wait), which hides the launch gap between the
// path's kernels. `extra` may add one more attribute (a cluster shape).
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const cudaLaunchAttribute* extra, Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (extra) attr[n++] = *extra;
  lc.attrs = attr;
  lc.numAttrs = n;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// Rows per compaction chunk for an element size of 2 (bf16) or 4 (fp32) bytes.
int compact_chunk_rows(int dtype_bytes);
// Flag slots per (b, h) for caches of `rows` rows: chunk flags plus a chunk counter.
int compact_flag_slots(int rows, int dtype_bytes);

cudaError_t launch_score(const GroupParams& P, int dtype_bytes, cudaStream_t st);
cudaError_t launch_append(const GroupParams& P, int dtype_bytes, cudaStream_t st);
// Raise the select kernel's dynamic shared memory limit (current device) to
// hold EVICT_MAX_SELECT_ROWS keys.
cudaError_t prepare_select();
cudaError_t launch_select(const GroupParams& P, cudaStream_t st);
// Sets P.total_ctas.
cudaError_t launch_compact(GroupParams& P, int dtype_bytes, cudaStream_t st);
// Fused score + single eviction + one-row shift (the concatenation exceeds the
// budget by exactly one row and m <= evict1_max_block()).
int evict1_max_block();
// Raise the single-eviction kernel's dynamic shared memory limit (current device).
cudaError_t prepare_evict1();
cudaError_t launch_evict1(const GroupParams& P, int dtype_bytes, cudaStream_t st);
// Q-Filters key-SVD fallback: estimate and freeze every unit's filter from the
// keys present (kept rows, then the block) and re-score the kept rows.
cudaError_t prepare_freeze();
cudaError_t launch_freeze(const GroupParams& P, int dtype_bytes, cudaStream_t st);

}  // namespace evict
