// CurDKV-adapted block scoring (placeholder until the kernels land).
#include "api_internal.h"

namespace evict {

struct CurdkvState {};

void curdkv_layout(evict_handle*, size_t*, char*) {}

int curdkv_prepare(evict_handle*) {
  return fail(EVICT_EINVAL, "CurDKV is not available in this build yet");
}

int curdkv_update(evict_handle*, const void*, const void*, const int32_t*, int) {
  return fail(EVICT_EINVAL, "CurDKV is not available in this build yet");
}

}  // namespace evict
