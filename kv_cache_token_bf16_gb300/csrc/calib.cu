// Q-Filters calibration (placeholder until the kernels land).
#include "api_internal.h"

extern "C" int evict_qfilters_calibrate(const void*, int, int, int, int, int, float*, void*) {
  return evict::fail(EVICT_EINVAL, "calibration is not available in this build yet");
}
