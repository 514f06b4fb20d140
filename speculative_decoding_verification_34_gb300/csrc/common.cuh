// Internal helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>

#include "specverify.h"

namespace specverify {

// Per-thread message for spec_last_error().
void set_error(const char* fmt, ...);
void clear_error();
// Count of kernels launched by the library (spec_launch_count()).
void count_launch(uint64_t n = 1);

inline int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return SPEC_ECUDA;
}

}  // namespace specverify
