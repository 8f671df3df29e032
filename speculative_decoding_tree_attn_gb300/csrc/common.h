// Internal helpers shared by the libtreeverify translation units: error
// reporting for the C ABI, CUDA error checks and per-device properties.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "../../include/treeverify.h"

namespace tv {

// Records a printf-style message as this thread's last error and returns code.
int fail(int code, const char* fmt, ...);

// Clears the thread's last error (called at the start of each entry point).
void clear_error();

// Checks a CUDA runtime result; on failure records it and returns TV_ERR_CUDA.
int cuda_fail(cudaError_t e, const char* what);

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
  size_t max_smem_optin = 0;
};

// Properties of the current device (cached per device id).
int current_device_info(DeviceInfo* info);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace tv

#define TV_CUDA_TRY(expr)                                   \
  do {                                                      \
    cudaError_t tv_err_ = (expr);                           \
    if (tv_err_ != cudaSuccess) return tv::cuda_fail(tv_err_, #expr); \
  } while (0)

// Launch check: reports configuration errors of the last launch.
#define TV_LAUNCH_CHECK(what)                                \
  do {                                                       \
    cudaError_t tv_err_ = cudaGetLastError();                \
    if (tv_err_ != cudaSuccess) return tv::cuda_fail(tv_err_, what); \
  } while (0)
