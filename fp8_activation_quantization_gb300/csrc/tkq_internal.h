// tkq_internal.h -- launchers behind the C ABI (include/tkq.h).  Arguments are
// validated by the ABI layer before these are called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tkq {

// Number of SMs of the current device (cached per device; the environment
// variable TKQ_NUM_SMS overrides it for grid sizing experiments).
int num_sms();

// Address of the library's device status word on the current device (bit
// kDeviceTimeout: a bounded wait inside a kernel gave up).  Resolved once per
// device with cudaGetSymbolAddress.
unsigned int* device_status_word();

// Persistent grid: min(blocks needed, SMs x resident blocks per SM).
int persistent_grid(const void* kernel, int threads, size_t smem, int64_t blocks_needed);

cudaError_t launch_per_token_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                  int fmt, cudaStream_t stream);

cudaError_t launch_swiglu_cast(const void* x, const float* w, void* out, float* sf, int64_t T,
                               int64_t H, int fmt, cudaStream_t stream);

cudaError_t launch_swiglu_cast_t(const void* x, const float* w, void* out, float* sf,
                                 void* out_t, float* sf_t, int64_t T, int64_t H, int fmt,
                                 cudaStream_t stream);

}  // namespace tkq
