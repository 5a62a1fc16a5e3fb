// codec.cu -- the FP8 encoding step alone: the codes of fp32 values, unscaled,
// produced by pack4 of tkq_device.cuh (the cvt.rn.satfinite conversion every
// cast ends with).  A diagnostic of the library, not an operation of the
// source pages: the casts only ever hand the conversion quotients of magnitude
// about fmt_max or less, so this entry is what lets the hardware conversion be
// compared with the format definition on every binary32 bit pattern,
// including values beyond the largest finite one, infinities and NaN.
//
// An elementwise stream: each thread converts four values (one 16-byte load)
// into four codes (one 4-byte store), grid-stride.
#include <cuda_runtime.h>

#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;

template <int FMT>
__global__ void __launch_bounds__(kThreads)
    fp8_encode_kernel(const float4* __restrict__ x, uint32_t* __restrict__ out, int64_t n4) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
        const float4 v = ld_ro(x + i);
        st_stream_u32(out + i, pack4<FMT>(v.x, v.y, v.z, v.w));
    }
}

}  // namespace

cudaError_t launch_fp8_encode(const float* x, void* out, int64_t n, int fmt,
                              cudaStream_t stream) {
    const int64_t n4 = n / 4;
    if (n4 == 0) return cudaSuccess;
    auto* k = fmt == kFmtE4M3 ? &fp8_encode_kernel<kFmtE4M3> : &fp8_encode_kernel<kFmtE5M2>;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0,
                                     (n4 + kThreads - 1) / kThreads);
    if (const cudaError_t e = upload_checks(stream)) return e;
    k<<<grid, kThreads, 0, stream>>>(reinterpret_cast<const float4*>(x),
                                     static_cast<uint32_t*>(out), n4);
    return cudaGetLastError();
}

}  // namespace tkq
