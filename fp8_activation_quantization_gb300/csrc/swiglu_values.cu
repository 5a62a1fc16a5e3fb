// swiglu_values.cu -- the fp32 SwiGLU values y = silu(g) * u [* w] exactly as
// the SwiGLU casts compute them (swiglu2 of tkq_device.cuh on the same bf16
// operands), written out instead of quantized.  A diagnostic of the library,
// not an operation of the source pages: it lets the accuracy of the SM's
// ex2 / rcp based SwiGLU be checked value by value, which the casts' codes
// only show through rounding.
//
// An elementwise stream: each thread turns 8 gates and 8 ups (two 16-byte
// loads) into 8 fp32 values (two 16-byte stores); grid-stride over the
// 8-channel vectors of the [T, H] output.
#include <cuda_runtime.h>

#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;

template <bool WEIGHTED>
__global__ void __launch_bounds__(kThreads)
    swiglu_values_kernel(const uint4* __restrict__ x, const float* __restrict__ w,
                         float4* __restrict__ y, int64_t T, int64_t H) {
    const int64_t V = H >> 3;                      // 8-channel vectors per row
    const int64_t n = T * V;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const int64_t t = i / V;
        const int64_t v = i - t * V;
        float g[8], u[8], r[8];
        unpack8(ld_stream(x + t * (2 * V) + v), g);
        unpack8(ld_stream(x + t * (2 * V) + V + v), u);
        const float wt = WEIGHTED ? ld_ro(w + t) : 1.0f;
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            float2 p = swiglu2(make_float2(g[k], g[k + 1]), make_float2(u[k], u[k + 1]));
            if constexpr (WEIGHTED) p = mul2(p, make_float2(wt, wt));
            r[k] = p.x;
            r[k + 1] = p.y;
        }
        st_plain(y + 2 * i, make_float4(r[0], r[1], r[2], r[3]));
        st_plain(y + 2 * i + 1, make_float4(r[4], r[5], r[6], r[7]));
    }
}

}  // namespace

cudaError_t launch_swiglu_values(const void* x, const float* w, float* y, int64_t T, int64_t H,
                                 cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int64_t n = T * (H / 8);
    auto* k = w ? &swiglu_values_kernel<true> : &swiglu_values_kernel<false>;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0,
                                     (n + kThreads - 1) / kThreads);
    if (const cudaError_t e = upload_checks(stream)) return e;
    k<<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(x), w, reinterpret_cast<float4*>(y),
                                     T, H);
    return cudaGetLastError();
}

}  // namespace tkq
