// swiglu_values.cu -- the fp32 values the SwiGLU casts quantize, written out
// instead of quantized:
//   * y = silu(g) * u [* w], exactly as the forward casts compute it (swiglu2
//     of tkq_device.cuh on the same bf16 operands);
//   * [dg | du], the gradients of the same SwiGLU from dy, exactly as the
//     backward cast computes them (swiglu_grad2 and the weight product).
// Diagnostics of the library, not operations of the source pages: they let
// the accuracy of the SM's ex2 / rcp based evaluation be checked value by
// value, which the casts' codes only show through rounding.
//
// Elementwise streams: each thread turns 8 channels of one row (16-byte bf16
// loads) into 8 fp32 values per output (16-byte stores); grid-stride over the
// 8-channel vectors of the rows.
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

template <bool WEIGHTED>
__global__ void __launch_bounds__(kThreads)
    swiglu_backward_values_kernel(const uint4* __restrict__ x, const uint4* __restrict__ dy,
                                  const float* __restrict__ w, float4* __restrict__ y, int64_t T,
                                  int64_t H) {
    const int64_t V = H >> 3;                      // 8-channel vectors per half row
    const int64_t n = T * V;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const int64_t t = i / V;
        const int64_t v = i - t * V;
        float g[8], u[8], d[8], dg[8], du[8];
        unpack8(ld_stream(x + t * (2 * V) + v), g);
        unpack8(ld_stream(x + t * (2 * V) + V + v), u);
        unpack8(ld_stream(dy + t * V + v), d);
        const float wt = WEIGHTED ? ld_ro(w + t) : 1.0f;
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            float2 a, b;
            swiglu_grad2(make_float2(g[k], g[k + 1]), make_float2(u[k], u[k + 1]),
                         make_float2(d[k], d[k + 1]), a, b);
            if constexpr (WEIGHTED) {
                a = mul2(a, make_float2(wt, wt));
                b = mul2(b, make_float2(wt, wt));
            }
            dg[k] = a.x;
            dg[k + 1] = a.y;
            du[k] = b.x;
            du[k + 1] = b.y;
        }
        // row t of y holds 4V float4: dg in [0, 2V), du in [2V, 4V)
        float4* row = y + t * (4 * V);
        st_plain(row + 2 * v, make_float4(dg[0], dg[1], dg[2], dg[3]));
        st_plain(row + 2 * v + 1, make_float4(dg[4], dg[5], dg[6], dg[7]));
        st_plain(row + 2 * V + 2 * v, make_float4(du[0], du[1], du[2], du[3]));
        st_plain(row + 2 * V + 2 * v + 1, make_float4(du[4], du[5], du[6], du[7]));
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

cudaError_t launch_swiglu_backward_values(const void* x, const void* dy, const float* w, float* y,
                                          int64_t T, int64_t H, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int64_t n = T * (H / 8);
    auto* k = w ? &swiglu_backward_values_kernel<true> : &swiglu_backward_values_kernel<false>;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0,
                                     (n + kThreads - 1) / kThreads);
    if (const cudaError_t e = upload_checks(stream)) return e;
    k<<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(x), static_cast<const uint4*>(dy),
                                     w, reinterpret_cast<float4*>(y), T, H);
    return cudaGetLastError();
}

}  // namespace tkq
