// per_token_cast.cu -- plain per-token-group FP8 cast of a bf16 [T, C] matrix.
//
// The operation is the per_token_cast of "DeepSeek开源TileKernels：用Python写的
// GPU算子逼近硬件性能上限" (itsolotime.com) §3.2: per 1x128 group, absmax ->
// scale -> FP8 codes of x / s.
//
// GB300 design: the input is a flat sequence of 1x128 groups (row-major [T, C]
// with C % 128 == 0 puts group g at byte 256*g of x, 128*g of out and 4*g of
// sf), so the kernel needs no row/column indexing.  Eight lanes share a group:
// lane j holds elements [8j, 8j+8) and [64+8j, 64+8j+8), so each of the two
// 16-byte loads of a warp reads four whole 128-byte lines and each 8-byte code
// store writes four whole 64-byte runs.  The group absmax is three xor
// shuffles.  A persistent grid (SMs x resident blocks) walks the groups with
// UNROLL independent steps in flight per warp to keep enough bytes in flight
// for HBM3e.  No shared memory, no tensor cores: the kernel is bound by HBM.
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <int FMT>
__global__ void __launch_bounds__(kThreads)
    per_token_cast_kernel(const uint4* __restrict__ x, uint2* __restrict__ out,
                          float* __restrict__ sf, int64_t n_groups) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;  // group within the warp's four
    const int j = lane & 7;     // position within the group
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    const int64_t n_quads = (n_groups + 3) >> 2;

    for (int64_t q0 = warp; q0 < n_quads; q0 += n_warps * kUnroll) {
        uint4 a[kUnroll], b[kUnroll];
        int64_t g[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            g[u] = (q0 + u * n_warps) * 4 + sub;
            if (g[u] < n_groups) {
                a[u] = ld_stream(x + g[u] * 16 + j);
                b[u] = ld_stream(x + g[u] * 16 + 8 + j);
            } else {
                a[u] = make_uint4(0, 0, 0, 0);
                b[u] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float v[16];
            unpack8(a[u], v);
            unpack8(b[u], v + 8);
            float m = fmaxf(absmax8(v), absmax8(v + 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            float s, inv;
            group_scale<FMT>(m, s, inv);
            if (g[u] < n_groups) {
                st_stream(out + g[u] * 16 + j, quantize8<FMT>(v, s, inv));
                st_stream(out + g[u] * 16 + 8 + j, quantize8<FMT>(v + 8, s, inv));
                if (j == 0) st_stream(sf + g[u], s);
            }
        }
    }
}

template <int FMT>
cudaError_t launch(const void* x, void* out, float* sf, int64_t n_groups, cudaStream_t stream) {
    const void* k = reinterpret_cast<const void*>(&per_token_cast_kernel<FMT>);
    const int64_t warps_needed = (n_groups + 3) / 4;
    const int grid = persistent_grid(k, kThreads, 0, (warps_needed + 7) / 8);
    per_token_cast_kernel<FMT><<<grid, kThreads, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint2*>(out), sf, n_groups);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_per_token_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                  int fmt, cudaStream_t stream) {
    const int64_t n_groups = T * (C / 128);
    if (n_groups == 0) return cudaSuccess;
    return fmt == kFmtE4M3 ? launch<kFmtE4M3>(x, out, sf, n_groups, stream)
                           : launch<kFmtE5M2>(x, out, sf, n_groups, stream);
}

}  // namespace tkq
