// swiglu_cast.cu -- SwiGLU (optionally times a per-row routing weight) fused
// with the per-token-group FP8 cast.
//
// The operation is swiglu_forward_and_per_token_cast of "DeepSeek开源
// TileKernels：用Python写的GPU算子逼近硬件性能上限" (itsolotime.com) §3.3:
// y = g / (1 + exp(-g)) * u [* w] in fp32, then absmax -> scale -> FP8 codes
// per 1x128 group of y, all in registers in one pass over HBM.
//
// GB300 design: the same flat group walk as the plain cast.  Output group
// g = t * (H/128) + j covers y[t, 128j : 128j+128]; it reads the 256-byte gate
// run at x[t, 128j] and the 256-byte up run at x[t, H + 128j].  The row index
// comes from a multiply-shift division by H/128.  Eight lanes per group, two
// 16-byte loads per half per lane, three xor shuffles for the absmax, and a
// persistent grid with UNROLL independent groups per warp in flight.
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 2;

template <int FMT, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads)
    swiglu_cast_kernel(const uint4* __restrict__ x, const float* __restrict__ w,
                       uint2* __restrict__ out, float* __restrict__ sf, uint32_t n_groups,
                       FastDiv div_g, int64_t row_u4, int64_t half_u4) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;
    const int j = lane & 7;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;
    const int64_t n_quads = (static_cast<int64_t>(n_groups) + 3) >> 2;

    for (int64_t q0 = warp; q0 < n_quads; q0 += n_warps * kUnroll) {
        uint4 ga[kUnroll], gb[kUnroll], ua[kUnroll], ub[kUnroll];
        float wt[kUnroll];
        int64_t g[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            g[u] = (q0 + u * n_warps) * 4 + sub;
            wt[u] = 1.0f;
            if (g[u] < n_groups) {
                const uint32_t gi = static_cast<uint32_t>(g[u]);
                const uint32_t t = fast_div(gi, div_g);
                const uint32_t cg = gi - t * div_g.d;
                const uint4* p = x + static_cast<int64_t>(t) * row_u4 + cg * 16;
                ga[u] = ld_stream(p + j);
                gb[u] = ld_stream(p + 8 + j);
                ua[u] = ld_stream(p + half_u4 + j);
                ub[u] = ld_stream(p + half_u4 + 8 + j);
                if constexpr (WEIGHTED) wt[u] = ld_stream_f32(w + t);
            } else {
                ga[u] = gb[u] = ua[u] = ub[u] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float gv[16], uv[16], y[16];
            unpack8(ga[u], gv);
            unpack8(gb[u], gv + 8);
            unpack8(ua[u], uv);
            unpack8(ub[u], uv + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                y[i] = swiglu(gv[i], uv[i]);
                if constexpr (WEIGHTED) y[i] = __fmul_rn(y[i], wt[u]);
            }
            float m = fmaxf(absmax8(y), absmax8(y + 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            float s, inv;
            group_scale<FMT>(m, s, inv);
            if (g[u] < n_groups) {
                st_stream(out + g[u] * 16 + j, quantize8_mul<FMT>(y, inv));
                st_stream(out + g[u] * 16 + 8 + j, quantize8_mul<FMT>(y + 8, inv));
                if (j == 0) st_stream(sf + g[u], s);
            }
        }
    }
}

FastDiv make_fast_div(uint32_t d) {
    // l = ceil(log2 d); m = floor(2^32 (2^l - d) / d) + 1; sh1 = min(l, 1);
    // sh2 = max(l - 1, 0)
    uint32_t l = 0;
    while ((uint64_t{1} << l) < d) ++l;
    const uint64_t m = (((uint64_t{1} << l) - d) << 32) / d + 1;
    FastDiv f;
    f.d = d;
    f.m = static_cast<uint32_t>(m);
    f.sh1 = l < 1 ? l : 1;
    f.sh2 = l > 1 ? l - 1 : 0;
    return f;
}

template <int FMT, bool WEIGHTED>
cudaError_t launch(const void* x, const float* w, void* out, float* sf, int64_t T, int64_t H,
                   cudaStream_t stream) {
    const void* k = reinterpret_cast<const void*>(&swiglu_cast_kernel<FMT, WEIGHTED>);
    const int64_t G = H / 128;
    const int64_t n_groups = T * G;
    const int64_t warps_needed = (n_groups + 3) / 4;
    const int grid = persistent_grid(k, kThreads, 0, (warps_needed + 7) / 8);
    swiglu_cast_kernel<FMT, WEIGHTED><<<grid, kThreads, 0, stream>>>(
        static_cast<const uint4*>(x), w, static_cast<uint2*>(out), sf,
        static_cast<uint32_t>(n_groups), make_fast_div(static_cast<uint32_t>(G)), H / 4, H / 8);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_cast(const void* x, const float* w, void* out, float* sf, int64_t T,
                               int64_t H, int fmt, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (fmt == kFmtE4M3)
        return w ? launch<kFmtE4M3, true>(x, w, out, sf, T, H, stream)
                 : launch<kFmtE4M3, false>(x, w, out, sf, T, H, stream);
    return w ? launch<kFmtE5M2, true>(x, w, out, sf, T, H, stream)
             : launch<kFmtE5M2, false>(x, w, out, sf, T, H, stream);
}

}  // namespace tkq
