// cast_back.cu -- FP8 codes back to fp32 / bf16 ("TileKernels 与 DeepGEMM 的分界线"
// (chatdocs.ruinique.com) §2 operator table, cast_back):
//   out[t, c] = fl32(decode(code[t, c]) * s),  s = sf[t / gr, c / gc].
// Every E4M3 and E5M2 value is exactly a binary16 value (E5M2 is the upper
// byte of a binary16; E4M3's 3-bit mantissa and exponents 2^-9..2^8 fit
// binary16's range and precision), so the hardware conversion
// cvt.rn.f16x2.{e4m3,e5m2}x2 followed by an exact f16 -> f32 widening yields
// decode(code) exactly, and one binary32 multiply gives the result bit-exact.
// bf16 outputs round that fp32 product to nearest even.
//
// An HBM-bound stream (1 byte in, 4 or 2 bytes out per element): persistent
// CTAs of 256 threads walk units of rows; one thread turns 16 codes (one
// 16-byte load) of each of four rows into 16 outputs per row (64 or 32 bytes of
// 16-byte stores), with the four loads in flight together.
#include <cuda_runtime.h>

#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;

// Two FP8 codes (low byte = first element) -> binary16x2 (low half = first).
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t two) {
    uint32_t h;
    const uint16_t b = static_cast<uint16_t>(two);
    if constexpr (FMT == kFmtE4M3)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(b));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h) : "h"(b));
    return h;
}

__device__ __forceinline__ void f16x2_to_f32(uint32_t h, float& lo, float& hi) {
    asm("{ .reg .f16 l, u;\n\t"
        "mov.b32 {l, u}, %2;\n\t"
        "cvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, u; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

// 16 codes -> 16 exact values.
template <int FMT>
__device__ __forceinline__ void decode16(const uint4& q, float* v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[k]), v[4 * k + 0], v[4 * k + 1]);
        f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[k] >> 16), v[4 * k + 2], v[4 * k + 3]);
    }
}

// Two floats -> bf16x2, round to nearest even (low half = a).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Rows per thread and unit: the loads of kRowsPerThread rows are issued before
// any of them is used, so each thread keeps 4 x 16 bytes in flight.
constexpr int kRowsPerThread = 4;

// Work is split into units of R x kRowsPerThread rows (R = max(1, 256 / V),
// V = C / 16 vectors per row).  Thread i serves vector column i % V (and
// i % V + 256, ... for wide rows) of rows r, r + R, r + 2R, r + 3R of the unit,
// r = i / V, so rows of any width keep the threads busy.  GR_SHIFT: log2 of the
// scale group's rows (0 or 7).
template <int FMT, int GC, int GR_SHIFT, bool BF16>
__global__ void __launch_bounds__(kThreads, 3)
    cast_back_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ sf,
                     void* __restrict__ out, int64_t T, int64_t C, int R) {
    const int64_t V = C >> 4;
    const int r_in = static_cast<int>(threadIdx.x / V);  // < R when the thread is used
    const int v0 = static_cast<int>(threadIdx.x - static_cast<int64_t>(r_in) * V);
    if (r_in >= R) return;
    const int64_t G = C / GC;  // scales per row of sf
    const int64_t unit_rows = static_cast<int64_t>(R) * kRowsPerThread;
    const int64_t n_units = (T + unit_rows - 1) / unit_rows;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int64_t t0 = u * unit_rows + r_in;
        for (int64_t v = v0; v < V; v += kThreads) {
            uint4 q[kRowsPerThread];
#pragma unroll
            for (int k = 0; k < kRowsPerThread; ++k) {
                const int64_t t = t0 + static_cast<int64_t>(k) * R;
                q[k] = t < T ? ld_stream(reinterpret_cast<const uint4*>(codes + t * C) + v)
                             : make_uint4(0, 0, 0, 0);
            }
            const int64_t c = v * 16;
#pragma unroll
            for (int k = 0; k < kRowsPerThread; ++k) {
                const int64_t t = t0 + static_cast<int64_t>(k) * R;
                if (t >= T) break;
                const float* srow = sf + (t >> GR_SHIFT) * G;
                float s[16];
                if constexpr (GC == 1) {
                    const float4* s4 = reinterpret_cast<const float4*>(srow + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = ld_ro(s4 + i);
                        s[4 * i] = f.x; s[4 * i + 1] = f.y; s[4 * i + 2] = f.z; s[4 * i + 3] = f.w;
                    }
                } else {
                    const float one = ld_ro(srow + c / GC);
#pragma unroll
                    for (int i = 0; i < 16; ++i) s[i] = one;
                }
                float y[16];
                decode16<FMT>(q[k], y);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const float2 p = mul2(make_float2(y[i], y[i + 1]), make_float2(s[i], s[i + 1]));
                    y[i] = p.x;
                    y[i + 1] = p.y;
                }
                if constexpr (BF16) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + t * C + c);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        st_stream(dst + i, make_uint4(pack_bf16x2(y[8 * i], y[8 * i + 1]),
                                                      pack_bf16x2(y[8 * i + 2], y[8 * i + 3]),
                                                      pack_bf16x2(y[8 * i + 4], y[8 * i + 5]),
                                                      pack_bf16x2(y[8 * i + 6], y[8 * i + 7])));
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(out) + t * C + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_stream(dst + i, make_uint4(__float_as_uint(y[4 * i]),
                                                      __float_as_uint(y[4 * i + 1]),
                                                      __float_as_uint(y[4 * i + 2]),
                                                      __float_as_uint(y[4 * i + 3])));
                }
            }
        }
    }
}

template <int FMT, int GC, int GR_SHIFT, bool BF16>
cudaError_t launch(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                   cudaStream_t stream) {
    auto* k = &cast_back_kernel<FMT, GC, GR_SHIFT, BF16>;
    const int64_t V = C / 16;
    const int R = V >= kThreads ? 1 : static_cast<int>(kThreads / V);
    const int64_t unit_rows = static_cast<int64_t>(R) * kRowsPerThread;
    const int64_t n_units = (T + unit_rows - 1) / unit_rows;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0, n_units);
    if (const cudaError_t e = upload_checks(stream)) return e;
    k<<<grid, kThreads, 0, stream>>>(static_cast<const uint8_t*>(codes), sf, out, T, C, R);
    return cudaGetLastError();
}

template <int FMT, bool BF16>
cudaError_t launch_g(const void* codes, const float* sf, void* out, int64_t T, int64_t C, int gr,
                     int gc, cudaStream_t stream) {
    if (gc == 1) return launch<FMT, 1, 7, BF16>(codes, sf, out, T, C, stream);  // 128 x 1
    if (gr == 1) return launch<FMT, 128, 0, BF16>(codes, sf, out, T, C, stream);  // 1 x 128
    return launch<FMT, 128, 7, BF16>(codes, sf, out, T, C, stream);              // 128 x 128
}

template <int FMT>
cudaError_t launch_gc(const void* codes, const float* sf, void* out, int64_t T, int64_t C, int gr,
                      int gc, bool bf16, cudaStream_t stream) {
    return bf16 ? launch_g<FMT, true>(codes, sf, out, T, C, gr, gc, stream)
                : launch_g<FMT, false>(codes, sf, out, T, C, gr, gc, stream);
}

}  // namespace

cudaError_t launch_cast_back(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                             int gr, int gc, int fmt, bool out_bf16, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return fmt == kFmtE4M3 ? launch_gc<kFmtE4M3>(codes, sf, out, T, C, gr, gc, out_bf16, stream)
                           : launch_gc<kFmtE5M2>(codes, sf, out, T, C, gr, gc, out_bf16, stream);
}

}  // namespace tkq
