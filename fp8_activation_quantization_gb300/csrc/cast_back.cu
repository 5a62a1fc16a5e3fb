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
// CTAs of 256 threads walk units of 4096 consecutive codes (rows wrap inside
// a unit); each thread turns 16 codes (one 16-byte load) into 16 outputs in a
// shared buffer, and the unit's 8 or 16 KB of output leave as one bulk-async
// store (cp.async.bulk global <- shared), double-buffered per CTA.  Written from the
// threads with 16-byte stores, this 1:2 read:write mix ran at 5.7 TB/s; the
// bulk stores and the occupancy of a lean kernel move it faster.
#include <cuda_runtime.h>

#include "tkq_async.cuh"
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

// Two floats -> bf16x2, round to nearest even (low half = a).
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Bulk-async store of `bytes` (a multiple of 16) from shared memory to global
// memory, tracked as one bulk group of the issuing thread; checked like every
// other store in the checked build.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    if (!access_ok(dst, bytes, true)) return;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// A unit is a run of kChunk consecutive codes of the row-major [T, C] matrix
// (16 per thread; the last unit may be shorter), rows wrapping inside it; its
// outputs are contiguous, so they leave as one bulk store.
constexpr int kChunk = kThreads * 16;

// Per unit: each thread loads its 16 codes (one 16-byte load) and their scale,
// waits until the shared buffer it writes (one of two) has been read by the
// bulk store issued from it two units earlier, decodes and scales eight
// values at a time into the buffer, and thread 0 issues the unit's bulk store.
// Many CTAs per SM (few registers) keep loads and stores in flight; the bulk
// stores write the output in 8 or 16 KB runs, which moves this 1:2
// read:write mix faster than 16-byte stores from the threads.  GR_SHIFT:
// log2 of the scale group's rows (0 or 7).
template <int FMT, int GC, int GR_SHIFT, bool BF16>
__global__ void __launch_bounds__(kThreads, BF16 ? 8 : 6)
    cast_back_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ sf,
                     uint8_t* __restrict__ out, int64_t T, int64_t C) {
    grid_dependency_sync();  // the previous grid on the stream is done
    constexpr int kOutBytes = BF16 ? 2 : 4;
    constexpr int kVecs = kOutBytes;   // 16-byte output vectors per thread and unit
    __shared__ __align__(128) uint4 buf[2][kThreads * kVecs];
    const int64_t total = T * C;
    const int64_t n_units = (total + kChunk - 1) / kChunk;
    const int64_t G = C / GC;                        // scales per row of sf
    // (row, column) of this CTA's unit starts u * kChunk, u = blockIdx.x +
    // k * gridDim.x, advanced by constants instead of divided out per unit
    const int64_t step = static_cast<int64_t>(gridDim.x) * kChunk;
    const int64_t step_t = step / C, step_c = step - step_t * C;
    int64_t t0 = static_cast<int64_t>(blockIdx.x) * kChunk / C;
    int64_t c0 = static_cast<int64_t>(blockIdx.x) * kChunk - t0 * C;
    const uint32_t Cu = static_cast<uint32_t>(C);
    int b = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, b ^= 1) {
        const int64_t f0 = u * kChunk;
        const int len = static_cast<int>(total - f0 < kChunk ? total - f0 : kChunk);
        const bool active = 16 * static_cast<int>(threadIdx.x) < len;
        // this thread's vector: row t, column c (rows wrap inside a unit)
        int64_t t = t0;
        uint32_t c = static_cast<uint32_t>(c0) + 16u * threadIdx.x;
        if (C >= kChunk) {
            if (c >= Cu) {
                c -= Cu;
                ++t;
            }
        } else {
            const uint32_t wrap = c / Cu;
            t += wrap;
            c -= wrap * Cu;
        }
        const float* srow = sf + (t >> GR_SHIFT) * G;
        uint4 q = make_uint4(0, 0, 0, 0);
        float s1 = 0.0f;
        if (active) {
            q = ld_stream(reinterpret_cast<const uint4*>(codes + f0) + threadIdx.x);
            if constexpr (GC != 1) s1 = ld_ro(srow + c / GC);
        }
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();   // buffer b is free
        if (active) {
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float y[8], sc[8];
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[2 * h]), y[0], y[1]);
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[2 * h] >> 16), y[2], y[3]);
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[2 * h + 1]), y[4], y[5]);
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(w[2 * h + 1] >> 16), y[6], y[7]);
                if constexpr (GC == 1) {
                    const float4* s4 = reinterpret_cast<const float4*>(srow + c + 8 * h);
                    const float4 a = ld_ro(s4), e = ld_ro(s4 + 1);
                    sc[0] = a.x; sc[1] = a.y; sc[2] = a.z; sc[3] = a.w;
                    sc[4] = e.x; sc[5] = e.y; sc[6] = e.z; sc[7] = e.w;
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) sc[i] = s1;
                }
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const float2 p =
                        mul2(make_float2(y[i], y[i + 1]), make_float2(sc[i], sc[i + 1]));
                    y[i] = p.x;
                    y[i + 1] = p.y;
                }
                uint4* dst = &buf[b][threadIdx.x * kVecs];
                if constexpr (BF16) {
                    dst[h] = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                        pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                } else {
                    dst[2 * h] = make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]),
                                            __float_as_uint(y[2]), __float_as_uint(y[3]));
                    dst[2 * h + 1] = make_uint4(__float_as_uint(y[4]), __float_as_uint(y[5]),
                                                __float_as_uint(y[6]), __float_as_uint(y[7]));
                }
            }
        }
        // the buffer's generic-proxy writes before the bulk copy reads it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0)
            bulk_store(out + f0 * kOutBytes, &buf[b][0], static_cast<uint32_t>(len) * kOutBytes);
        t0 += step_t;
        c0 += step_c;
        if (c0 >= C) {
            c0 -= C;
            ++t0;
        }
    }
    // the shared buffers must outlive the copies that read them
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <int FMT, int GC, int GR_SHIFT, bool BF16>
cudaError_t launch(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                   cudaStream_t stream) {
    auto* k = &cast_back_kernel<FMT, GC, GR_SHIFT, BF16>;
    const int64_t n_units = (T * C + kChunk - 1) / kChunk;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0, n_units);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kThreads, 0, stream, true, static_cast<const uint8_t*>(codes), sf,
                      static_cast<uint8_t*>(out), T, C);
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
