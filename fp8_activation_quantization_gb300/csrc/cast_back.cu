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
// a unit); each thread turns 16 codes (two 8-code or four 4-code pieces, see
// PieceShape) into 16 outputs in a shared buffer, and the unit's 8 or 16 KB
// of output leave as one bulk-async store (cp.async.bulk global <- shared),
// double-buffered per CTA.  Written from the
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

// A thread's 16 codes of a unit are kPieces pieces of kPiece consecutive
// codes, piece p at unit offset p * kPieceStride + kPiece * thread: each piece
// makes 16 output bytes, which land next to the neighbouring thread's piece
// in the shared buffer, so every 16-byte store of a warp covers 512
// consecutive bytes (no bank conflicts; one 16-code run per thread would put
// a thread's two or four 16-byte stores 32 or 64 bytes apart, two-way
// conflicts).  A unit's length is a multiple of 128 codes (C is), so a piece
// is wholly in or out of it, and never crosses a 128-column scale group.
template <bool BF16>
struct PieceShape {
    static constexpr int kPiece = BF16 ? 8 : 4;          // codes per piece
    static constexpr int kPieces = 16 / kPiece;           // pieces per thread
    static constexpr int kStride = kThreads * kPiece;     // unit offset between pieces
};

__device__ __forceinline__ uint2 ld_stream_u2(const uint8_t* p) {
    uint2 r = make_uint2(0, 0);
    if (!access_ok(p, 8, false)) return r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ld_stream_u1(const uint8_t* p) {
    uint32_t r = 0;
    if (!access_ok(p, 4, false)) return r;
    asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// Per unit: each thread loads its pieces' codes and scales, waits until the
// shared buffer it writes (one of two) has been read by the bulk store issued
// from it two units earlier, decodes and scales the pieces into the buffer,
// and thread 0 issues the unit's bulk store.  Many CTAs per SM (few
// registers) keep loads and stores in flight; the bulk stores write the
// output in 8 or 16 KB runs, which moves this 1:2 read:write mix faster than
// 16-byte stores from the threads.  GR_SHIFT: log2 of the scale group's rows
// (0 or 7).
template <int FMT, int GC, int GR_SHIFT, bool BF16>
__global__ void __launch_bounds__(kThreads, BF16 ? 8 : 6)
    cast_back_kernel(const uint8_t* __restrict__ codes, const float* __restrict__ sf,
                     uint8_t* __restrict__ out, int64_t T, int64_t C, int prefetch_units) {
    using PS = PieceShape<BF16>;
    constexpr int kOutBytes = BF16 ? 2 : 4;
    __shared__ __align__(128) uint4 buf[2][kThreads * PS::kPieces];
    const int64_t total = T * C;
    const int64_t n_units = (total + kChunk - 1) / kChunk;
    grid_dependency_launch();
    // the codes of the CTA's first prefetch_units units go to L2 while the
    // grid before this one drains; then wait until it is done
    if (threadIdx.x == 0) {
        for (int p = 0; p < prefetch_units; ++p) {
            const int64_t u = blockIdx.x + static_cast<int64_t>(p) * gridDim.x;
            if ((u + 1) * kChunk <= total) prefetch_l2(codes + u * kChunk, kChunk);
        }
    }
    grid_dependency_wait();
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
        uint32_t q[PS::kPieces][PS::kPiece / 4];
        float sc[PS::kPieces][PS::kPiece];
        bool live[PS::kPieces];
#pragma unroll
        for (int p = 0; p < PS::kPieces; ++p) {
            const int off = p * PS::kStride + PS::kPiece * static_cast<int>(threadIdx.x);
            live[p] = off < len;
            // this piece's row t and column c (rows wrap inside a unit)
            int64_t t = t0;
            uint32_t c = static_cast<uint32_t>(c0) + static_cast<uint32_t>(off);
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
#pragma unroll
            for (int k = 0; k < PS::kPiece / 4; ++k) q[p][k] = 0;
#pragma unroll
            for (int k = 0; k < PS::kPiece; ++k) sc[p][k] = 0.0f;
            if (live[p]) {
                if constexpr (BF16) {
                    const uint2 v = ld_stream_u2(codes + f0 + off);
                    q[p][0] = v.x;
                    q[p][1] = v.y;
                } else {
                    q[p][0] = ld_stream_u1(codes + f0 + off);
                }
                if constexpr (GC == 1) {
#pragma unroll
                    for (int k = 0; k < PS::kPiece; k += 4) {
                        const float4 a = ld_ro(reinterpret_cast<const float4*>(srow + c + k));
                        sc[p][k] = a.x;
                        sc[p][k + 1] = a.y;
                        sc[p][k + 2] = a.z;
                        sc[p][k + 3] = a.w;
                    }
                } else {
                    const float s1 = ld_ro(srow + c / GC);
#pragma unroll
                    for (int k = 0; k < PS::kPiece; ++k) sc[p][k] = s1;
                }
            }
        }
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();   // buffer b is free
#pragma unroll
        for (int p = 0; p < PS::kPieces; ++p) {
            if (!live[p]) continue;
            float y[PS::kPiece];
#pragma unroll
            for (int k = 0; k < PS::kPiece / 4; ++k) {
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(q[p][k]), y[4 * k], y[4 * k + 1]);
                f16x2_to_f32(fp8x2_to_f16x2<FMT>(q[p][k] >> 16), y[4 * k + 2], y[4 * k + 3]);
            }
#pragma unroll
            for (int i = 0; i < PS::kPiece; i += 2) {
                const float2 r = mul2(make_float2(y[i], y[i + 1]),
                                      make_float2(sc[p][i], sc[p][i + 1]));
                y[i] = r.x;
                y[i + 1] = r.y;
            }
            uint4& dst = buf[b][p * kThreads + threadIdx.x];
            if constexpr (BF16)
                dst = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                 pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            else
                dst = make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]),
                                 __float_as_uint(y[2]), __float_as_uint(y[3]));
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
                      static_cast<uint8_t*>(out), T, C, prologue_prefetch_units(T * C));
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
