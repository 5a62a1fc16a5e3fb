// token_cast.cu -- the plain per_token_cast of a bf16 or fp32 [T, C] matrix
// ("DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限"
// (itsolotime.com) §3.2): per 1x128 group along channels, absmax -> scale
// s = fl32(max(amax, 1e-4) / fmt_max) -> the FP8 codes of the exact binary32
// quotient fl(x / s) (bit-exact), or with TKQ_Q_RECIPROCAL those of
// x * fl(1 / s).
//
// GB300 design: with C a multiple of 128, a row-major [T, C] matrix is, group
// by group, one flat sequence: group g holds elements [128 g, 128 g + 128) and
// its row-major fp32 scale is sf[g].  The cast is therefore a flat stream over
// the T * C / 128 groups with no row or tile bookkeeping and no ragged edge:
// a warp takes units of four consecutive groups (lane l: 16 consecutive
// elements, eight lanes per group, the group absmax in three xor shuffles),
// grid-stride over persistent CTAs of 256 threads (five per SM for bf16
// input, four for fp32).  Each lane issues the global loads of its next unit
// before it works on the current one, so two units per warp are in flight; a
// warp's loads are 16-byte vectors covering 1 KB (bf16) or 2 KB (fp32) of
// consecutive input, its code stores 16-byte vectors covering 512 B.
// (A TMA ring in shared memory is not needed for this access pattern: the
// flat stream measured 8-14 % faster than one on the same inputs.)
//
// Scale layouts other than row-major fp32 (TKQ_SF_* flags) need the row and
// group index of g; the column-major layouts also own padding rows
// T <= row < round_up(T, 4), whose scales are zeros: the walk then runs over
// round_up(T, 4) rows' groups, and groups past the last row load nothing and
// store only that zero scale.
#include <cuda_runtime.h>

#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// The 16 input values of lane `lane` in unit u, as 16-byte vectors: two of
// bf16 or four of fp32.
template <bool F32>
struct Slice {
    static constexpr int kVecs = F32 ? 4 : 2;
    uint4 q[kVecs];

    __device__ __forceinline__ void load(const uint4* x, int64_t u, int lane) {
        const uint4* p = x + (u * 32 + lane) * kVecs;
#pragma unroll
        for (int k = 0; k < kVecs; ++k) q[k] = ld_stream(p + k);
    }
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int k = 0; k < kVecs; ++k) q[k] = make_uint4(0, 0, 0, 0);
    }
    __device__ __forceinline__ void values(float* v) const {
        if constexpr (F32) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[4 * k] = __uint_as_float(q[k].x);
                v[4 * k + 1] = __uint_as_float(q[k].y);
                v[4 * k + 2] = __uint_as_float(q[k].z);
                v[4 * k + 3] = __uint_as_float(q[k].w);
            }
        } else {
            unpack8(q[0], v);
            unpack8(q[1], v + 8);
        }
    }
};

// n_groups = T * G groups hold data; n_walk >= n_groups groups are visited
// (the column-major layouts' padding rows); G = C / 128 groups per row.
// CTAs per SM: five (<= 48 registers) for bf16 input, four (<= 64) for fp32,
// whose lanes hold twice the input bytes.  Measured back to back on
// [8192, 7168] bf16, five took every option set from 29.1-29.4 us (four) to
// 27.9-28.3 us: the extra warps keep more loads in flight, and the two
// layouts that spill a few bytes at that cap gained as much as the rest.  Six
// (<= 40 registers) spill 16-56 bytes per thread.
template <bool F32>
constexpr int ctas_per_sm() {
    return F32 ? 4 : 5;
}

template <int FMT, bool F32, unsigned SFC>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<F32>())
    token_cast_kernel(const uint4* __restrict__ x, uint4* __restrict__ out,
                      float* __restrict__ sf, SfLayout lay, int64_t n_groups, int64_t n_walk,
                      int prefetch_units) {
    grid_dependency_launch();
    // LAYOUT: the scales are not flat row-major fp32 (store_scale needs the
    // group's row and index in the row); a fixed option set's flags are
    // compile-time constants from here on
    constexpr bool LAYOUT = SFC != kSfcNone && SFC != kSfcReciprocal;
    if constexpr (SFC != kSfcNone && SFC != kSfcRuntime) lay.flags = SFC;
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;    // group within the unit
    const int j = lane & 7;       // lane within the group
    const int64_t units = (n_walk + 3) / 4;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kWarps;
    int64_t u = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    // the warp's first prefetch_units (<= 4) units go to L2 while the grid
    // before this one drains; then wait until it is done.  (A loop bounded by
    // prefetch_units alone compiled the fp32 instance into one that ran
    // 52.1 us instead of 48.3 us on [8192, 7168]; this unrolled form does not.)
    constexpr unsigned kUnitBytes = 32 * Slice<F32>::kVecs * 16;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int64_t up = u + p * step;
        if (p < prefetch_units && lane == 0 && up < units && up * 4 + 3 < n_groups)
            prefetch_l2(x + up * 32 * Slice<F32>::kVecs, kUnitBytes);
    }
    grid_dependency_wait();

    // row and group-in-row of this lane's group, for the scale layouts: found
    // by one division here, then advanced by the fixed stride with one carry
    int64_t row = 0, drow = 0;
    int gj = 0, dgj = 0;
    if constexpr (LAYOUT) {
        const int64_t g0 = u * 4 + sub;
        row = g0 / lay.groups;
        gj = static_cast<int>(g0 - row * lay.groups);
        drow = step * 4 / lay.groups;
        dgj = static_cast<int>(step * 4 - drow * lay.groups);
    }

    Slice<F32> cur;
    cur.clear();
    if (u < units && u * 4 + sub < n_groups) cur.load(x, u, lane);
    for (; u < units; u += step) {
        const int64_t g = u * 4 + sub;
        const bool live = g < n_groups;
        float v[16];
        cur.values(v);
        // the next unit's loads go out before this unit's arithmetic
        const int64_t un = u + step;
        if (un < units && un * 4 + sub < n_groups) cur.load(x, un, lane);

        float m = fmaxf(absmax8(v), absmax8(v + 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        float sc, inv;
        group_scale<FMT>(m, sc, inv);
        bool exact_div = true;
        if constexpr (SFC != kSfcNone) {
            if (lay.flags & kQReciprocal) exact_div = false;
            if (lay.flags & (kSfRoundPow2 | kSfPacked)) {
                // y / s = y * 2^-k is then exact, so the product needs no correction
                pow2_scale(sc, inv);
                exact_div = false;
            }
        }
        if (live) {
            uint2 lo, hi;
            if (exact_div) {
                lo = quantize8<FMT>(v, sc, inv);
                hi = quantize8<FMT>(v + 8, sc, inv);
            } else {
                lo = quantize8_mul<FMT>(v, inv);
                hi = quantize8_mul<FMT>(v + 8, inv);
            }
            st_stream(out + u * 32 + lane, make_uint4(lo.x, lo.y, hi.x, hi.y));
        }
        if constexpr (LAYOUT) {
            if (j == 0 && g < n_walk) store_scale(sf, lay, row, live, gj, sc);
            row += drow;
            gj += dgj;
            if (gj >= lay.groups) {
                gj -= lay.groups;
                ++row;
            }
        } else {
            if (j == 0 && live) st_stream(sf + g, sc);
        }
    }
}

template <int FMT, bool F32, unsigned SFC>
cudaError_t launch_layout(const void* x, void* out, float* sf, const SfLayout& lay,
                          int64_t n_groups, int64_t n_walk, cudaStream_t stream) {
    auto* k = &token_cast_kernel<FMT, F32, SFC>;
    const int64_t units = (n_walk + 3) / 4;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0,
                                     (units + kWarps - 1) / kWarps);
    if (const cudaError_t e = upload_checks(stream)) return e;
    const int64_t in_bytes = n_groups * 128 * (F32 ? 4 : 2);
    return launch_pdl(k, grid, kThreads, 0, stream, true, static_cast<const uint4*>(x),
                      static_cast<uint4*>(out), sf, lay, n_groups, n_walk,
                      prologue_prefetch_units(in_bytes));
}

// The instance for the launch's flags: fixed option sets for no options, the
// reciprocal reading alone and the two GEMM layouts, else flags at run time
// (measured back to back on the plain_outlier workload, the run-time instance
// took 29.8 us with the reciprocal reading against 28.9 us without options).
template <int FMT, bool F32>
cudaError_t launch_sfc(const void* x, void* out, float* sf, const SfLayout& lay,
                       int64_t n_groups, int64_t n_walk, cudaStream_t stream) {
    switch (sfc_of(lay.flags, true)) {
        case kSfcNone:
            return launch_layout<FMT, F32, kSfcNone>(x, out, sf, lay, n_groups, n_walk, stream);
        case kSfcReciprocal:
            return launch_layout<FMT, F32, kSfcReciprocal>(x, out, sf, lay, n_groups, n_walk,
                                                           stream);
        case kSfcUe8m0ColMajor:
            return launch_layout<FMT, F32, kSfcUe8m0ColMajor>(x, out, sf, lay, n_groups, n_walk,
                                                              stream);
        case kSfcF32ColMajor:
            return launch_layout<FMT, F32, kSfcF32ColMajor>(x, out, sf, lay, n_groups, n_walk,
                                                            stream);
        default:
            return launch_layout<FMT, F32, kSfcRuntime>(x, out, sf, lay, n_groups, n_walk,
                                                        stream);
    }
}

template <bool F32>
cudaError_t launch(const void* x, void* out, void* sf, int64_t T, int64_t C, int fmt,
                   unsigned sf_flags, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    SfLayout lay;
    lay.flags = sf_flags;
    lay.groups = static_cast<int>(C / 128);
    lay.words = (lay.groups + 3) / 4;
    lay.rows4 = (T + 3) / 4 * 4;
    const int64_t n_groups = T * lay.groups;
    const int64_t n_walk = (sf_flags & kSfColMajor) ? lay.rows4 * lay.groups : n_groups;
    float* s = static_cast<float*>(sf);
    return fmt == kFmtE4M3 ? launch_sfc<kFmtE4M3, F32>(x, out, s, lay, n_groups, n_walk, stream)
                           : launch_sfc<kFmtE5M2, F32>(x, out, s, lay, n_groups, n_walk, stream);
}

}  // namespace

cudaError_t launch_per_token_cast(const void* x, void* out, void* sf, int64_t T, int64_t C,
                                  int fmt, unsigned sf_flags, cudaStream_t stream) {
    return launch<false>(x, out, sf, T, C, fmt, sf_flags, stream);
}

cudaError_t launch_per_token_cast_f32(const float* x, void* out, void* sf, int64_t T, int64_t C,
                                      int fmt, unsigned sf_flags, cudaStream_t stream) {
    return launch<true>(x, out, sf, T, C, fmt, sf_flags, stream);
}

}  // namespace tkq
