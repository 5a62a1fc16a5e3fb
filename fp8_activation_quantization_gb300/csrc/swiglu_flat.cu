// swiglu_flat.cu -- swiglu_forward_and_per_token_cast of a bf16 [T, 2H]
// gate|up matrix, optionally times a per-row routing weight and with the
// optional clamp (gate <= c, -c <= up <= c) whose changed values are counted
// ("DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限"
// (itsolotime.com) §3.3), as a flat stream: the second of the library's two
// kernels for this operation.  It computes the same values and codes as the
// TMA-ring kernel of row_cast.cu (the same packed steps of tkq_device.cuh, in
// the same order), so the two are bit-identical.  Measured on both, this one
// is faster without a routing weight at every size, and with one on launches
// up to a few hundred MB, where the ring's fill and drain cost more than its
// deeper queue of loads saves; the launcher picks (swiglu_flat_chosen).
//
// GB300 design: the output groups g = t * GH + j (GH = H / 128) are visited in
// order, a warp taking units of four (lane l: 16 consecutive channels of group
// 4u + l / 8, eight lanes per group, the absmax in three xor shuffles),
// grid-stride over persistent CTAs of 256 threads.  Each lane keeps its
// group's row t and block j and advances them by the fixed grid stride (one
// division at the start), reads its 32-byte runs of gate and up straight from
// global memory, and issues the loads of its next unit before the arithmetic
// of the current one.  Codes leave as one 16-byte store per lane; codes
// [T, H] and row-major scales [T, GH] are flat in g.  The column-major scale
// layouts own padding rows T <= t < round_up(T, 4) with zero scales, so the
// walk then covers round_up(T, 4) rows and groups past row T - 1 load nothing
// and store only those zeros.
#include <cuda_runtime.h>

#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Bound c, counter, and c in both halves of a bf16 pair when c is a bf16
// value (else 0: the clamp then runs in fp32).
struct FlatClamp {
    float value;
    unsigned long long* count;
    uint32_t c2;
};

// One lane's place in the walk: unit u, its group g, the group's row t and
// block j (0 <= j < GH).  next() moves to unit u + step, i.e. group g + 4 step,
// with the row and block advanced by (dt, dj) = divmod(4 step, GH) and one
// carry.
struct Walk {
    int64_t u, g, t;
    int j;
    int64_t dt;
    int dj, GH;

    __device__ __forceinline__ Walk(int64_t u0, int sub, int64_t step, int gh) : GH(gh) {
        u = u0;
        g = u0 * 4 + sub;
        t = g / gh;
        j = static_cast<int>(g - t * gh);
        dt = (step * 4) / gh;
        dj = static_cast<int>(step * 4 - dt * gh);
    }
    __device__ __forceinline__ void next(int64_t step) {
        u += step;
        g += step * 4;
        t += dt;
        j += dj;
        if (j >= GH) {
            j -= GH;
            ++t;
        }
    }
};

// A lane's 16 gate and 16 up values as raw 16-byte vectors, and its row's
// routing weight.
template <bool WEIGHTED>
struct Slice {
    uint4 g[2], u[2];
    float w;

    __device__ __forceinline__ void clear() {
        g[0] = g[1] = u[0] = u[1] = make_uint4(0, 0, 0, 0);
        w = 1.0f;
    }
    // x: [T, 2H] bf16, H / 4 16-byte vectors per row; the lane's channels are
    // 128 j + 16 k .. + 16 of row t, gate at column c and up at H + c
    __device__ __forceinline__ void load(const uint4* x, const float* wt, int64_t t, int j, int k,
                                         int64_t H) {
        const uint4* pg = x + t * (H / 4) + j * 16 + k * 2;
        const uint4* pu = pg + H / 8;
        g[0] = ld_stream(pg);
        g[1] = ld_stream(pg + 1);
        u[0] = ld_stream(pu);
        u[1] = ld_stream(pu + 1);
        if constexpr (WEIGHTED) w = ld_ro(wt + t);
    }
};

// The clamp of an instance: none, on packed bf16 pairs (the bound is a bf16
// value), or in fp32.
enum ClampKind { kNoClamp, kClampBf16, kClampF32 };

// n_groups = T * GH groups hold data; n_walk >= n_groups are visited.
template <int FMT, bool WEIGHTED, int CLAMP, bool SFX>
__global__ void __launch_bounds__(kThreads, CLAMP == kClampF32 ? 3 : 4)
    swiglu_flat_kernel(const uint4* __restrict__ x, const float* __restrict__ w,
                       uint4* __restrict__ out, float* __restrict__ sf, SfLayout lay, int64_t H,
                       int64_t n_groups, int64_t n_walk, FlatClamp clamp, int prefetch_units) {
    grid_dependency_launch();
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 3;   // group within the unit
    const int k = lane & 7;      // lane within the group
    const int GH = static_cast<int>(H / 128);
    const int64_t units = (n_walk + 3) / 4;
    const int64_t step = static_cast<int64_t>(gridDim.x) * kWarps;

    Walk cur(static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5), sub, step, GH);
    {
        // the gate and up runs of the warp's first prefetch_units units go to
        // L2 while the grid before this one drains; then wait until it is done
        Walk pre = cur;
        for (int p = 0; p < prefetch_units; ++p) {
            if (k == 0 && pre.u < units && pre.g < n_groups) {
                const uint4* pg = x + pre.t * (H / 4) + pre.j * 16;
                prefetch_l2(pg, 256);
                prefetch_l2(pg + H / 8, 256);
            }
            pre.next(step);
        }
    }
    grid_dependency_wait();
    Slice<WEIGHTED> in;
    in.clear();
    if (cur.u < units && cur.g < n_groups) in.load(x, w, cur.t, cur.j, k, H);
    uint32_t n_clamped = 0;
    while (cur.u < units) {
        const int64_t g = cur.g, t = cur.t;
        const int j = cur.j;
        const bool live = g < n_groups;
        uint4 gq[2] = {in.g[0], in.g[1]}, uq[2] = {in.u[0], in.u[1]};
        const float wt = in.w;
        // the next unit's loads go out before this unit's arithmetic
        cur.next(step);
        if (cur.u < units && cur.g < n_groups) in.load(x, w, cur.t, cur.j, k, H);

        float gv[16], uv[16];
        uint32_t n = 0;
        if constexpr (CLAMP == kClampBf16) {
            // clamp and count on the packed pairs
            uint32_t n2 = 0;  // at most 16 a half
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                clamp_pairs_bf16(gq[h].x, uq[h].x, clamp.c2, n2);
                clamp_pairs_bf16(gq[h].y, uq[h].y, clamp.c2, n2);
                clamp_pairs_bf16(gq[h].z, uq[h].z, clamp.c2, n2);
                clamp_pairs_bf16(gq[h].w, uq[h].w, clamp.c2, n2);
            }
            n = clamped_total(n2);
        }
        unpack8(gq[0], gv);
        unpack8(gq[1], gv + 8);
        unpack8(uq[0], uv);
        unpack8(uq[1], uv + 8);
        if constexpr (CLAMP == kClampF32) {
            const float c = clamp.value;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                n += (gv[e] > c) + (fabsf(uv[e]) > c);
                gv[e] = fminf(gv[e], c);
                uv[e] = fmaxf(fminf(uv[e], c), -c);
            }
        }
        if constexpr (CLAMP != kNoClamp) {
            if (live) n_clamped += n;
        }

        float v[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
            float2 y = swiglu2(make_float2(gv[e], gv[e + 1]), make_float2(uv[e], uv[e + 1]));
            if constexpr (WEIGHTED) y = mul2(y, make_float2(wt, wt));
            v[e] = y.x;
            v[e + 1] = y.y;
        }

        float m = fmaxf(absmax8(v), absmax8(v + 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        float sc, inv;
        group_scale<FMT>(m, sc, inv);
        if constexpr (SFX) {
            if (lay.flags & (kSfRoundPow2 | kSfPacked)) pow2_scale(sc, inv);  // inv = 2^-k exactly
        }
        if (live) {
            const uint2 lo = quantize8_mul<FMT>(v, inv), hi = quantize8_mul<FMT>(v + 8, inv);
            st_stream(out + g * 8 + k, make_uint4(lo.x, lo.y, hi.x, hi.y));
        }
        if (k == 0) {
            if constexpr (SFX) {
                store_scale(sf, lay, t, live, j, sc);
            } else {
                if (live) st_stream(sf + g, sc);
            }
        }
    }
    if constexpr (CLAMP != kNoClamp) {
        // one atomic per warp, and none when nothing was clamped
        unsigned long long c = n_clamped;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0 && c && clamp.count) atomic_add_count(clamp.count, c);
    }
}

template <int FMT, bool WEIGHTED, int CLAMP, bool SFX>
cudaError_t launch_layout(const void* x, const float* w, void* out, float* sf,
                          const SfLayout& lay, int64_t H, int64_t n_groups, int64_t n_walk,
                          FlatClamp clamp, cudaStream_t stream) {
    auto* k = &swiglu_flat_kernel<FMT, WEIGHTED, CLAMP, SFX>;
    const int64_t units = (n_walk + 3) / 4;
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, 0,
                                     (units + kWarps - 1) / kWarps);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kThreads, 0, stream, true, static_cast<const uint4*>(x), w,
                      static_cast<uint4*>(out), sf, lay, H, n_groups, n_walk, clamp,
                      prologue_prefetch_units(n_groups * 512));
}

template <int FMT, bool WEIGHTED, int CLAMP>
cudaError_t launch_flags(const void* x, const float* w, void* out, float* sf,
                         const SfLayout& lay, int64_t H, int64_t n_groups, int64_t n_walk,
                         FlatClamp clamp, cudaStream_t stream) {
    return lay.flags
               ? launch_layout<FMT, WEIGHTED, CLAMP, true>(x, w, out, sf, lay, H, n_groups, n_walk,
                                                           clamp, stream)
               : launch_layout<FMT, WEIGHTED, CLAMP, false>(x, w, out, sf, lay, H, n_groups,
                                                            n_walk, clamp, stream);
}

template <int FMT>
cudaError_t launch_fmt(const void* x, const float* w, void* out, float* sf, const SfLayout& lay,
                       int64_t H, int64_t n_groups, int64_t n_walk, const FlatClamp* clamp,
                       cudaStream_t stream) {
    const FlatClamp c = clamp ? *clamp : FlatClamp{0.0f, nullptr, 0u};
    if (clamp && c.c2)
        return w ? launch_flags<FMT, true, kClampBf16>(x, w, out, sf, lay, H, n_groups, n_walk, c,
                                                       stream)
                 : launch_flags<FMT, false, kClampBf16>(x, w, out, sf, lay, H, n_groups, n_walk,
                                                        c, stream);
    if (clamp)
        return w ? launch_flags<FMT, true, kClampF32>(x, w, out, sf, lay, H, n_groups, n_walk, c,
                                                      stream)
                 : launch_flags<FMT, false, kClampF32>(x, w, out, sf, lay, H, n_groups, n_walk, c,
                                                       stream);
    return w ? launch_flags<FMT, true, kNoClamp>(x, w, out, sf, lay, H, n_groups, n_walk, c,
                                                 stream)
             : launch_flags<FMT, false, kNoClamp>(x, w, out, sf, lay, H, n_groups, n_walk, c,
                                                  stream);
}

}  // namespace

cudaError_t launch_swiglu_cast_flat(const void* x, const float* w, void* out, void* sf, int64_t T,
                                    int64_t H, int fmt, unsigned sf_flags, const float* clamp,
                                    unsigned long long* clamp_count, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int64_t GH = H / 128;
    SfLayout lay;
    lay.flags = sf_flags;
    lay.groups = static_cast<int>(GH);
    lay.words = (lay.groups + 3) / 4;
    lay.rows4 = (T + 3) / 4 * 4;
    const int64_t n_groups = T * GH;
    const int64_t n_walk = (sf_flags & kSfColMajor) ? lay.rows4 * GH : n_groups;
    FlatClamp c{0.0f, clamp_count, 0u};
    if (clamp) {
        c.value = *clamp;
        c.c2 = bf16x2_bound(*clamp);
    }
    float* s = static_cast<float*>(sf);
    const FlatClamp* cp = clamp ? &c : nullptr;
    if (fmt == kFmtE4M3)
        return launch_fmt<kFmtE4M3>(x, w, out, s, lay, H, n_groups, n_walk, cp, stream);
    return launch_fmt<kFmtE5M2>(x, w, out, s, lay, H, n_groups, n_walk, cp, stream);
}

}  // namespace tkq
