// row_cast.cu -- the per-token-group FP8 casts of SwiGLU values with
// row-major outputs (the plain per_token_cast is token_cast.cu):
//   * swiglu_forward_and_per_token_cast of a bf16 [T, 2H] gate|up matrix,
//     optionally times a per-row routing weight and with the optional clamp
//     (gate <= c, -c <= up <= c) whose changed values are counted
//     ("DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限"
//     (itsolotime.com) §3.3);
//   * swiglu_backward_and_per_token_cast ("TileKernels 与 DeepGEMM 的分界线"
//     (chatdocs.ruinique.com) §2 and §6 step 13): the gradients [dg | du] of
//     the same SwiGLU from the upstream gradient dy, cast per token.
// Per 1x128 group: absmax -> scale s = max(amax, 1e-4) / fmt_max -> FP8 codes.
//
// GB300 design: persistent CTAs (3 per SM) stream "chunks" of 32 rows x one
// 128-channel block.  Warp 8 is the producer: one lane loads each chunk with
// one 2-D TMA box per operand (32 x 128 bf16 = 8 KB: gate and up; or gate, up
// and dy) into a shared ring of 64-72 KB (4 SwiGLU, 3 backward chunks in
// flight per CTA).  Rows past T are
// zero-filled by the TMA unit and never stored, so ragged T needs no special
// path.  Warps 0..7 are
// consumers: warp w owns rows 4w..4w+3 of the chunk, eight lanes per row
// (lane j holds elements [8j, 8j+8) and [64+8j, 64+8j+8), read as two
// conflict-free 16-byte shared loads per operand), the group absmax is three
// xor shuffles, and codes leave as 8-byte stores (eight lanes write one
// 64-byte run).  The codes are those of y * fl(1 / s), as the page's kernel
// computes them.
// Elementwise fp32 steps run on packed pairs (tkq_device.cuh); a clamp bound
// that is a bf16 value is applied, and its changes counted, on the packed bf16
// input pairs before they are widened (same values, half the instructions).
// Every mbarrier wait is bounded (tkq_async.cuh).
#include <cuda.h>

#include "tkq_async.cuh"
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRows = 32;                 // rows per chunk (4 per consumer warp)
constexpr int kBoxBytes = kRows * 256;    // one 32 x 128 bf16 box

// The clamp modes come in two kinds fixed at compile time: the bound is a bf16
// value (the clamp runs on the packed bf16 inputs) or not (fp32 clamp); a
// choice made inside the loop costs the latency-bound kernels measurably.
enum Mode {
    kSwiglu, kSwigluWeighted, kSwigluClamp, kSwigluWeightedClamp, kSwigluClampF32,
    kSwigluWeightedClampF32, kBackward, kBackwardWeighted
};

template <int MODE>
struct ModeTraits {
    static constexpr bool kBwd = MODE == kBackward || MODE == kBackwardWeighted;
    static constexpr bool kClampBf16 = MODE == kSwigluClamp || MODE == kSwigluWeightedClamp;
    static constexpr bool kClamp =
        kClampBf16 || MODE == kSwigluClampF32 || MODE == kSwigluWeightedClampF32;
    static constexpr bool kWeighted = MODE == kSwigluWeighted || MODE == kSwigluWeightedClamp ||
                                      MODE == kSwigluWeightedClampF32 ||
                                      MODE == kBackwardWeighted;
    static constexpr int kOperands = kBwd ? 3 : 2;  // boxes per chunk
    static constexpr int kRowBytes = 256;            // one box row in shared memory
    static constexpr int kStageBytes = kOperands * kRows * kRowBytes;
    static constexpr int kRingBytes = kBwd ? 3 * kStageBytes : 65536;
    static constexpr int kStages = kRingBytes / kStageBytes;
};

template <int MODE>
struct alignas(1024) RowSmem {
    uint8_t stage[ModeTraits<MODE>::kStages][ModeTraits<MODE>::kStageBytes];
    uint64_t full[ModeTraits<MODE>::kStages];
    uint64_t empty[ModeTraits<MODE>::kStages];
    int abort;
};

// absmax of one 1x128 group held by eight lanes (16 values each), its scale,
// and the codes (of the products by fl32(1/s)) and scale stored for a live
// row.  SFX: the launch uses scale-layout options (power-of-two scales, packed
// UE8M0, column-major); without it the scales are row-major fp32 at sfp.
template <int FMT, bool SFX>
__device__ __forceinline__ void emit_group(const float* v, bool live, uint2* o, float* sfp,
                                           int j, void* sf, const SfLayout& lay, int64_t row,
                                           int gj) {
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
        st_stream(o + j, quantize8_mul<FMT>(v, inv));
        st_stream(o + 8 + j, quantize8_mul<FMT>(v + 8, inv));
    }
    if (j == 0) {
        if constexpr (SFX) {
            store_scale(sf, lay, row, live, gj, sc);
        } else {
            if (live) st_stream(sfp, sc);
        }
    }
}

// 16 bf16 of one operand for lane j: elements [8j, 8j+8) and [64+8j, 64+8j+8).
__device__ __forceinline__ void load16(const uint8_t* p, float* v) {
    unpack8(*reinterpret_cast<const uint4*>(p), v);
    unpack8(*reinterpret_cast<const uint4*>(p + 128), v + 8);
}

// The SwiGLU clamp of one launch: bound c (> 0), the counter that the number
// of changed input values is added to (may be null), and c in both halves of
// a bf16 pair when c is a bf16 value (else 0: the clamp then runs in fp32).
struct Clamp {
    float value;
    unsigned long long* count;
    uint32_t c2;
};

// tmap: x [T, C] (plain) or [T, 2H] (gate | up); tmap_dy: dy [T, H] (backward
// only).  C_out: channels per output operand (C or H).
template <int FMT, int MODE, bool SFX>
__global__ void __launch_bounds__(kThreads, 3)
    row_cast_kernel(const __grid_constant__ CUtensorMap tmap,
                    const __grid_constant__ CUtensorMap tmap_dy, const float* __restrict__ w,
                    uint2* __restrict__ out, float* __restrict__ sf, SfLayout lay, int64_t T,
                    int C_out, Clamp clamp, unsigned int* __restrict__ status) {
    using MT = ModeTraits<MODE>;
    extern __shared__ uint8_t smem_raw[];
    RowSmem<MODE>& sm = *reinterpret_cast<RowSmem<MODE>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t CB = static_cast<uint32_t>(C_out) >> 7;
    const uint32_t RB = static_cast<uint32_t>((T + kRows - 1) / kRows);

    if (threadIdx.x == 0) {
        for (int s = 0; s < MT::kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_launch();
    if constexpr (!MT::kBwd) {
        // the gate and up boxes of the CTA's first kStages row blocks go to
        // L2 while the grid before this one drains (the backward cast is
        // launched without that overlap: with it and this prefetch of its
        // three operands it measured 1.7 % slower, with the prefetch alone
        // 0.15 % slower)
        if (warp == kConsumerWarps && lane == 0) {
            int k = 0;
            for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < RB && k < MT::kStages;
                 tw.next(), ++k) {
                const int y0 = static_cast<int>(tw.row * kRows);
                const int x0 = static_cast<int>(tw.col * 128);
                tma_prefetch_2d(&tmap, x0, y0);
                tma_prefetch_2d(&tmap, C_out + x0, y0);
            }
        }
    }
    grid_dependency_wait();  // the previous grid on the stream is done

    // ------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            uint32_t issued = 0;
            RingPos<MT::kStages> pos;
            for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < RB; tw.next(), ++issued) {
                if (!mbar_wait_bounded(&sm.empty[pos.stage], pos.phase ^ 1u, &sm.abort, status)) {
                    *static_cast<volatile int*>(&sm.abort) = 1;
                    break;
                }
                const int y0 = static_cast<int>(tw.row * kRows);
                const int x0 = static_cast<int>(tw.col * 128);
                uint8_t* dst = sm.stage[pos.stage];
                uint64_t* full = &sm.full[pos.stage];
                mbar_arrive_expect_tx(full, MT::kStageBytes);
                tma_load_2d(dst, &tmap, x0, y0, full);
                tma_load_2d(dst + kBoxBytes, &tmap, C_out + x0, y0, full);
                if constexpr (MT::kOperands == 3)
                    tma_load_2d(dst + 2 * kBoxBytes, &tmap_dy, x0, y0, full);
                pos.advance();
            }
            // every copy this CTA issued must have landed before it may exit
            const uint32_t first = issued > MT::kStages ? issued - MT::kStages : 0;
            for (uint32_t k = first; k < issued; ++k)
                mbar_wait_bounded(&sm.full[k % MT::kStages], (k / MT::kStages) & 1u, nullptr,
                                  status);
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int sub = lane >> 3;          // row within the warp's four
    const int j = lane & 7;             // position within the group
    const int r = warp * 4 + sub;       // row within the chunk
    // output row pitch (elements) and scales per output row
    const int64_t out_ld = MT::kBwd ? 2 * static_cast<int64_t>(C_out) : C_out;
    const uint32_t sf_ld = MT::kBwd ? 2 * CB : CB;
    uint64_t n_clamped = 0;
    RingPos<MT::kStages> pos;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < RB; tw.next(), pos.advance()) {
        const int s = static_cast<int>(pos.stage);
        const int cb = static_cast<int>(tw.col);
        const int64_t row = static_cast<int64_t>(tw.row) * kRows + r;
        const bool live = row < T;

        float wt = 1.0f;
        if constexpr (MT::kWeighted) {
            if (live) wt = ld_ro(w + row);
        }

        // the warp leaves as a whole if any lane's wait gave up, so that no
        // lane is left behind at a shuffle
        const bool ok = mbar_wait_bounded(&sm.full[s], pos.phase, &sm.abort, status);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) *static_cast<volatile int*>(&sm.abort) = 1;  // stop the producer
            break;
        }
        const uint8_t* p = sm.stage[s] + r * MT::kRowBytes + j * (MT::kRowBytes / 16);
        uint2* o = out + (row * out_ld + cb * 128) / 8;
        float* sfp = sf + row * sf_ld + cb;
        if constexpr (!MT::kBwd) {
            float g[16], u[16], v[16];
            if constexpr (MT::kClamp) {
                uint4 gq[2] = {*reinterpret_cast<const uint4*>(p),
                               *reinterpret_cast<const uint4*>(p + 128)};
                uint4 uq[2] = {*reinterpret_cast<const uint4*>(p + kBoxBytes),
                               *reinterpret_cast<const uint4*>(p + kBoxBytes + 128)};
                uint32_t n = 0;
                if constexpr (MT::kClampBf16) {
                    // c is a bf16 value: clamp and count on the packed pairs
                    const uint32_t c2 = clamp.c2;
                    uint32_t n2 = 0;  // at most 16 a half
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        clamp_pairs_bf16(gq[h].x, uq[h].x, c2, n2);
                        clamp_pairs_bf16(gq[h].y, uq[h].y, c2, n2);
                        clamp_pairs_bf16(gq[h].z, uq[h].z, c2, n2);
                        clamp_pairs_bf16(gq[h].w, uq[h].w, c2, n2);
                    }
                    n = clamped_total(n2);
                    unpack8(gq[0], g);
                    unpack8(gq[1], g + 8);
                    unpack8(uq[0], u);
                    unpack8(uq[1], u + 8);
                } else {
                    unpack8(gq[0], g);
                    unpack8(gq[1], g + 8);
                    unpack8(uq[0], u);
                    unpack8(uq[1], u + 8);
                    const float c = clamp.value;
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        n += (g[k] > c) + (fabsf(u[k]) > c);
                        g[k] = fminf(g[k], c);
                        u[k] = fmaxf(fminf(u[k], c), -c);
                    }
                }
                if (live) n_clamped += n;
            } else {
                load16(p, g);
                load16(p + kBoxBytes, u);
            }
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float2 y = swiglu2(make_float2(g[k], g[k + 1]), make_float2(u[k], u[k + 1]));
                if constexpr (MT::kWeighted) y = mul2(y, make_float2(wt, wt));
                v[k] = y.x;
                v[k + 1] = y.y;
            }
            emit_group<FMT, SFX>(v, live, o, sfp, j, sf, lay, row, cb);
        } else {
            float g[16], u[16], d[16], dg[16], du[16];
            load16(p, g);
            load16(p + kBoxBytes, u);
            load16(p + 2 * kBoxBytes, d);
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float2 a, b;
                swiglu_grad2(make_float2(g[k], g[k + 1]), make_float2(u[k], u[k + 1]),
                             make_float2(d[k], d[k + 1]), a, b);
                if constexpr (MT::kWeighted) {
                    a = mul2(a, make_float2(wt, wt));
                    b = mul2(b, make_float2(wt, wt));
                }
                dg[k] = a.x;
                dg[k + 1] = a.y;
                du[k] = b.x;
                du[k + 1] = b.y;
            }
            emit_group<FMT, SFX>(dg, live, o, sfp, j, sf, lay, row, cb);
            emit_group<FMT, SFX>(du, live, o + C_out / 8, sfp + CB, j, sf, lay, row,
                                          static_cast<int>(CB) + cb);
        }
        // Release the stage only now: the stores above consume every value
        // read from it, so the shared loads have completed before the arrive
        // is issued (an arrive placed right after the loads can retire while
        // they are still pending, and the refill then overwrites their data).
        // The proxy fence orders these generic-proxy reads before the refill,
        // which the TMA unit performs in the async proxy.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    if constexpr (MT::kClamp) {
        // one atomic per warp, and none when nothing was clamped
        unsigned long long t = n_clamped;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0 && t && clamp.count) atomic_add_count(clamp.count, t);
    }
}

template <int FMT, int MODE, bool SFX>
cudaError_t launch_mode(const CUtensorMap& map, const CUtensorMap& map_dy, const float* w,
                        void* out, float* sf, const SfLayout& lay, int64_t T, int64_t C_out,
                        Clamp clamp, cudaStream_t stream) {
    auto* k = &row_cast_kernel<FMT, MODE, SFX>;
    const size_t smem = sizeof(RowSmem<MODE>) + 1024;
    const int64_t n_chunks = ((T + kRows - 1) / kRows) * (C_out / 128);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, smem, n_chunks);
    if (const cudaError_t e = upload_checks(stream)) return e;
    // the backward cast measured slower with programmatic dependent launch
    return launch_pdl(k, grid, kThreads, smem, stream, !ModeTraits<MODE>::kBwd, map, map_dy, w,
                      static_cast<uint2*>(out), sf, lay, T, static_cast<int>(C_out), clamp,
                      device_status_word());
}

template <int FMT, int MODE>
cudaError_t launch(const void* x, const void* dy, const float* w, void* out, void* sf,
                   int64_t T, int64_t C_out, unsigned sf_flags, Clamp clamp,
                   cudaStream_t stream) {
    using MT = ModeTraits<MODE>;
    // x as a bf16 [T, 2H] matrix (gate | up)
    CUtensorMap map, map_dy;
    if (!encode_bf16_2d(&map, x, 2 * C_out, T, 128, kRows)) return cudaErrorInvalidValue;
    if constexpr (MT::kBwd) {
        if (!encode_bf16_2d(&map_dy, dy, C_out, T, 128, kRows)) return cudaErrorInvalidValue;
    } else {
        map_dy = map;  // unused
    }
    SfLayout lay;
    lay.flags = sf_flags;
    lay.groups = static_cast<int>((MT::kBwd ? 2 : 1) * C_out / 128);
    lay.words = (lay.groups + 3) / 4;
    lay.rows4 = (T + 3) / 4 * 4;
    float* sff = static_cast<float*>(sf);
    return sf_flags
               ? launch_mode<FMT, MODE, true>(map, map_dy, w, out, sff, lay, T, C_out, clamp,
                                              stream)
               : launch_mode<FMT, MODE, false>(map, map_dy, w, out, sff, lay, T, C_out, clamp,
                                               stream);
}

template <int MODE>
cudaError_t launch_fmt(int fmt, const void* x, const void* dy, const float* w, void* out,
                       void* sf, int64_t T, int64_t C_out, unsigned sf_flags,
                       cudaStream_t stream, Clamp clamp = Clamp{0.0f, nullptr, 0u}) {
    if (T == 0) return cudaSuccess;
    return fmt == kFmtE4M3
               ? launch<kFmtE4M3, MODE>(x, dy, w, out, sf, T, C_out, sf_flags, clamp, stream)
               : launch<kFmtE5M2, MODE>(x, dy, w, out, sf, T, C_out, sf_flags, clamp, stream);
}

}  // namespace

cudaError_t launch_swiglu_cast(const void* x, const float* w, void* out, void* sf, int64_t T,
                               int64_t H, int fmt, unsigned sf_flags, const float* clamp,
                               unsigned long long* clamp_count, cudaStream_t stream) {
    if (swiglu_flat_chosen(T, H, w != nullptr))
        return launch_swiglu_cast_flat(x, w, out, sf, T, H, fmt, sf_flags, clamp, clamp_count,
                                       stream);
    if (clamp) {
        const Clamp c{*clamp, clamp_count, bf16x2_bound(*clamp)};
        if (c.c2)
            return w ? launch_fmt<kSwigluWeightedClamp>(fmt, x, nullptr, w, out, sf, T, H,
                                                        sf_flags, stream, c)
                     : launch_fmt<kSwigluClamp>(fmt, x, nullptr, w, out, sf, T, H, sf_flags,
                                                stream, c);
        return w ? launch_fmt<kSwigluWeightedClampF32>(fmt, x, nullptr, w, out, sf, T, H,
                                                       sf_flags, stream, c)
                 : launch_fmt<kSwigluClampF32>(fmt, x, nullptr, w, out, sf, T, H, sf_flags,
                                               stream, c);
    }
    return w ? launch_fmt<kSwigluWeighted>(fmt, x, nullptr, w, out, sf, T, H, sf_flags, stream)
             : launch_fmt<kSwiglu>(fmt, x, nullptr, w, out, sf, T, H, sf_flags, stream);
}

cudaError_t launch_swiglu_backward_cast(const void* x, const void* dy, const float* w, void* out,
                                        void* sf, int64_t T, int64_t H, int fmt,
                                        unsigned sf_flags, cudaStream_t stream) {
    return w ? launch_fmt<kBackwardWeighted>(fmt, x, dy, w, out, sf, T, H, sf_flags, stream)
             : launch_fmt<kBackward>(fmt, x, dy, w, out, sf, T, H, sf_flags, stream);
}

}  // namespace tkq
