// swiglu_cast_t.cu -- SwiGLU + per-token FP8 cast + transposed (token-axis)
// FP8 cast in one pass over HBM.
//
// The operation is the SwiGLU + FP8 + transpose triple fusion of the quant/
// section of "刚刚！DeepSeek开源高性能GPU算子库TileKernels" (info.datadowell.com),
// i.e. swiglu_forward_and_per_token_cast ("DeepSeek开源TileKernels：用Python写的
// GPU算子逼近硬件性能上限" (itsolotime.com) §3.3) plus a per_channel_cast of the
// transposed y ("TileKernels 与 DeepGEMM 的分界线" (chatdocs.ruinique.com) §2,
// "per_channel_cast (+transpose / fused)").  Both outputs are quantized from the
// same fp32 y.  With a clamp the gate is clamped to <= c and the up projection to
// [-c, c] before the SwiGLU, and the number of changed values is added to a
// counter (one atomic per warp), as in §3.3 of the second page; a bound that is
// a bf16 value is applied on the packed bf16 input pairs before widening.
//
// GB300 design: one persistent CTA per SM walks 128-token x 128-channel tiles
// of y.  Warp 16 is the producer: one lane streams the gate and up tiles of the
// CTA's upcoming tiles (2 x 32 KB, one 2-D TMA box each) into a 3-stage shared
// ring, so up to 192 KB per SM are in flight while the consumers compute.
// Warps 0..15 are consumers; warp w owns tokens 8w..8w+7 of the tile and lane
// l owns channels 4l..4l+3, i.e. an 8 x 4 block of y per thread, read from the
// ring with conflict-free 8-byte shared loads (a warp reads one 256-byte row).
// Once its row codes are stored (they consume every value the warp read) the
// warp releases the stage to the producer; the column work runs from registers.
//   * Row groups (1 x 128 channels = one warp row): a butterfly absmax across
//     the 32 lanes that halves the live values at each xor step (9 shuffles
//     for 8 rows); lanes 4r..4r+3 then hold row r, one of them forms the
//     row's scale and publishes its reciprocal through shared memory.  Codes
//     leave as 4-byte stores, one 128-byte run per warp store instruction.
//   * Column groups (128 tokens x 1 channel): per-thread maxima over 8 tokens,
//     a 16 x 128 shared table reduced by 128 threads, scales broadcast through
//     shared memory.  Codes are transposed through a 16 KB byte tile
//     [channel][token] whose 8-byte token units are XOR-swizzled by
//     (channel / 4) & 15 so that each half-warp's 8-byte writes cover 32
//     distinct banks; the tile leaves as 16-byte stores, eight lanes per
//     128-byte run of out_t.  (The TileKernels transpose of the same page, §6,
//     rotates a column index by the thread id and pads the tile for the same
//     purpose.)
// All mbarrier waits are bounded (tkq_async.cuh); on a timeout the consumers
// agree through a barrier-with-OR and leave together, and the producer waits
// (bounded) for its issued copies before it returns.
#include <cuda.h>

#include "tkq_async.cuh"
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kStages = 3;
// Tiles whose boxes the producer sends to L2 before the dependency wait: the
// ring's first fill and the tile after it.  Measured back to back on
// [131072, 4096] (us; no prefetch / 1 / 2 / 4 tiles): 233.2 / 231.7 / 235.1 /
// 232.7 without options, 241.5 / 240.6 / 237.2 / 238.2 with the clamp c = 4,
// 232.0 / 230.1 / 228.3 / 229.1 with UE8M0 column-major scales.  This kernel's
// speed moves with small changes of its code, so no depth wins every
// instance; four is the one that beats no prefetch in all three.
constexpr int kPrefetchTiles = 4;
constexpr int kTileBytes = 128 * 128 * 2;    // one bf16 128 x 128 box
constexpr int kStageBytes = 2 * kTileBytes;  // gate + up
constexpr int kBarConsumers = 1;             // named barrier of the consumer warps

struct alignas(1024) SharedStorage {
    uint8_t stage[kStages][kStageBytes];
    uint2 codes[128][16];                   // [channel][8-token unit], swizzled
    float colmax[kConsumerWarps][128];
    float cinv[128];
    float rowinv[kConsumerWarps][8];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort;
};

// Scale layouts of an instance (kSfc* of tkq_device.cuh): none (fp32
// row-major, as documented for tkq_swiglu_cast_t), the layouts a TMA-fed FP8
// GEMM reads fixed at compile time (UE8M0 packed column-major, fp32
// column-major), or any TKQ_SF_* combination read from the launch's flags at
// run time.  The fixed instances exist because the run-time one is measurably
// slower in this latency-bound body (244.7 against 232.0 us for UE8M0
// column-major on the swiglu_t workload, back to back; the flag-free instance
// takes 233.4 us).

// The clamp of an instance: none, on packed bf16 pairs (the bound is a bf16
// value), or in fp32.  Fixed at compile time for the same reason as the
// layouts: with the choice made inside the loop the clamped step took 248.0 us,
// with the bf16 clamp fixed 241.4 us (the unclamped one 233.4 us).
enum ClampKind { kNoClamp, kClampBf16, kClampF32 };

// SFC: the instance's scale layout (above) for the row scales (lay_r,
// [T, H/128]) and the column scales (lay_c, [H, T/128]).
template <int FMT, bool WEIGHTED, int CLAMP, unsigned SFC>
__global__ void __launch_bounds__(kThreads, 1)
    swiglu_cast_t_kernel(const __grid_constant__ CUtensorMap tmap, const float* __restrict__ w,
                         uint8_t* __restrict__ out, float* __restrict__ sf,
                         uint4* __restrict__ out_t, float* __restrict__ sf_t, int64_t T, int H,
                         SfLayout lay_r, SfLayout lay_c, float clamp, uint32_t clamp2,
                         unsigned long long* __restrict__ clamp_count,
                         unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    SharedStorage& sm = *reinterpret_cast<SharedStorage*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t CB = static_cast<uint32_t>(H) >> 7;
    const uint32_t TB = static_cast<uint32_t>(T >> 7);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_launch();
    if (warp == kConsumerWarps && lane == 0) {
        // the gate and up boxes of the CTA's first kPrefetchTiles tiles go to
        // L2 while the grid before this one drains
        int k = 0;
        for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB && k < kPrefetchTiles;
             tw.next(), ++k) {
            tma_prefetch_2d(&tmap, static_cast<int>(tw.col * 128), static_cast<int>(tw.row * 128));
            tma_prefetch_2d(&tmap, static_cast<int>(H + tw.col * 128),
                            static_cast<int>(tw.row * 128));
        }
    }
    grid_dependency_wait();  // the previous grid on the stream is done

    // ------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            uint32_t issued = 0;
            RingPos<kStages> pos;
            for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB; tw.next(), ++issued) {
                if (!mbar_wait_bounded(&sm.empty[pos.stage], pos.phase ^ 1u, &sm.abort, status)) {
                    *static_cast<volatile int*>(&sm.abort) = 1;
                    break;
                }
                const int y0 = static_cast<int>(tw.row * 128);
                const int x0 = static_cast<int>(tw.col * 128);
                uint64_t* full = &sm.full[pos.stage];
                mbar_arrive_expect_tx(full, kStageBytes);
                tma_load_2d(sm.stage[pos.stage], &tmap, x0, y0, full);
                tma_load_2d(sm.stage[pos.stage] + kTileBytes, &tmap, H + x0, y0, full);
                pos.advance();
            }
            // every copy this CTA issued must have landed before it may exit
            const uint32_t first = issued > kStages ? issued - kStages : 0;
            for (uint32_t k = first; k < issued; ++k)
                mbar_wait_bounded(&sm.full[k % kStages], (k / kStages) & 1u, nullptr, status);
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int ct = threadIdx.x;  // 0 .. kConsumers-1
    constexpr bool SFX = SFC != kSfcNone;
    if constexpr (SFX && SFC != kSfcRuntime) {
        // a fixed layout: its flags are compile-time constants from here on
        lay_r.flags = SFC;
        lay_c.flags = SFC;
    }
    uint64_t n_clamped = 0;
    // routing weights of this thread's 8 tokens, loaded one tile ahead so that
    // their latency overlaps the previous tile's work
    [[maybe_unused]] float wt_next[8];
    if constexpr (WEIGHTED) {
        const TileWalk first(blockIdx.x, gridDim.x, CB);
        if (first.row < TB) {
            const int64_t r0 = static_cast<int64_t>(first.row) * 128 + warp * 8;
#pragma unroll
            for (int r = 0; r < 8; ++r) wt_next[r] = ld_ro(w + r0 + r);
        }
    }
    RingPos<kStages> pos;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB; tw.next(), pos.advance()) {
        const int s = static_cast<int>(pos.stage);
        const uint32_t tb = tw.row;
        const int cb = static_cast<int>(tw.col);
        const int64_t t0 = static_cast<int64_t>(tb) * 128;
        const int c0 = cb * 128;
        const int64_t row0 = t0 + warp * 8;

        float wt[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) wt[r] = 1.0f;
        if constexpr (WEIGHTED) {
#pragma unroll
            for (int r = 0; r < 8; ++r) wt[r] = wt_next[r];
            TileWalk nx = tw;
            nx.next();
            if (nx.row < TB) {
                const int64_t r0 = static_cast<int64_t>(nx.row) * 128 + warp * 8;
#pragma unroll
                for (int r = 0; r < 8; ++r) wt_next[r] = ld_ro(w + r0 + r);
            }
        }

        const bool ok = mbar_wait_bounded(&sm.full[s], pos.phase, &sm.abort, status);

        // ---- y = silu(g) * u [* w] for this thread's 8 x 4 block ----------
        float y[8][4];
        {
            // clamp counts of this tile: per half of the packed-bf16 clamp, and
            // of the fp32 clamp
            [[maybe_unused]] __nv_bfloat162 n2 = __float2bfloat162_rn(0.0f);
            [[maybe_unused]] uint32_t n1 = 0;
            const uint8_t* g_base = sm.stage[s] + warp * 8 * 256 + lane * 8;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                uint2 gq = make_uint2(0, 0), uq = make_uint2(0, 0);
                if (ok) {
                    gq = *reinterpret_cast<const uint2*>(g_base + r * 256);
                    uq = *reinterpret_cast<const uint2*>(g_base + kTileBytes + r * 256);
                }
                float gv[4], uv[4];
                if constexpr (CLAMP == kClampBf16) {
                    // c is a bf16 value: clamp and count on the packed pairs
                    // (at most 4 per half and row: 32 per tile)
                    clamp_pairs_bf16(gq.x, uq.x, clamp2, n2);
                    clamp_pairs_bf16(gq.y, uq.y, clamp2, n2);
                    unpack4(gq, gv);
                    unpack4(uq, uv);
                } else if constexpr (CLAMP == kClampF32) {
                    unpack4(gq, gv);
                    unpack4(uq, uv);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        n1 += (gv[k] > clamp) + (fabsf(uv[k]) > clamp);
                        gv[k] = fminf(gv[k], clamp);
                        uv[k] = fmaxf(fminf(uv[k], clamp), -clamp);
                    }
                } else {
                    unpack4(gq, gv);
                    unpack4(uq, uv);
                }
#pragma unroll
                for (int k = 0; k < 4; k += 2) {
                    float2 p =
                        swiglu2(make_float2(gv[k], gv[k + 1]), make_float2(uv[k], uv[k + 1]));
                    if constexpr (WEIGHTED) p = mul2(p, make_float2(wt[r], wt[r]));
                    y[r][k] = p.x;
                    y[r][k + 1] = p.y;
                }
            }
            if constexpr (CLAMP != kNoClamp) n_clamped += clamped_total(n2) + n1;
        }

        // ---- column maxima over this thread's 8 tokens -> shared table ----
        {
            float4 cm;
            float* c = &cm.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float m = fabsf(y[0][k]);
#pragma unroll
                for (int r = 1; r < 8; ++r) m = fmaxf(m, fabsf(y[r][k]));
                c[k] = m;
            }
            *reinterpret_cast<float4*>(&sm.colmax[warp][lane * 4]) = cm;
        }

        // ---- row groups: butterfly absmax across the warp --------------------
        {
            float m[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                m[r] = fmaxf(fmaxf(fabsf(y[r][0]), fabsf(y[r][1])),
                             fmaxf(fabsf(y[r][2]), fabsf(y[r][3])));
            const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
            float a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float send = b4 ? m[q] : m[4 + q];
                const float mine = b4 ? m[4 + q] : m[q];
                a[q] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 16));
            }
            float b[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float send = b3 ? a[q] : a[2 + q];
                const float mine = b3 ? a[2 + q] : a[q];
                b[q] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 8));
            }
            float c;
            {
                const float send = b2 ? b[0] : b[1];
                const float mine = b2 ? b[1] : b[0];
                c = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 4));
            }
            c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 2));
            c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 1));
            // lanes 4r .. 4r+3 hold the absmax of row r of this warp's 8 rows;
            // one of them publishes the row's reciprocal scale to the warp
            float s_own, inv_own;
            group_scale<FMT>(c, s_own, inv_own);
            if constexpr (SFX) {
                if (lay_r.flags & (kSfRoundPow2 | kSfPacked)) pow2_scale(s_own, inv_own);
            }
            if ((lane & 3) == 0) {
                if constexpr (SFX)
                    store_scale(sf, lay_r, row0 + (lane >> 2), true, cb, s_own);
                else
                    st_stream(sf + (row0 + (lane >> 2)) * CB + cb, s_own);
                sm.rowinv[warp][lane >> 2] = inv_own;
            }
            __syncwarp();
            float rinv[8];
            *reinterpret_cast<float4*>(rinv) =
                *reinterpret_cast<const float4*>(&sm.rowinv[warp][0]);
            *reinterpret_cast<float4*>(rinv + 4) =
                *reinterpret_cast<const float4*>(&sm.rowinv[warp][4]);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint32_t code = quantize4_mul<FMT>(y[r], rinv[r]);
                st_stream_u32(reinterpret_cast<uint32_t*>(out + (row0 + r) * H + c0) + lane, code);
            }
        }
        // Release the stage only now: the row-code stores above consume all 32
        // values this thread read from it, so its shared loads have completed
        // before the arrive is issued (an arrive placed right after the loads
        // can retire while they are pending, and the refill then overwrites
        // their data; releasing right after the column-maxima stores instead
        // measured 2 % slower).  After a timed-out wait the stores above hold
        // values computed from zeros; the status word marks the whole launch.
        // The proxy fence orders these generic-proxy reads before the refill,
        // which the TMA unit performs in the async proxy.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);

        // all consumers agree whether to go on (a wait may have given up)
        if (named_bar_or(kBarConsumers, kConsumers, !ok)) {
            if (ct == 0) *static_cast<volatile int*>(&sm.abort) = 1;  // stop the producer
            break;
        }

        // ---- column scales ------------------------------------------------
        if (ct < 128) {
            float m = sm.colmax[0][ct];
#pragma unroll
            for (int q = 1; q < kConsumerWarps; ++q) m = fmaxf(m, sm.colmax[q][ct]);
            float s_c, inv_c;
            group_scale<FMT>(m, s_c, inv_c);
            if constexpr (SFX) {
                if (lay_c.flags & (kSfRoundPow2 | kSfPacked)) pow2_scale(s_c, inv_c);
            }
            sm.cinv[ct] = inv_c;
            if constexpr (SFX)
                store_scale(sf_t, lay_c, c0 + ct, true, static_cast<int>(tb), s_c);
            else
                st_stream(sf_t + static_cast<int64_t>(c0 + ct) * TB + tb, s_c);
        }
        named_bar_sync(kBarConsumers, kConsumers);

        // ---- column codes into the swizzled [channel][token] tile -----------
        {
            const float4 ci4 = *reinterpret_cast<const float4*>(&sm.cinv[lane * 4]);
            const float civ[4] = {ci4.x, ci4.y, ci4.z, ci4.w};
            const int unit = warp ^ (lane & 15);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float col[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) col[r] = y[r][k];
                sm.codes[lane * 4 + k][unit] = quantize8_mul<FMT>(col, civ[k]);
            }
        }
        named_bar_sync(kBarConsumers, kConsumers);

        // ---- code tile -> out_t rows c0.., tokens t0..t0+127 ----------------
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int c = p * 64 + (ct >> 3);
            const int ch = ct & 7;            // tokens 16ch .. 16ch+15
            const int sw = (c >> 2) & 15;     // swizzle of row c
            uint4 v = *reinterpret_cast<const uint4*>(&sm.codes[c][2 * (ch ^ (sw >> 1))]);
            if (sw & 1) v = make_uint4(v.z, v.w, v.x, v.y);
            st_stream(out_t + ((static_cast<int64_t>(c0 + c) * T + t0) >> 4) + ch, v);
        }
        // The next tile writes colmax before its first consumer barrier and
        // codes only after its second, so every read of this tile's shared data
        // is complete before it is overwritten.
    }
    if constexpr (CLAMP != kNoClamp) {
        // one atomic per warp, and none when nothing was clamped
        unsigned long long t = n_clamped;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (lane == 0 && t && clamp_count) atomic_add_count(clamp_count, t);
    }
}

template <int FMT, bool WEIGHTED, int CLAMP, unsigned SFC>
cudaError_t launch(const void* x, const float* w, void* out, float* sf, void* out_t,
                   float* sf_t, int64_t T, int64_t H, const SfLayout& lay_r,
                   const SfLayout& lay_c, float clamp, unsigned long long* clamp_count,
                   cudaStream_t stream) {
    // x as a bf16 [T, 2H] matrix (gate | up), read in 128 x 128 boxes
    CUtensorMap map;
    if (!encode_bf16_2d(&map, x, 2 * H, T, 128, 128)) return cudaErrorInvalidValue;

    auto* k = &swiglu_cast_t_kernel<FMT, WEIGHTED, CLAMP, SFC>;
    const size_t smem = sizeof(SharedStorage) + 1024;
    const int64_t n_tiles = (T / 128) * (H / 128);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, smem, n_tiles);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kThreads, smem, stream, true, map, w, static_cast<uint8_t*>(out),
                      sf, static_cast<uint4*>(out_t), sf_t, T, static_cast<int>(H), lay_r, lay_c,
                      clamp, CLAMP == kClampBf16 ? bf16x2_bound(clamp) : 0u, clamp_count,
                      device_status_word());
}

// The layout of a [rows, groups] scale matrix under sf_flags.
SfLayout layout_of(unsigned sf_flags, int64_t rows, int64_t groups) {
    SfLayout lay;
    lay.flags = sf_flags;
    lay.groups = static_cast<int>(groups);
    lay.words = static_cast<int>((groups + 3) / 4);
    lay.rows4 = (rows + 3) / 4 * 4;
    return lay;
}

template <int FMT, int CLAMP, unsigned SFC>
cudaError_t launch_sfc(const void* x, const float* w, void* out, float* sf, void* out_t,
                       float* sf_t, int64_t T, int64_t H, const SfLayout& lr, const SfLayout& lc,
                       float clamp, unsigned long long* clamp_count, cudaStream_t stream) {
    return w ? launch<FMT, true, CLAMP, SFC>(x, w, out, sf, out_t, sf_t, T, H, lr, lc, clamp,
                                             clamp_count, stream)
             : launch<FMT, false, CLAMP, SFC>(x, w, out, sf, out_t, sf_t, T, H, lr, lc, clamp,
                                              clamp_count, stream);
}

template <int FMT, int CLAMP>
cudaError_t launch_w(const void* x, const float* w, void* out, float* sf, void* out_t,
                     float* sf_t, int64_t T, int64_t H, unsigned sf_flags, float clamp,
                     unsigned long long* clamp_count, cudaStream_t stream) {
    const SfLayout lr = layout_of(sf_flags, T, H / 128), lc = layout_of(sf_flags, H, T / 128);
    // the reciprocal-reading bit changes nothing here (the SwiGLU casts always
    // multiply by the reciprocal)
    const unsigned f = sfc_of(sf_flags, false);
    if (f == kSfcNone)
        return launch_sfc<FMT, CLAMP, kSfcNone>(x, w, out, sf, out_t, sf_t, T, H, lr, lc, clamp,
                                                clamp_count, stream);
    if (f == kSfcUe8m0ColMajor)
        return launch_sfc<FMT, CLAMP, kSfcUe8m0ColMajor>(x, w, out, sf, out_t, sf_t, T, H, lr, lc,
                                                         clamp, clamp_count, stream);
    if (f == kSfcF32ColMajor)
        return launch_sfc<FMT, CLAMP, kSfcF32ColMajor>(x, w, out, sf, out_t, sf_t, T, H, lr, lc,
                                                       clamp, clamp_count, stream);
    return launch_sfc<FMT, CLAMP, kSfcRuntime>(x, w, out, sf, out_t, sf_t, T, H, lr, lc, clamp,
                                               clamp_count, stream);
}

}  // namespace

cudaError_t launch_swiglu_cast_t(const void* x, const float* w, void* out, float* sf,
                                 void* out_t, float* sf_t, int64_t T, int64_t H, int fmt,
                                 unsigned sf_flags, const float* clamp,
                                 unsigned long long* clamp_count, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const float c = clamp ? *clamp : 0.0f;
    const int kind = !clamp ? kNoClamp : (bf16x2_bound(c) ? kClampBf16 : kClampF32);
    if (fmt == kFmtE4M3) {
        if (kind == kClampBf16)
            return launch_w<kFmtE4M3, kClampBf16>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c,
                                                  clamp_count, stream);
        if (kind == kClampF32)
            return launch_w<kFmtE4M3, kClampF32>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c,
                                                 clamp_count, stream);
        return launch_w<kFmtE4M3, kNoClamp>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c,
                                            nullptr, stream);
    }
    if (kind == kClampBf16)
        return launch_w<kFmtE5M2, kClampBf16>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c,
                                              clamp_count, stream);
    if (kind == kClampF32)
        return launch_w<kFmtE5M2, kClampF32>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c,
                                             clamp_count, stream);
    return launch_w<kFmtE5M2, kNoClamp>(x, w, out, sf, out_t, sf_t, T, H, sf_flags, c, nullptr,
                                        stream);
}

}  // namespace tkq
