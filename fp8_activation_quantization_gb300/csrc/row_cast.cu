// row_cast.cu -- the per-token-group FP8 casts with row-major outputs:
//   * the plain per_token_cast of a bf16 [T, C] matrix ("DeepSeek开源TileKernels：
//     用Python写的GPU算子逼近硬件性能上限" (itsolotime.com) §3.2), and
//   * swiglu_forward_and_per_token_cast of a bf16 [T, 2H] gate|up matrix,
//     optionally times a per-row routing weight (same page, §3.3).
// Per 1x128 group: absmax -> scale s = max(amax, 1e-4) / fmt_max -> FP8 codes.
//
// GB300 design: a persistent CTA per (SM x 3) streams "chunks" of 32 rows x
// one 128-channel block.  Warp 8 is the producer: one lane loads each chunk
// with one 2-D TMA box per operand (gate, and up for SwiGLU: 8 KB each) into a
// 64 KB ring of stages (8 plain or 4 SwiGLU chunks in flight per CTA).  Rows past
// T are zero-filled by the TMA unit and never stored, so ragged T needs no
// special path.  Warps 0..7 are consumers: warp w owns rows 4w..4w+3 of the
// chunk, eight lanes per row (lane j holds elements [8j, 8j+8) and
// [64+8j, 64+8j+8), read as two conflict-free 16-byte shared loads), the
// group absmax is three xor shuffles, and codes leave as 8-byte stores (eight
// lanes write one 64-byte run).  The plain cast writes the codes of the exact
// binary32 quotient fl(x / s) (see `quotient`), so it is bit-exact; the SwiGLU
// casts write the codes of y * fl(1 / s) as the page's kernel does.
// Every mbarrier wait is bounded (tkq_async.cuh).
#include <cuda.h>

#include "tkq_async.cuh"
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroupsPerLane = 1;               // row groups per lane per chunk
constexpr int kRows = 32 * kGroupsPerLane;      // rows per chunk
constexpr int kBoxBytes = kRows * 256;          // one kRows x 128 bf16 box
constexpr int kMinBlocksPerSm = 3;
constexpr int kRingBytes = 65536;               // shared ring per CTA

enum Mode { kPlain = 0, kSwiglu = 1, kSwigluWeighted = 2 };

template <int MODE>
struct ModeTraits {
    static constexpr int kOperands = MODE == kPlain ? 1 : 2;  // boxes per chunk
    static constexpr int kStageBytes = kOperands * kBoxBytes;
    static constexpr int kStages = kRingBytes / kStageBytes;
};

template <int MODE>
struct alignas(1024) RowSmem {
    uint8_t stage[ModeTraits<MODE>::kStages][ModeTraits<MODE>::kStageBytes];
    uint64_t full[ModeTraits<MODE>::kStages];
    uint64_t empty[ModeTraits<MODE>::kStages];
    int abort;
};

template <int FMT, int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSm)
    row_cast_kernel(const __grid_constant__ CUtensorMap tmap, const float* __restrict__ w,
                    uint2* __restrict__ out, float* __restrict__ sf, int64_t T, int C_out,
                    unsigned int* __restrict__ status) {
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
                uint64_t* full = &sm.full[pos.stage];
                mbar_arrive_expect_tx(full, MT::kStageBytes);
                tma_load_2d(sm.stage[pos.stage], &tmap, x0, y0, full);
                if constexpr (MT::kOperands == 2)
                    tma_load_2d(sm.stage[pos.stage] + kBoxBytes, &tmap, C_out + x0, y0, full);
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
    const int sub = lane >> 3;          // row within a block of four
    const int j = lane & 7;             // position within the group
    RingPos<MT::kStages> pos;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < RB; tw.next(), pos.advance()) {
        const int s = static_cast<int>(pos.stage);
        const int cb = static_cast<int>(tw.col);
        const int64_t row_base = static_cast<int64_t>(tw.row) * kRows;

        float wt[kGroupsPerLane];
#pragma unroll
        for (int q = 0; q < kGroupsPerLane; ++q) {
            wt[q] = 1.0f;
            if constexpr (MODE == kSwigluWeighted) {
                const int64_t row = row_base + q * 32 + warp * 4 + sub;
                if (row < T) wt[q] = __ldg(w + row);
            }
        }

        if (!mbar_wait_bounded(&sm.full[s], pos.phase, &sm.abort, status)) {
            *static_cast<volatile int*>(&sm.abort) = 1;  // stop the producer
            break;
        }
#pragma unroll
        for (int q = 0; q < kGroupsPerLane; ++q) {
            const int r = q * 32 + warp * 4 + sub;  // row within the chunk
            const int64_t row = row_base + r;
            const uint8_t* p = sm.stage[s] + r * 256 + j * 16;
            float v[16];
            if constexpr (MODE == kPlain) {
                unpack8(*reinterpret_cast<const uint4*>(p), v);
                unpack8(*reinterpret_cast<const uint4*>(p + 128), v + 8);
            } else {
                float g[16], u[16];
                unpack8(*reinterpret_cast<const uint4*>(p), g);
                unpack8(*reinterpret_cast<const uint4*>(p + 128), g + 8);
                unpack8(*reinterpret_cast<const uint4*>(p + kBoxBytes), u);
                unpack8(*reinterpret_cast<const uint4*>(p + kBoxBytes + 128), u + 8);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    v[k] = swiglu(g[k], u[k]);
                    if constexpr (MODE == kSwigluWeighted) v[k] = __fmul_rn(v[k], wt[q]);
                }
            }
            float m = fmaxf(absmax8(v), absmax8(v + 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            float sc, inv;
            group_scale<FMT>(m, sc, inv);
            if (row < T) {
                uint2* o = out + (row * C_out + cb * 128) / 8;
                uint2 lo, hi;
                if constexpr (MODE == kPlain) {
                    lo = quantize8<FMT>(v, sc, inv);
                    hi = quantize8<FMT>(v + 8, sc, inv);
                } else {
                    lo = quantize8_mul<FMT>(v, inv);
                    hi = quantize8_mul<FMT>(v + 8, inv);
                }
                st_stream(o + j, lo);
                st_stream(o + 8 + j, hi);
                if (j == 0) st_stream(sf + row * CB + cb, sc);
            }
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
}

template <int FMT, int MODE>
cudaError_t launch(const void* x, const float* w, void* out, float* sf, int64_t T, int64_t C_out,
                   cudaStream_t stream) {
    // x as a bf16 [T, cols] matrix: C columns (plain) or 2H (gate | up)
    const int64_t cols = ModeTraits<MODE>::kOperands * C_out;
    CUtensorMap map;
    if (!encode_bf16_2d(&map, x, cols, T, 128, kRows)) return cudaErrorInvalidValue;

    auto* k = &row_cast_kernel<FMT, MODE>;
    const size_t smem = sizeof(RowSmem<MODE>) + 1024;
    const int64_t n_chunks = ((T + kRows - 1) / kRows) * (C_out / 128);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kThreads, smem, n_chunks);
    k<<<grid, kThreads, smem, stream>>>(map, w, static_cast<uint2*>(out), sf, T,
                                        static_cast<int>(C_out), device_status_word());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_per_token_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                  int fmt, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return fmt == kFmtE4M3 ? launch<kFmtE4M3, kPlain>(x, nullptr, out, sf, T, C, stream)
                           : launch<kFmtE5M2, kPlain>(x, nullptr, out, sf, T, C, stream);
}

cudaError_t launch_swiglu_cast(const void* x, const float* w, void* out, float* sf, int64_t T,
                               int64_t H, int fmt, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (fmt == kFmtE4M3)
        return w ? launch<kFmtE4M3, kSwigluWeighted>(x, w, out, sf, T, H, stream)
                 : launch<kFmtE4M3, kSwiglu>(x, w, out, sf, T, H, stream);
    return w ? launch<kFmtE5M2, kSwigluWeighted>(x, w, out, sf, T, H, stream)
             : launch<kFmtE5M2, kSwiglu>(x, w, out, sf, T, H, stream);
}

}  // namespace tkq
