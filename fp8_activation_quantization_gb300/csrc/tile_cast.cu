// tile_cast.cu -- FP8 casts whose groups span 128 tokens ("TileKernels 与
// DeepGEMM 的分界线" (chatdocs.ruinique.com) §2 operator table):
//   * per_channel_cast: groups of 128 consecutive tokens of one channel,
//     codes in place ([T, C]) or as the transposed copy ([C, T]);
//   * per_block_cast: one scale per 128 x 128 block.
// Scale s = fl32(max(amax, 1e-4) / fmt_max) ("DeepSeek开源TileKernels：用Python
// 写的GPU算子逼近硬件性能上限" (itsolotime.com) §3.1, §3.2); codes are those of
// the exact binary32 quotient fl(x / s), so results are bit-exact.
//
// GB300 design: persistent kernels, one CTA per SM, a producer warp streaming
// TMA boxes into a shared ring (every wait bounded) and consumer warps that
// hold 32 values each.  With one CTA per SM the per-tile dependent chain of a
// group step (maxima -> barrier -> scale -> codes) is exposed unless another
// group of warps works meanwhile, so the transposed per-channel and the
// per-block casts run two independent consumer groups; the in-place
// per-channel cast, whose chain hides behind its stores, runs one group of 16.
// Ragged T (per-block only): rows past T are zero-filled by TMA (zeros do not
// change an absmax) and never stored.
#include <cuda.h>

#include "tkq_async.cuh"
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kTileBytes = 128 * 128 * 2;   // one 128 x 128 bf16 box

// The producer lane of every kernel here: TMA boxes of box_cols x 128 bf16 for
// the CTA's tiles (tile walk start blockIdx.x, step gridDim.x, CB tiles per
// row), ring position by issue order; on exit it waits (bounded) for the copies
// it issued.
template <int STAGES, int TILE_BYTES>
__device__ __forceinline__ void produce_tiles(uint8_t (*stage)[TILE_BYTES], uint64_t* full,
                                              uint64_t* empty, int* abort, const CUtensorMap* tmap,
                                              uint32_t CB, uint32_t TB, int box_cols,
                                              unsigned int* status) {
    uint32_t issued = 0;
    RingPos<STAGES> pos;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB; tw.next(), ++issued) {
        if (!mbar_wait_bounded(&empty[pos.stage], pos.phase ^ 1u, abort, status)) {
            *static_cast<volatile int*>(abort) = 1;
            break;
        }
        mbar_arrive_expect_tx(&full[pos.stage], TILE_BYTES);
        tma_load_2d(stage[pos.stage], tmap, static_cast<int>(tw.col) * box_cols,
                    static_cast<int>(tw.row * 128), &full[pos.stage]);
        pos.advance();
    }
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t k = first; k < issued; ++k)
        mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1u, nullptr, status);
}

// Called by the producer lane between grid_dependency_launch and
// grid_dependency_wait: the boxes of the CTA's first STAGES tiles (those it
// loads first) go to L2 while the grid before this one drains.
template <int STAGES>
__device__ __forceinline__ void prefetch_first_tiles(const CUtensorMap* tmap, uint32_t CB,
                                                     uint32_t TB, int box_cols) {
    int k = 0;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB && k < STAGES; tw.next(), ++k)
        tma_prefetch_2d(tmap, static_cast<int>(tw.col) * box_cols,
                        static_cast<int>(tw.row * 128));
}

// ---------------------------------------------------------------------------
// In-place per-channel cast: 16 consumer warps, each holding an 8-token x
// 4-channel block of a 128 x 128 tile (warp w: tokens 8w..8w+7, lane l:
// channels 4l..4l+3), a 4-stage ring.  Column maxima over a thread's 8 tokens
// go to a 16 x 128 shared table; 128 threads form the column scales; codes
// leave as 4-byte stores (a warp writes one 128-byte run per row).
// ---------------------------------------------------------------------------
constexpr int kChWarps = 16;
constexpr int kChConsumers = kChWarps * 32;
constexpr int kChThreads = kChConsumers + 32;
constexpr int kChStages = 4;

struct alignas(1024) ChSmem {
    uint8_t stage[kChStages][kTileBytes];
    float colmax[kChWarps][128];
    float cs[128];
    float cinv[128];
    uint64_t full[kChStages];
    uint64_t empty[kChStages];
    int abort;
};

template <int FMT>
__global__ void __launch_bounds__(kChThreads, 1)
    channel_kernel(const __grid_constant__ CUtensorMap tmap, uint8_t* __restrict__ out,
                   float* __restrict__ sf, int64_t T, int C, unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    ChSmem& sm = *reinterpret_cast<ChSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t CB = static_cast<uint32_t>(C) >> 7;
    const uint32_t TB = static_cast<uint32_t>(T >> 7);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kChStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kChWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_launch();
    if (warp == kChWarps && lane == 0) prefetch_first_tiles<kChStages>(&tmap, CB, TB, 128);
    grid_dependency_wait();  // the previous grid on the stream is done
    if (warp == kChWarps) {
        if (lane == 0)
            produce_tiles<kChStages, kTileBytes>(sm.stage, sm.full, sm.empty, &sm.abort, &tmap, CB,
                                                 TB, 128, status);
        return;
    }

    const int ct = threadIdx.x;
    RingPos<kChStages> pos;
    for (TileWalk tw(blockIdx.x, gridDim.x, CB); tw.row < TB; tw.next(), pos.advance()) {
        const int s = static_cast<int>(pos.stage);
        const uint32_t tb = tw.row;
        const int c0 = static_cast<int>(tw.col) * 128;
        const int64_t row0 = static_cast<int64_t>(tb) * 128 + warp * 8;

        const bool ok = mbar_wait_bounded(&sm.full[s], pos.phase, &sm.abort, status);
        float v[8][4];
        {
            const uint8_t* base = sm.stage[s] + warp * 8 * 256 + lane * 8;
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                uint2 q = make_uint2(0, 0);
                if (ok) q = *reinterpret_cast<const uint2*>(base + r * 256);
                unpack4(q, v[r]);
            }
        }
        // column maxima over this thread's 8 tokens -> shared table
        {
            float4 cm;
            float* c = &cm.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float m = fabsf(v[0][k]);
#pragma unroll
                for (int r = 1; r < 8; ++r) m = fmaxf(m, fabsf(v[r][k]));
                c[k] = m;
            }
            *reinterpret_cast<float4*>(&sm.colmax[warp][lane * 4]) = cm;
        }
        if (named_bar_or(1, kChConsumers, !ok)) {
            if (ct == 0) *static_cast<volatile int*>(&sm.abort) = 1;
            break;
        }
        if (ct < 128) {
            float m = sm.colmax[0][ct];
#pragma unroll
            for (int q = 1; q < kChWarps; ++q) m = fmaxf(m, sm.colmax[q][ct]);
            float s_c, inv_c;
            group_scale<FMT>(m, s_c, inv_c);
            sm.cs[ct] = s_c;
            sm.cinv[ct] = inv_c;
            st_stream(sf + static_cast<int64_t>(tb) * C + c0 + ct, s_c);
        }
        named_bar_sync(1, kChConsumers);
        const float4 cs4 = *reinterpret_cast<const float4*>(&sm.cs[lane * 4]);
        const float4 ci4 = *reinterpret_cast<const float4*>(&sm.cinv[lane * 4]);
        const float csv[4] = {cs4.x, cs4.y, cs4.z, cs4.w};
        const float civ[4] = {ci4.x, ci4.y, ci4.z, ci4.w};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t code = quantize4_each<FMT>(v[r], csv, civ);
            st_stream_u32(reinterpret_cast<uint32_t*>(out + (row0 + r) * C + c0) + lane, code);
        }
        // Release the stage once the values read from it are consumed (the
        // stores above depend on all of them), behind an async-proxy fence.
        // The next tile writes colmax before its first barrier and cs / cinv
        // only after it, so this tile's reads of both are complete first.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
}

template <int FMT>
cudaError_t launch_channel(const void* x, void* out, float* sf, int64_t T, int64_t C,
                           cudaStream_t stream) {
    CUtensorMap map;
    if (!encode_bf16_2d(&map, x, C, T, 128, 128)) return cudaErrorInvalidValue;
    auto* k = &channel_kernel<FMT>;
    const size_t smem = sizeof(ChSmem) + 1024;
    const int64_t n_tiles = (T / 128) * (C / 128);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kChThreads, smem, n_tiles);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kChThreads, smem, stream, true, map, static_cast<uint8_t*>(out),
                      sf, T, static_cast<int>(C), device_status_word());
}

// ---------------------------------------------------------------------------
// Transposed per-channel cast with two independent consumer groups.
//
// With one lock-stepped group of 16 warps a tile's dependent chain (column
// maxima, barrier, four warps forming scales, barrier, codes into the shared
// tile, barrier, tile out) is exposed once per tile.  Here two groups of 8
// warps take alternate half-width tiles (128 tokens x 64 channels) from one
// 8-stage TMA ring, each with its own named barrier, column table and code
// tile, so one group's chain overlaps the other's work.  A thread holds 16
// tokens x 2 channels (warp w of a group: tokens 16w..16w+15; lane l:
// channels 2l, 2l+1), i.e. one 16-byte run of codes per channel; the code tile
// [channel][16-token unit] is XOR-swizzled by (channel / 2) & 7 so that both
// the 16-byte writes (eight lanes: eight rows) and the 16-byte reads (eight
// threads: one row) hit distinct bank groups.
// ---------------------------------------------------------------------------
constexpr int kCtGroupWarps = 8;
constexpr int kCtGroupThreads = kCtGroupWarps * 32;
constexpr int kCtGroups = 2;
constexpr int kCtThreads = kCtGroups * kCtGroupThreads + 32;
constexpr int kCtStages = 8;
constexpr int kCtTileCols = 64;
constexpr int kCtTileBytes = 128 * kCtTileCols * 2;

struct CtGroupSmem {
    uint4 codes[kCtTileCols][8];          // [channel][16-token unit], swizzled
    float colmax[kCtGroupWarps][kCtTileCols];
    float cs[kCtTileCols];
    float cinv[kCtTileCols];
};

struct alignas(1024) CtSmem {
    uint8_t stage[kCtStages][kCtTileBytes];
    CtGroupSmem g[kCtGroups];
    uint64_t full[kCtStages];
    uint64_t empty[kCtStages];
    int abort;
};

template <int FMT>
__global__ void __launch_bounds__(kCtThreads, 1)
    channel_t_kernel(const __grid_constant__ CUtensorMap tmap, uint8_t* __restrict__ out,
                     float* __restrict__ sf, int64_t T, int C, unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    CtSmem& sm = *reinterpret_cast<CtSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t CB = static_cast<uint32_t>(C) / kCtTileCols;
    const uint32_t TB = static_cast<uint32_t>(T >> 7);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCtStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCtGroupWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_launch();
    if (warp == kCtGroups * kCtGroupWarps && lane == 0)
        prefetch_first_tiles<kCtStages>(&tmap, CB, TB, kCtTileCols);
    grid_dependency_wait();  // the previous grid on the stream is done

    if (warp == kCtGroups * kCtGroupWarps) {   // producer
        if (lane == 0)
            produce_tiles<kCtStages, kCtTileBytes>(sm.stage, sm.full, sm.empty, &sm.abort, &tmap,
                                                   CB, TB, kCtTileCols, status);
        return;
    }

    // ------------------------------------------------------ consumer groups
    const int grp = warp / kCtGroupWarps;
    const int wg = warp - grp * kCtGroupWarps;
    const int gt = threadIdx.x - grp * kCtGroupThreads;   // thread within the group
    const int bar = 1 + grp;                             // the group's named barrier
    CtGroupSmem& G = sm.g[grp];
    uint32_t i = static_cast<uint32_t>(grp);            // CTA-local tile index
    for (TileWalk tw(blockIdx.x + grp * gridDim.x, kCtGroups * gridDim.x, CB); tw.row < TB;
         tw.next(), i += kCtGroups) {
        const uint32_t s = i % kCtStages;
        const uint32_t tb = tw.row;
        const int64_t t0 = static_cast<int64_t>(tb) * 128;
        const int c0 = static_cast<int>(tw.col) * kCtTileCols;

        const bool ok = mbar_wait_bounded(&sm.full[s], (i / kCtStages) & 1u, &sm.abort, status);
        float v[16][2];
        {
            const uint8_t* base = sm.stage[s] + (16 * wg) * (kCtTileCols * 2) + lane * 4;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const uint32_t q =
                    ok ? *reinterpret_cast<const uint32_t*>(base + r * kCtTileCols * 2) : 0u;
                v[r][0] = bf16_lo(q);
                v[r][1] = bf16_hi(q);
            }
        }
        // column maxima over this thread's 16 tokens (two chains per column)
        {
            float2 cm;
            float* c = &cm.x;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float a = fabsf(v[0][k]), b = fabsf(v[1][k]);
#pragma unroll
                for (int r = 2; r < 16; r += 2) {
                    a = fmaxf(a, fabsf(v[r][k]));
                    b = fmaxf(b, fabsf(v[r + 1][k]));
                }
                c[k] = fmaxf(a, b);
            }
            *reinterpret_cast<float2*>(&G.colmax[wg][lane * 2]) = cm;
        }
        if (named_bar_or(bar, kCtGroupThreads, !ok)) {
            if (gt == 0) *static_cast<volatile int*>(&sm.abort) = 1;
            break;
        }
        if (gt < kCtTileCols) {
            float m = G.colmax[0][gt];
#pragma unroll
            for (int q = 1; q < kCtGroupWarps; ++q) m = fmaxf(m, G.colmax[q][gt]);
            float s_c, inv_c;
            group_scale<FMT>(m, s_c, inv_c);
            G.cs[gt] = s_c;
            G.cinv[gt] = inv_c;
            st_stream(sf + static_cast<int64_t>(c0 + gt) * TB + tb, s_c);
        }
        named_bar_sync(bar, kCtGroupThreads);
        {
            const float2 cs2 = *reinterpret_cast<const float2*>(&G.cs[lane * 2]);
            const float2 ci2 = *reinterpret_cast<const float2*>(&G.cinv[lane * 2]);
            const float csv[2] = {cs2.x, cs2.y};
            const float civ[2] = {ci2.x, ci2.y};
            const int unit = wg ^ (lane & 7);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float col[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) col[r] = v[r][k];
                const uint2 lo = quantize8<FMT>(col, csv[k], civ[k]);
                const uint2 hi = quantize8<FMT>(col + 8, csv[k], civ[k]);
                G.codes[lane * 2 + k][unit] = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        // release the stage (its values are consumed) behind an async-proxy fence
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);

        named_bar_sync(bar, kCtGroupThreads);   // the code tile is complete
        uint4* out_t = reinterpret_cast<uint4*>(out);
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int c = p * 32 + (gt >> 3);
            const int u = gt & 7;
            const uint4 q = G.codes[c][u ^ ((c >> 1) & 7)];
            st_stream(out_t + ((static_cast<int64_t>(c0 + c) * T + t0) >> 4) + u, q);
        }
        // The next tile of this group writes colmax before its first barrier
        // and the code tile only after its second, so these reads come first.
    }
}

// ---------------------------------------------------------------------------
// Per-block cast with two independent consumer groups.
//
// A block's scale needs all of its 128 x 128 values, so a group takes whole
// blocks: two groups of 8 warps alternate blocks from one 6-stage ring of
// 128 x 128 TMA boxes, each with its own named barrier and max table.  Warp w
// of a group covers tokens 16w..16w+15 in two halves of 8 rows (lane l:
// channels 4l..4l+3): pass 1 reads both halves from the stage for the thread's
// absmax (four independent chains per half), the warp max is one redux.sync on
// the bit patterns (non-negative binary32 values order like their bits), the
// group's table of 8 warp maxima is reduced the same way after one barrier,
// and pass 2 reads the halves again from the (still resident) stage to write
// the codes.  One group's dependent chain overlaps the other's work.
// ---------------------------------------------------------------------------
constexpr int kBgStages = 6;

struct alignas(1024) BgSmem {
    uint8_t stage[kBgStages][kTileBytes];
    uint32_t bmax[kCtGroups][2][kCtGroupWarps];   // [group][iteration parity][warp]
    uint64_t full[kBgStages];
    uint64_t empty[kBgStages];
    int abort;
};

// rows 8 h .. 8 h + 7 of warp wg's 16, 4 channels of lane `lane`, from a stage
__device__ __forceinline__ void load_half(const uint8_t* stage, int wg, int h, int lane, bool ok,
                                          float (&v)[8][4]) {
    const uint8_t* base = stage + (16 * wg + 8 * h) * 256 + lane * 8;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        uint2 q = make_uint2(0, 0);
        if (ok) q = *reinterpret_cast<const uint2*>(base + r * 256);
        unpack4(q, v[r]);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kCtThreads, 1)
    block_cast_kernel(const __grid_constant__ CUtensorMap tmap, uint8_t* __restrict__ out,
                      float* __restrict__ sf, int64_t T, int C, unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    BgSmem& sm = *reinterpret_cast<BgSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t{1023});
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t CB = static_cast<uint32_t>(C) >> 7;
    const uint32_t TB = static_cast<uint32_t>((T + 127) >> 7);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBgStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCtGroupWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_launch();
    if (warp == kCtGroups * kCtGroupWarps && lane == 0)
        prefetch_first_tiles<kBgStages>(&tmap, CB, TB, 128);
    grid_dependency_wait();  // the previous grid on the stream is done

    if (warp == kCtGroups * kCtGroupWarps) {   // producer
        if (lane == 0)
            produce_tiles<kBgStages, kTileBytes>(sm.stage, sm.full, sm.empty, &sm.abort, &tmap, CB,
                                                 TB, 128, status);
        return;
    }

    // ------------------------------------------------------ consumer groups
    const int grp = warp / kCtGroupWarps;
    const int wg = warp - grp * kCtGroupWarps;
    const int gt = threadIdx.x - grp * kCtGroupThreads;
    const int bar = 1 + grp;
    uint32_t parity = 0;
    uint32_t i = static_cast<uint32_t>(grp);            // CTA-local tile index
    for (TileWalk tw(blockIdx.x + grp * gridDim.x, kCtGroups * gridDim.x, CB); tw.row < TB;
         tw.next(), i += kCtGroups) {
        const uint32_t s = i % kBgStages;
        const uint32_t tb = tw.row;
        const int c0 = static_cast<int>(tw.col) * 128;
        const int64_t row0 = static_cast<int64_t>(tb) * 128 + 16 * wg;

        const bool ok = mbar_wait_bounded(&sm.full[s], (i / kBgStages) & 1u, &sm.abort, status);
        float m = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8][4];
            load_half(sm.stage[s], wg, h, lane, ok, v);
            float mk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mk[k] = fabsf(v[0][k]);
#pragma unroll
                for (int r = 1; r < 8; ++r) mk[k] = fmaxf(mk[k], fabsf(v[r][k]));
            }
            m = fmaxf(m, fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])));
        }
        const uint32_t mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
        if (lane == 0) sm.bmax[grp][parity][wg] = mw;
        if (named_bar_or(bar, kCtGroupThreads, !ok)) {
            if (gt == 0) *static_cast<volatile int*>(&sm.abort) = 1;
            break;
        }
        // lanes l, l + 8, l + 16, l + 24 read warp l's maximum
        const uint32_t bw = __reduce_max_sync(0xffffffffu, sm.bmax[grp][parity][lane & 7]);
        float sc, inv;
        group_scale<FMT>(__uint_as_float(bw), sc, inv);
        // rows of this warp that exist (fewer than 16 only in a last, short block row)
        const int64_t left = T - row0;
        const int live = left < 16 ? static_cast<int>(left) : 16;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[8][4];
            load_half(sm.stage[s], wg, h, lane, true, v);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (8 * h + r < live)
                    st_stream_u32(
                        reinterpret_cast<uint32_t*>(out + (row0 + 8 * h + r) * C + c0) + lane,
                        quantize4<FMT>(v[r], sc, inv));
            }
        }
        if (gt == 0) st_stream(sf + static_cast<int64_t>(tb) * CB + tw.col, sc);
        // release the stage after the stores that consume its values
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
        parity ^= 1u;
    }
}

template <int FMT>
cudaError_t launch_block(const void* x, void* out, float* sf, int64_t T, int64_t C,
                         cudaStream_t stream) {
    CUtensorMap map;
    if (!encode_bf16_2d(&map, x, C, T, 128, 128)) return cudaErrorInvalidValue;
    auto* k = &block_cast_kernel<FMT>;
    const size_t smem = sizeof(BgSmem) + 1024;
    const int64_t n_tiles = ((T + 127) / 128) * (C / 128);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kCtThreads, smem,
                                     (n_tiles + 1) / 2);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kCtThreads, smem, stream, true, map, static_cast<uint8_t*>(out),
                      sf, T, static_cast<int>(C), device_status_word());
}

template <int FMT>
cudaError_t launch_channel_t(const void* x, void* out, float* sf, int64_t T, int64_t C,
                             cudaStream_t stream) {
    CUtensorMap map;
    if (!encode_bf16_2d(&map, x, C, T, kCtTileCols, 128)) return cudaErrorInvalidValue;
    auto* k = &channel_t_kernel<FMT>;
    const size_t smem = sizeof(CtSmem) + 1024;
    const int64_t n_tiles = (T / 128) * (C / kCtTileCols);
    const int grid = persistent_grid(reinterpret_cast<const void*>(k), kCtThreads, smem,
                                     (n_tiles + 1) / 2);
    if (const cudaError_t e = upload_checks(stream)) return e;
    return launch_pdl(k, grid, kCtThreads, smem, stream, true, map, static_cast<uint8_t*>(out),
                      sf, T, static_cast<int>(C), device_status_word());
}

}  // namespace

cudaError_t launch_per_channel_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                    int fmt, bool transpose, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (transpose)
        return fmt == kFmtE4M3 ? launch_channel_t<kFmtE4M3>(x, out, sf, T, C, stream)
                               : launch_channel_t<kFmtE5M2>(x, out, sf, T, C, stream);
    return fmt == kFmtE4M3 ? launch_channel<kFmtE4M3>(x, out, sf, T, C, stream)
                           : launch_channel<kFmtE5M2>(x, out, sf, T, C, stream);
}

cudaError_t launch_per_block_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                  int fmt, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    return fmt == kFmtE4M3 ? launch_block<kFmtE4M3>(x, out, sf, T, C, stream)
                           : launch_block<kFmtE5M2>(x, out, sf, T, C, stream);
}

}  // namespace tkq
