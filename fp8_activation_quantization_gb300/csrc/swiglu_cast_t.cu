// swiglu_cast_t.cu -- SwiGLU + per-token FP8 cast + transposed (token-axis)
// FP8 cast in one pass.
//
// The operation is the SwiGLU + FP8 + transpose triple fusion of the quant/
// section of "刚刚！DeepSeek开源高性能GPU算子库TileKernels" (info.datadowell.com),
// i.e. swiglu_forward_and_per_token_cast ("DeepSeek开源TileKernels：用Python写的
// GPU算子逼近硬件性能上限" (itsolotime.com) §3.3) plus a per_channel_cast of the
// transposed y ("TileKernels 与 DeepGEMM 的分界线" (chatdocs.ruinique.com) §2,
// "per_channel_cast (+transpose / fused)").  Both outputs are quantized from the
// same fp32 y.
//
// GB300 design.  A CTA owns a 128-token x 128-channel tile of y at a time and
// walks tiles with a persistent grid.  Thread layout (256 threads = 8 warps):
// lane & 15 picks an 8-channel chunk, warp * 2 + lane / 16 picks an 8-token
// block, so each thread holds an 8 x 8 block of y in registers.  Per warp load
// instruction the 16 lanes of a half-warp read one 256-byte run of a row, so
// global loads are fully coalesced.
//   * Row groups (1 x 128 channels): the 16 lanes of a half-warp own the same 8
//     rows; their absmax is a butterfly that halves the live values at each of
//     four xor-shuffle steps (8 shuffles instead of 32), after which lane pair
//     (2r, 2r+1) holds row r's absmax, computes its scale once, and shuffles
//     scale and reciprocal back to the other lanes.  Codes go straight from
//     registers to HBM as 8-byte stores (a half-warp writes a 128-byte row run).
//   * Column groups (128 tokens x 1 channel): per-thread maxima over 8 tokens,
//     one halving xor-16 step, a 8 x 128 shared-memory table reduced by 128
//     threads, scales broadcast through shared memory.  The column codes are
//     transposed through a 16 KB shared tile of bytes [channel][token] whose
//     8-byte token units are XOR-swizzled by (channel / 8) so that the 8-byte
//     writes of a half-warp hit 32 distinct banks; the tile leaves as 16-byte
//     stores, eight lanes per 128-byte row run of out_t.  (The transpose
//     walkthrough of the TileKernels page, §6, rotates the column index by the
//     thread id and pads the tile for the same purpose.)
// No tensor cores: the kernel is bound by HBM bandwidth.
#include "tkq_device.cuh"
#include "tkq_internal.h"

namespace tkq {
namespace {

constexpr int kThreads = 256;

template <int FMT, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads, 2)
    swiglu_cast_t_kernel(const uint4* __restrict__ x, const float* __restrict__ w,
                         uint2* __restrict__ out, float* __restrict__ sf,
                         uint4* __restrict__ out_t, float* __restrict__ sf_t, int64_t T, int H) {
    __shared__ __align__(16) float s_colmax[8][128];
    __shared__ __align__(16) float s_cs[128];
    __shared__ __align__(16) float s_cinv[128];
    __shared__ __align__(16) uint2 s_codes[128][16];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int cc = lane & 15;                // channel chunk (8 channels)
    const int half = lane >> 4;              // which row block of the warp
    const int rb = warp * 2 + half;          // token block (8 tokens)
    const int CB = H >> 7;                   // channel tiles
    const int64_t TB = T >> 7;               // token tiles
    const int64_t n_tiles = TB * CB;
    const int64_t row_u4 = H >> 2;           // uint4 per input row (2H bf16)
    const int64_t half_u4 = H >> 3;          // uint4 offset of the up half
    const int64_t out_row_u2 = H >> 3;       // uint2 per output row

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t tb = tile / CB;
        const int cb = static_cast<int>(tile - tb * CB);
        const int64_t t0 = tb * 128;
        const int c0 = cb * 128;

        // ---- load the 8 x 8 block of gate and up --------------------------
        uint4 gq[8], uq[8];
        float wt[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int64_t row = t0 + rb * 8 + r;
            const uint4* p = x + row * row_u4 + (c0 >> 3) + cc;
            gq[r] = ld_stream(p);
            uq[r] = ld_stream(p + half_u4);
            wt[r] = 1.0f;
            if constexpr (WEIGHTED) wt[r] = ld_stream_f32(w + row);
        }

        // ---- y = silu(g) * u [* w] ----------------------------------------
        float y[8][8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float gv[8], uv[8];
            unpack8(gq[r], gv);
            unpack8(uq[r], uv);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                y[r][k] = swiglu(gv[k], uv[k]);
                if constexpr (WEIGHTED) y[r][k] = __fmul_rn(y[r][k], wt[r]);
            }
        }

        // ---- column maxima over this thread's 8 tokens, halved across the
        //      two row blocks of the warp, into shared memory ----------------
        {
            float cm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float m = fabsf(y[0][k]);
#pragma unroll
                for (int r = 1; r < 8; ++r) m = fmaxf(m, fabsf(y[r][k]));
                cm[k] = m;
            }
            float4 keep;
            float* kp = &keep.x;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float send = half ? cm[i] : cm[4 + i];
                const float mine = half ? cm[4 + i] : cm[i];
                kp[i] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 16));
            }
            *reinterpret_cast<float4*>(&s_colmax[warp][cc * 8 + half * 4]) = keep;
        }

        // ---- row groups: butterfly absmax over the 16 lanes of the half-warp
        {
            float m[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) m[r] = absmax8(y[r]);
            const int b3 = (cc >> 3) & 1, b2 = (cc >> 2) & 1, b1 = (cc >> 1) & 1;
            float a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float send = b3 ? m[i] : m[4 + i];
                const float mine = b3 ? m[4 + i] : m[i];
                a[i] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 8));
            }
            float b[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float send = b2 ? a[i] : a[2 + i];
                const float mine = b2 ? a[2 + i] : a[i];
                b[i] = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 4));
            }
            float c;
            {
                const float send = b1 ? b[0] : b[1];
                const float mine = b1 ? b[1] : b[0];
                c = fmaxf(mine, __shfl_xor_sync(0xffffffffu, send, 2));
            }
            c = fmaxf(c, __shfl_xor_sync(0xffffffffu, c, 1));
            // this lane now holds the absmax of row (cc >> 1) of its row block
            float s_own, inv_own;
            group_scale<FMT>(c, s_own, inv_own);
            const int64_t my_row = t0 + rb * 8 + (cc >> 1);
            if ((cc & 1) == 0) st_stream(sf + my_row * CB + cb, s_own);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int src = (lane & 16) | (r * 2);
                const float s = __shfl_sync(0xffffffffu, s_own, src);
                const float inv = __shfl_sync(0xffffffffu, inv_own, src);
                const int64_t row = t0 + rb * 8 + r;
                st_stream(out + row * out_row_u2 + (c0 >> 3) + cc, quantize8<FMT>(y[r], s, inv));
            }
        }

        __syncthreads();  // s_colmax complete

        // ---- column scales ------------------------------------------------
        if (tid < 128) {
            float m = s_colmax[0][tid];
#pragma unroll
            for (int q = 1; q < 8; ++q) m = fmaxf(m, s_colmax[q][tid]);
            float s, inv;
            group_scale<FMT>(m, s, inv);
            s_cs[tid] = s;
            s_cinv[tid] = inv;
            st_stream(sf_t + static_cast<int64_t>(c0 + tid) * TB + tb, s);
        }

        __syncthreads();  // s_cs / s_cinv ready

        // ---- column codes into the swizzled [channel][token] byte tile ----
        {
            float cs[8], ci[8];
            *reinterpret_cast<float4*>(cs) = *reinterpret_cast<const float4*>(&s_cs[cc * 8]);
            *reinterpret_cast<float4*>(cs + 4) = *reinterpret_cast<const float4*>(&s_cs[cc * 8 + 4]);
            *reinterpret_cast<float4*>(ci) = *reinterpret_cast<const float4*>(&s_cinv[cc * 8]);
            *reinterpret_cast<float4*>(ci + 4) = *reinterpret_cast<const float4*>(&s_cinv[cc * 8 + 4]);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float col[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) col[r] = y[r][k];
                s_codes[cc * 8 + k][rb ^ cc] = quantize8<FMT>(col, cs[k], ci[k]);
            }
        }

        __syncthreads();  // code tile complete

        // ---- code tile -> out_t rows c0.., tokens t0..t0+127 -------------
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int c = p * 32 + (tid >> 3);
            const int ch = tid & 7;          // 16-byte chunk = tokens 16ch .. 16ch+15
            const int sw = (c >> 3) & 15;    // swizzle of row c
            uint4 v = *reinterpret_cast<const uint4*>(&s_codes[c][2 * (ch ^ (sw >> 1))]);
            if (sw & 1) v = make_uint4(v.z, v.w, v.x, v.y);
            st_stream(out_t + ((static_cast<int64_t>(c0 + c) * T + t0) >> 4) + ch, v);
        }
        // The next tile's first shared-memory writes (s_colmax) come after this
        // tile's last reads of s_colmax (before the second barrier), and
        // s_codes is rewritten only after two more barriers.
    }
}

template <int FMT, bool WEIGHTED>
cudaError_t launch(const void* x, const float* w, void* out, float* sf, void* out_t,
                   float* sf_t, int64_t T, int64_t H, cudaStream_t stream) {
    const void* k = reinterpret_cast<const void*>(&swiglu_cast_t_kernel<FMT, WEIGHTED>);
    const int64_t n_tiles = (T / 128) * (H / 128);
    const int grid = persistent_grid(k, kThreads, 0, n_tiles);
    swiglu_cast_t_kernel<FMT, WEIGHTED><<<grid, kThreads, 0, stream>>>(
        static_cast<const uint4*>(x), w, static_cast<uint2*>(out), sf,
        static_cast<uint4*>(out_t), sf_t, T, static_cast<int>(H));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_swiglu_cast_t(const void* x, const float* w, void* out, float* sf,
                                 void* out_t, float* sf_t, int64_t T, int64_t H, int fmt,
                                 cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (fmt == kFmtE4M3)
        return w ? launch<kFmtE4M3, true>(x, w, out, sf, out_t, sf_t, T, H, stream)
                 : launch<kFmtE4M3, false>(x, w, out, sf, out_t, sf_t, T, H, stream);
    return w ? launch<kFmtE5M2, true>(x, w, out, sf, out_t, sf_t, T, H, stream)
             : launch<kFmtE5M2, false>(x, w, out, sf, out_t, sf_t, T, H, stream);
}

}  // namespace tkq
