/*
 * tkq.h -- C ABI of libtkq.so: per-token-group FP8 activation quantization on
 * GB300 (sm_103a).
 *
 * The operations follow the TileKernels quantization operators described in
 *   [P2] "DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限"
 *        (itsolotime.com), §3.1 (cast config, clamp_min_value), §3.2 (the
 *        per-token cast kernel), §3.3 (SwiGLU fused with the cast);
 *   [P1] "TileKernels 与 DeepGEMM 的分界线：DeepSeek 开源内核栈的分工"
 *        (chatdocs.ruinique.com), §2 operator table;
 *   [P4] "刚刚！DeepSeek开源高性能GPU算子库TileKernels" (info.datadowell.com),
 *        quant/ section (SwiGLU + FP8 + transpose in one pass).
 *
 * Common definitions
 * ------------------
 * group      Only 128 is accepted (1x128 groups along the quantized axis).
 * fmt        TKQ_FMT_E4M3 (float8_e4m3fn, largest finite 448) or
 *            TKQ_FMT_E5M2 (float8_e5m2, largest finite 57344).
 * scale      For each group, s = fl32(max(amax, 1e-4) / fmt_max) where amax is
 *            the largest |value| of the group ([P2] §3.1 and §3.2).
 * code       The saturating round-to-nearest-even FP8 code of the binary32
 *            quotient fl32(value / s); results beyond the largest finite value
 *            saturate to it.  The sign of zero is kept.
 * bf16       Inputs are bf16, row-major and contiguous.
 * outputs    Codes are one byte per element, row-major; scales are fp32.
 *
 * Memory, streams, errors
 * -----------------------
 * - Every pointer is a DEVICE pointer owned and allocated by the caller; the
 *   library allocates nothing and keeps no per-call state.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream).  TKQ_OK means "arguments valid and kernel launched";
 *   results are ready when the stream reaches that point.
 * - Argument errors are detected on the host before anything is launched and
 *   leave every buffer untouched: TKQ_ERR_NULL (a required pointer is NULL),
 *   TKQ_ERR_SHAPE (negative sizes, or an extent that is not a multiple of the
 *   group), TKQ_ERR_GROUP (group != 128), TKQ_ERR_FMT (unknown format),
 *   TKQ_ERR_ALIGN (x, out, out_t not 16-byte aligned, or sf, sf_t, w not
 *   4-byte aligned), TKQ_ERR_ALIAS (an output overlaps an input or another
 *   output), TKQ_ERR_FLAGS (unknown option bits), TKQ_ERR_VALUE (an invalid
 *   scalar argument: a clamp bound that is not finite and positive).
 *   T == 0 is an empty batch: TKQ_OK, nothing is launched and the pointers
 *   may be NULL.
 * - A failed launch returns TKQ_ERR_CUDA (cudaGetLastError after the launch).
 * - A kernel that runs into trouble on the device (a bounded wait for its
 *   copies that gave up, see tkq_read_device_status) cannot change the status
 *   its asynchronous call already returned; it records the event in the
 *   device status word, and tkq_read_device_status reports it as
 *   TKQ_ERR_TIMEOUT.
 * - Environment (for tests and measurements; no result depends on it):
 *   TKQ_NUM_SMS=n sizes the persistent grids for n SMs; TKQ_SWIGLU_KERNEL=flat
 *   or =ring runs the SwiGLU forward cast through one of its two bit-identical
 *   kernels, which are otherwise chosen by measured speed (the flat stream
 *   without a routing weight, and with one up to 384 MiB of input; the TMA
 *   ring for weighted launches above that).
 * - Inputs must be finite; NaN or Inf inputs give unspecified codes, and so
 *   does a SwiGLU value or gradient that overflows binary32.
 * - Calls on the same buffers from different streams must be ordered by the
 *   caller.
 */
#ifndef TKQ_H
#define TKQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TKQ_FMT_E4M3 = 0,
    TKQ_FMT_E5M2 = 1
} tkq_fmt;

typedef enum {
    TKQ_OK = 0,
    TKQ_ERR_NULL = 1,
    TKQ_ERR_SHAPE = 2,
    TKQ_ERR_GROUP = 3,
    TKQ_ERR_FMT = 4,
    TKQ_ERR_ALIGN = 5,
    TKQ_ERR_CUDA = 6,
    TKQ_ERR_TIMEOUT = 7,  /* a bounded in-kernel wait gave up (tkq_read_device_status) */
    TKQ_ERR_ALIAS = 8,
    TKQ_ERR_FLAGS = 9,
    TKQ_ERR_VALUE = 10
} tkq_status;

/* A cudaStream_t passed as an opaque pointer. */
typedef void* tkq_stream_t;

/*
 * Plain per-token cast ([P2] §3.2, per_token_cast; [P1] §6 steps 3 and 10).
 *   x   : bf16 [T, C], row-major
 *   out : FP8 codes [T, C], row-major
 *   sf  : fp32 [T, C/128], row-major; sf[t, j] scales x[t, 128j : 128j+128]
 * T >= 0 (any value, no tile alignment needed); C > 0, C % 128 == 0.
 */
tkq_status tkq_per_token_cast(const void* x, void* out, float* sf,
                              int64_t T, int64_t C, int group, int fmt,
                              tkq_stream_t stream);

/*
 * SwiGLU fused with the per-token cast ([P2] §3.3,
 * swiglu_forward_and_per_token_cast), optionally with a per-row routing
 * weight.  For every row t and channel c < H:
 *   g = x[t, c], u = x[t, H + c] (both widened to fp32),
 *   y = ((g / (1 + exp(-g))) * u) [* w[t]]       (binary32 arithmetic)
 * and y is cast as in tkq_per_token_cast.
 *   x   : bf16 [T, 2H], gate = columns [0, H), up = columns [H, 2H)
 *   w   : fp32 [T] or NULL (no weight)
 *   out : FP8 codes [T, H];  sf : fp32 [T, H/128]
 * T >= 0; H > 0, H % 128 == 0.
 * exp(-g) and the reciprocal come from the SM's ex2.approx / rcp.approx, so y
 * may differ from exactly rounded binary32 steps by a few ulp, and codes are
 * those of y times the rounded reciprocal of s (as the TileKernels kernel
 * multiplies by sf_inv, [P2] §3.2): they are not bit-pinned to a CPU
 * evaluation (parity: scales within 1e-6 relative, codes within one FP8 step).
 * tkq_swiglu_values returns the fp32 y itself.
 */
tkq_status tkq_swiglu_cast(const void* x, const float* w, void* out, float* sf,
                           int64_t T, int64_t H, int group, int fmt,
                           tkq_stream_t stream);

/*
 * SwiGLU + per-token cast + transposed cast in one pass ([P4] quant/ triple
 * fusion; [P1] §2 "per_channel_cast (+transpose / fused)").  Writes the same
 * out / sf as tkq_swiglu_cast (bit for bit) and, from the same fp32 y, a
 * column-major copy quantized with 1x128 groups along the token axis:
 *   out_t : FP8 codes [H, T]; out_t[c, t] is the code of y[t, c]
 *   sf_t  : fp32 [H, T/128]; sf_t[c, b] scales y[128b : 128b+128, c]
 * T >= 0 with T % 128 == 0; H > 0, H % 128 == 0.
 */
tkq_status tkq_swiglu_cast_t(const void* x, const float* w, void* out, float* sf,
                             void* out_t, float* sf_t,
                             int64_t T, int64_t H, int group, int fmt,
                             tkq_stream_t stream);

/*
 * Scale-factor layouts ([P2] §3.1: the round_sf, use_packed_ue8m0 and
 * use_tma_aligned_col_major_sf options of the cast config; [P1] §4C: the
 * scales are written directly in the layout a TMA-fed FP8 GEMM reads, so no
 * separate re-layout pass is needed).  Flags, combinable:
 *   TKQ_SF_ROUND_POW2    every scale is rounded up to a power of two,
 *                        s = 2^ceil(log2 s0) with s0 the plain fp32 scale;
 *                        codes are those of y / s (exact: a power-of-two
 *                        scaling).
 *   TKQ_SF_UE8M0_PACKED  each scale is stored as its UE8M0 byte (the biased
 *                        binary32 exponent; value 2^(byte - 127)), four
 *                        consecutive groups of a row per 32-bit word, group
 *                        4k+i in byte i (little-endian).  Implies ROUND_POW2.
 *   TKQ_SF_COL_MAJOR     scales stored column-major: entry (t, j) at
 *                        j * T4 + t, T4 = T rounded up to a multiple of 4, so
 *                        every column starts 16-byte aligned (sf must be
 *                        16-byte aligned); padding rows hold 0.
 * With G groups per row (C/128, H/128, or 2H/128 for the backward) and
 * W = ceil(G/4), sf is
 *   fp32 [T, G] (no flags), fp32 [G, T4] (COL_MAJOR),
 *   int32 [T, W] (UE8M0_PACKED), int32 [W, T4] (UE8M0_PACKED | COL_MAJOR);
 * bytes of a row's last word beyond group G-1 are 0.
 * One more flag, which does not change the scales or their layout, selects
 * the quotient reading of the plain per-token casts (tkq_per_token_cast_ex,
 * tkq_per_token_cast_f32):
 *   TKQ_Q_RECIPROCAL     codes of fl32(x * fl32(1 / s)), the product by the
 *                        correctly rounded reciprocal of the scale ([P2] §3.2:
 *                        the kernel multiplies by sf_inv), instead of the
 *                        exact quotient fl32(x / s).  Bit-exact against the
 *                        same reading of the definition.  With power-of-two
 *                        scales the readings agree.  The SwiGLU casts always
 *                        multiply this way, so there the flag changes nothing.
 * Unknown bits give TKQ_ERR_FLAGS.
 */
#define TKQ_SF_ROUND_POW2 1u
#define TKQ_SF_UE8M0_PACKED 2u
#define TKQ_SF_COL_MAJOR 4u
#define TKQ_Q_RECIPROCAL 8u

/* Size in bytes of the scale buffer for T rows of groups_per_row groups under
 * sf_flags, or -1 for invalid arguments. */
int64_t tkq_sf_bytes(int64_t T, int64_t groups_per_row, unsigned sf_flags);

/*
 * Per-token cast of an fp32 input ([P2] §3.2: the per-token cast kernel takes
 * a BF16 or FP32 [num_tokens, hidden] matrix): x fp32 [T, C], row-major,
 * 16-byte aligned;
 * otherwise tkq_per_token_cast_ex (codes of the exact quotient fl32(x / s),
 * bit-exact; sf in the layout sf_flags selects).
 */
tkq_status tkq_per_token_cast_f32(const float* x, void* out, void* sf, int64_t T, int64_t C,
                                  int group, int fmt, unsigned sf_flags, tkq_stream_t stream);

/* tkq_per_token_cast, tkq_swiglu_cast and tkq_swiglu_backward_cast with a
 * scale-factor layout (sf_flags above; sf sized by tkq_sf_bytes).  With
 * sf_flags == 0 they are the calls above.  tkq_swiglu_cast_t_ex applies the
 * same layout to both of its scale outputs: sf as a [T, H/128] matrix (sized
 * tkq_sf_bytes(T, H/128, sf_flags)) and sf_t as an [H, T/128] matrix (sized
 * tkq_sf_bytes(H, T/128, sf_flags)); the codes of both copies are those of
 * the product by the reciprocal of the (possibly power-of-two) scale. */
tkq_status tkq_per_token_cast_ex(const void* x, void* out, void* sf, int64_t T, int64_t C,
                                 int group, int fmt, unsigned sf_flags, tkq_stream_t stream);
tkq_status tkq_swiglu_cast_ex(const void* x, const float* w, void* out, void* sf, int64_t T,
                              int64_t H, int group, int fmt, unsigned sf_flags,
                              tkq_stream_t stream);
tkq_status tkq_swiglu_backward_cast_ex(const void* x, const void* dy, const float* w, void* out,
                                       void* sf, int64_t T, int64_t H, int group, int fmt,
                                       unsigned sf_flags, tkq_stream_t stream);
tkq_status tkq_swiglu_cast_t_ex(const void* x, const float* w, void* out, void* sf, void* out_t,
                                void* sf_t, int64_t T, int64_t H, int group, int fmt,
                                unsigned sf_flags, tkq_stream_t stream);

/*
 * Device status word.  The kernels fed by TMA bulk copies (the transposed,
 * per-channel and per-block casts, and the SwiGLU casts on long launches) wait
 * on shared-memory barriers for those copies; every such wait gives up after
 * one second, sets TKQ_DEVICE_TIMEOUT in the current device's status word and
 * lets the kernel return (its outputs are then incomplete) instead of hanging.
 * tkq_read_device_status synchronizes the current device, stores the word in
 * *flags and, if clear != 0, resets it.  Returns TKQ_ERR_TIMEOUT when the word
 * it read holds TKQ_DEVICE_TIMEOUT (*flags is set then too), else TKQ_OK.
 * Errors: TKQ_ERR_NULL (flags NULL), TKQ_ERR_CUDA (the synchronization or
 * copy failed).
 * (Not from the source pages: this is the library's failure reporting.)
 */
#define TKQ_DEVICE_TIMEOUT 1u
tkq_status tkq_read_device_status(uint32_t* flags, int clear);

/*
 * Self-test of the bounded-wait machinery: launches one CTA on `stream` that
 * waits on a barrier nothing ever arrives on, for limit_ns nanoseconds
 * (0 < limit_ns <= 2e9), then records TKQ_DEVICE_TIMEOUT in the status word and
 * returns.  No memory is touched besides the status word.  Errors:
 * TKQ_ERR_SHAPE (limit out of range), TKQ_ERR_CUDA (launch failed).
 * (Not from the source pages.)
 */
tkq_status tkq_selftest_wait_timeout(int64_t limit_ns, tkq_stream_t stream);

/*
 * SwiGLU backward fused with the per-token cast ([P1] §2 operator table and
 * §6 step 13, swiglu_backward_and_per_token_cast; the pages give no formula,
 * so this is the derivative of y = silu(g) * u [* w]).  For every row t and
 * channel c < H, with g = x[t, c], u = x[t, H + c], d = dy[t, c] and
 * sigma = 1 / (1 + exp(-g)):
 *   dg = d * u * sigma * (1 + g * (1 - sigma)) [* w[t]]
 *   du = d * g * sigma [* w[t]]
 * and the fp32 matrix [dg | du] is cast per token.
 *   x   : bf16 [T, 2H] (gate | up, as given to the forward)
 *   dy  : bf16 [T, H], gradient of the forward output y
 *   w   : fp32 [T] or NULL
 *   out : FP8 codes [T, 2H] (dg in columns [0, H), du in [H, 2H))
 *   sf  : fp32 [T, 2H/128]
 * T >= 0; H > 0, H % 128 == 0.  Codes are those of the product by the
 * reciprocal scale, like tkq_swiglu_cast.
 */
tkq_status tkq_swiglu_backward_cast(const void* x, const void* dy, const float* w, void* out,
                                    float* sf, int64_t T, int64_t H, int group, int fmt,
                                    tkq_stream_t stream);

/*
 * Per-channel cast ([P1] §2 operator table, per_channel_cast (+transpose)):
 * groups of 128 consecutive tokens of one channel, with the scale and code
 * rules of the common definitions (exact quotient, bit-exact).
 *   x   : bf16 [T, C], row-major
 *   transpose == 0:  out FP8 codes [T, C] (in place of x's layout),
 *                    sf fp32 [T/128, C]; sf[b, c] scales x[128b : 128b+128, c]
 *   transpose != 0:  out FP8 codes [C, T] (the column-major copy, row c holds
 *                    channel c), sf fp32 [C, T/128]
 * T >= 0, T % 128 == 0; C > 0, C % 128 == 0.  Alignment: x, out 16 bytes,
 * sf 4 bytes.
 */
tkq_status tkq_per_channel_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                int group, int fmt, int transpose, tkq_stream_t stream);

/*
 * Per-block cast ([P1] §2 operator table, per_block_cast): one scale per
 * block of 128 tokens x 128 channels; the last block row may be short (its
 * amax covers the rows that exist).
 *   x   : bf16 [T, C], row-major
 *   out : FP8 codes [T, C]
 *   sf  : fp32 [ceil(T/128), C/128]; sf[b, j] scales x[128b:128b+128, 128j:128j+128]
 * T >= 0; C > 0, C % 128 == 0.  Alignment: x, out 16 bytes, sf 4 bytes.
 */
tkq_status tkq_per_block_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                              int block, int fmt, tkq_stream_t stream);

/*
 * Cast back ([P1] §2 operator table, cast_back): dequantization
 *   out[t, c] = fl32(decode(codes[t, c]) * sf[t / group_rows, c / group_cols])
 * where decode is the exact value of the FP8 code (NaN codes give NaN).
 *   codes : FP8 codes [T, C], row-major
 *   sf    : fp32 [ceil(T/group_rows), C/group_cols], row-major
 *   out   : fp32 [T, C] (out_dtype TKQ_OUT_F32) or bf16 [T, C]
 *           (TKQ_OUT_BF16: the fp32 result rounded to nearest even)
 * (group_rows, group_cols) is (1, 128) for per-token scales, (128, 1) for
 * per-channel scales and (128, 128) for per-block scales; anything else is
 * TKQ_ERR_GROUP.  T >= 0; C > 0, C % 128 == 0.  Alignment: codes, out 16
 * bytes; sf 16 bytes when group_cols == 1, else 4.  out_dtype other than the
 * two below is TKQ_ERR_FMT.
 */
#define TKQ_OUT_F32 0
#define TKQ_OUT_BF16 1
tkq_status tkq_cast_back(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                         int group_rows, int group_cols, int fmt, int out_dtype,
                         tkq_stream_t stream);

/*
 * SwiGLU casts with the clamp of [P2] §3.3 (use_clamp, swiglu_clamp_value):
 * before the SwiGLU, the gate is clamped from above, g = min(g, c), and the up
 * projection on both sides, u = max(min(u, c), -c).  The number of input
 * values the clamp changes (gates above c, ups above c or below -c; a value
 * equal to c is unchanged) is ADDED to *clamp_count: the caller zeroes the
 * counter, and consecutive calls accumulate (the page counts clamps with a sum
 * reducer and an atomic add; counting each changed value is this library's
 * reading).  Otherwise these are tkq_swiglu_cast_ex and tkq_swiglu_cast_t_ex.
 *   clamp_value : c, finite and > 0, else TKQ_ERR_VALUE
 *   clamp_count : DEVICE pointer to one uint64 (8-byte aligned, overlapping
 *                 no other buffer of the call), or NULL for no count.
 */
tkq_status tkq_swiglu_cast_clamp(const void* x, const float* w, void* out, void* sf, int64_t T,
                                 int64_t H, int group, int fmt, unsigned sf_flags,
                                 float clamp_value, uint64_t* clamp_count, tkq_stream_t stream);
tkq_status tkq_swiglu_cast_t_clamp(const void* x, const float* w, void* out, void* sf,
                                   void* out_t, void* sf_t, int64_t T, int64_t H, int group,
                                   int fmt, unsigned sf_flags, float clamp_value,
                                   uint64_t* clamp_count, tkq_stream_t stream);

/*
 * Diagnostic (not an operation of the source pages): the fp32 SwiGLU values
 *   y[t, c] = silu(x[t, c]) * x[t, H + c] [* w[t]]
 * computed exactly as tkq_swiglu_cast and tkq_swiglu_cast_t compute them
 * before quantizing (the SM's ex2 / rcp, see tkq_swiglu_cast), written out so
 * that their accuracy can be checked value by value.
 *   x : bf16 [T, 2H];  w : fp32 [T] or NULL;  y : fp32 [T, H], 16-byte aligned
 * T >= 0; H > 0, H % 128 == 0.
 */
tkq_status tkq_swiglu_values(const void* x, const float* w, float* y, int64_t T, int64_t H,
                             tkq_stream_t stream);

/*
 * Diagnostic (not an operation of the source pages): the fp32 gradients the
 * SwiGLU backward cast quantizes, computed exactly as tkq_swiglu_backward_cast
 * computes them (the SM's ex2 / rcp, the weight product), written out:
 *   y[t, c] = dg,  y[t, H + c] = du   (formulas of tkq_swiglu_backward_cast)
 *   x : bf16 [T, 2H];  dy : bf16 [T, H];  w : fp32 [T] or NULL;
 *   y : fp32 [T, 2H], 16-byte aligned, overlapping none of the inputs
 * T >= 0; H > 0, H % 128 == 0.
 */
tkq_status tkq_swiglu_backward_values(const void* x, const void* dy, const float* w, float* y,
                                      int64_t T, int64_t H, tkq_stream_t stream);

/*
 * Diagnostic (not an operation of the source pages): the FP8 codes of n fp32
 * values, unscaled, by the conversion every cast ends with (saturating
 * round-to-nearest-even, cvt.rn.satfinite; NaN gives a NaN code).  Lets the
 * hardware conversion be compared with the format definition on any value.
 *   x : fp32 [n], 16-byte aligned;  out : FP8 codes [n], 4-byte aligned
 * n >= 0, n % 4 == 0 (else TKQ_ERR_SHAPE); fmt as for the casts.
 */
tkq_status tkq_fp8_encode(const float* x, void* out, int64_t n, int fmt, tkq_stream_t stream);

/*
 * Access checking (not from the source pages; the stand-in for a memory
 * checker).  The same sources built with -DTKQ_CHECKED give libtkq_checked.so,
 * a test build in which every global load and store of the kernels is first
 * checked against the buffers of the current call (loads: its inputs and
 * outputs; stores: its outputs, sized as documented for each call).  An access
 * not wholly inside them is skipped, sets TKQ_DEVICE_OUT_OF_BOUNDS in the
 * device status word (tkq_read_device_status) and records the first byte of
 * the first such access that lies outside the buffers, read with
 * tkq_read_check_address (bit 63 set for a store).  The checked build keeps one
 * table per kernel source file, so its calls must not run concurrently.  In
 * the release build no access is checked: the status bit is never set and the
 * address reads 0.
 */
#define TKQ_DEVICE_OUT_OF_BOUNDS 2u
/* 1 in the checked build, 0 in the release build. */
int tkq_checked_build(void);
/* Synchronizes the current device, then returns (and with clear != 0 resets)
 * the first refused address.  Errors: TKQ_ERR_NULL, TKQ_ERR_CUDA. */
tkq_status tkq_read_check_address(uint64_t* addr, int clear);

/* Static, human-readable name of a status code (never NULL). */
const char* tkq_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int tkq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TKQ_H */
