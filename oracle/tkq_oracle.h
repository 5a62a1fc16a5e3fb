/*
 * tkq_oracle.h -- plain, slow, single-threaded CPU oracle for per-token-group
 * FP8 activation quantization (plain cast, SwiGLU-fused cast, transposed cast).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm use it.  It shares no code, header, table or
 * constant with the CUDA library; the only thing the two sides have in common
 * is the seeded input generator, which holds none of the method's arithmetic.
 *
 * Sources (web pages about DeepSeek TileKernels):
 *  [P2] "DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件性能上限"
 *       (itsolotime.com): §3.1 quantisation config (clamp_min_value),
 *       §3.2 per-token cast kernel (group absmax -> scale -> codes),
 *       §3.3 SwiGLU fused with the cast (y = silu(g) * u * w, g the gate and u
 *       the up half).
 *  [P1] "TileKernels 与 DeepGEMM 的分界线：DeepSeek 开源内核栈的分工"
 *       (chatdocs.ruinique.com): §2 operator table (per_token_cast,
 *       per_channel_cast (+transpose / fused), swiglu_forward_and_per_token_cast).
 *  [P4] "刚刚！DeepSeek开源高性能GPU算子库TileKernels" (info.datadowell.com):
 *       quant/ section, the SwiGLU + FP8 + transpose triple fusion.
 *
 * Arithmetic: every floating-point step is a single IEEE binary32 operation
 * in round-to-nearest-even (the pages evaluate in fp32: [P2] §3.3 widens both
 * halves with T.float32).  exp() is taken in binary64 and rounded once to
 * binary32, i.e. a correctly rounded fp32 exponential in all but vanishingly
 * rare double-rounding cases.  The library must be compiled with
 * -ffp-contract=off so no multiply-add is fused.
 *
 * All arrays are caller-owned, host memory, row-major and contiguous.  bf16
 * values are passed as their raw uint16 bit patterns.
 */
#ifndef TKQ_ORACLE_H
#define TKQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* FP8 formats.  ORA_E4M3 = float8_e4m3fn (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448);
 * ORA_E5M2 = float8_e5m2 (1 sign, 5 exponent bits with bias 15, 2 mantissa
 * bits, IEEE-style infinities and NaNs, largest finite 57344). */
enum { ORA_E4M3 = 0, ORA_E5M2 = 1 };

/* Status: 0 on success, -1 on a bad argument (unknown format, group that does
 * not divide the extent, negative sizes). */

/* Largest finite value of the format (448 or 57344); 0 for an unknown fmt. */
double ora_fp8_max(int fmt);

/* Value of one FP8 code, from the format definition (NaN codes give NaN,
 * E5M2 infinity codes give +-inf). */
double ora_fp8_decode(uint8_t code, int fmt);

/* Saturating round-to-nearest-even FP8 code of one binary32 value.
 * |v| above the largest finite value (including +-inf) gives +-max
 * (0x7E/0xFE for E4M3, 0x7B/0xFB for E5M2); NaN gives 0x7F; the sign of zero
 * and of values that round to zero is kept (0x80 for negative). */
uint8_t ora_fp8_encode(float v, int fmt);

/* ora_fp8_encode over n values: out[i] = ora_fp8_encode(v[i], fmt). */
int ora_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out);

/* Group scale: fl32( max(amax, 1e-4f) / fmt_max ). */
float ora_group_scale(float amax, int fmt);

/* bf16 bit pattern -> binary32 (exact). */
float ora_bf16_to_f32(uint16_t b);

/* Plain per-token cast of a bf16 [T, C] matrix: for each row and each run of
 * `group` consecutive channels, s = ora_group_scale(max |x|), sf[t, j] = s,
 * out[t, c] = ora_fp8_encode(fl32(x[t, c] / s)).  out: [T, C] codes;
 * sf: [T, C/group] fp32. */
int ora_per_token_cast(const uint16_t* x, int64_t T, int64_t C, int64_t group,
                       int fmt, uint8_t* out, float* sf);

/* The same cast applied to an fp32 [T, C] matrix. */
int ora_cast_rows_f32(const float* y, int64_t T, int64_t C, int64_t group,
                      int fmt, uint8_t* out, float* sf);

/* Cast along the token axis of an fp32 [T, C] matrix: for each channel c and
 * each run b of `group` consecutive tokens, s = ora_group_scale(max_t |y[t,c]|),
 * sf_t[c, b] = s and out_t[c, t] = code of fl32(y[t, c] / s).
 * out_t: [C, T] codes (the column-major copy of [T, C]); sf_t: [C, T/group]. */
int ora_cast_cols_f32(const float* y, int64_t T, int64_t C, int64_t group,
                      int fmt, uint8_t* out_t, float* sf_t);

/* SwiGLU values of a bf16 [T, 2H] gate|up matrix (gate = columns [0, H),
 * up = columns [H, 2H)): y[t, c] = ((g / (1 + exp(-g))) * u) [* w[t]], each
 * operation rounded to binary32, left to right.  w may be NULL (no weight). */
int ora_swiglu_values(const uint16_t* x, const float* w, int64_t T, int64_t H,
                      float* y);

/* SwiGLU with the optional clamp of [P2] §3.3 (use_clamp,
 * swiglu_clamp_value): before the SwiGLU, g = min(g, c) and
 * u = max(min(u, c), -c).  clamp == NULL: no clamp (ora_swiglu_values);
 * otherwise *clamp = c, finite and > 0.  If n_clamped is not NULL it receives
 * the number of input values the clamp changed (gates above c, ups above c or
 * below -c).  The pages say only that clamps are counted with a sum reducer
 * and an atomic add; counting each changed value is the plain reading. */
int ora_swiglu_values_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                            const float* clamp, float* y, int64_t* n_clamped);

/* SwiGLU followed by the per-token cast of y: out [T, H], sf [T, H/group]. */
int ora_swiglu_cast(const uint16_t* x, const float* w, int64_t T, int64_t H,
                    int64_t group, int fmt, uint8_t* out, float* sf);

/* SwiGLU, the per-token cast of y, and the token-axis cast of the same fp32 y:
 * out [T, H], sf [T, H/group], out_t [H, T], sf_t [H, T/group].
 * T must be a multiple of group. */
int ora_swiglu_cast_t(const uint16_t* x, const float* w, int64_t T, int64_t H,
                      int64_t group, int fmt, uint8_t* out, float* sf,
                      uint8_t* out_t, float* sf_t);

/* ora_swiglu_cast and ora_swiglu_cast_t with the clamp of
 * ora_swiglu_values_clamp (same clamp and n_clamped arguments). */
int ora_swiglu_cast_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                          int64_t group, int fmt, const float* clamp, uint8_t* out, float* sf,
                          int64_t* n_clamped);
int ora_swiglu_cast_t_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                            int64_t group, int fmt, const float* clamp, uint8_t* out,
                            float* sf, uint8_t* out_t, float* sf_t, int64_t* n_clamped);

/* Scale-factor layout options (TileKernels CastOutputConfig round_sf,
 * use_packed_ue8m0, use_tma_aligned_col_major_sf: [P2] §3.1; their purpose,
 * feeding the GEMM's TMA in its own layout: [P1] §4C).
 *   ORA_SF_ROUND_POW2   s is rounded up to a power of two: 2^ceil(log2 s0),
 *                       s0 the fp32 scale of the plain rule.
 *   ORA_SF_UE8M0_PACKED each (power-of-two) scale is stored as its UE8M0 byte
 *                       (the biased binary32 exponent, value 2^(e-127)); four
 *                       consecutive groups of a row share one 32-bit word,
 *                       group 4k+i in byte i.  Implies ORA_SF_ROUND_POW2.
 *   ORA_SF_COL_MAJOR    scales stored column-major: element (t, j) at
 *                       j * T4 + t with T4 = T rounded up to a multiple of 4
 *                       (16-byte aligned columns); padding rows hold 0.
 * Layouts of sf (G groups per row, W = ceil(G / 4) words):
 *   default            fp32 [T, G]          ORA_SF_COL_MAJOR          fp32 [G, T4]
 *   ORA_SF_UE8M0_PACKED int32 [T, W]        UE8M0_PACKED|COL_MAJOR   int32 [W, T4]
 * Packed bytes of groups >= G in a row's last word are 0.
 * One more flag selects the quotient reading of the codes:
 *   ORA_Q_RECIPROCAL    codes of fl32(v * fl32(1 / s)), the product by the
 *                       correctly rounded reciprocal of the scale (the
 *                       TileKernels kernel multiplies by sf_inv: [P2] §3.2),
 *                       instead of the quotient fl32(v / s).  The scales and
 *                       their layout are unchanged; with power-of-two scales
 *                       the two readings agree. */
enum { ORA_SF_ROUND_POW2 = 1, ORA_SF_UE8M0_PACKED = 2, ORA_SF_COL_MAJOR = 4,
       ORA_Q_RECIPROCAL = 8 };

/* Power of two >= s (s a positive normal binary32): 2^ceil(log2 s). */
float ora_pow2_ceil(float s);

/* Bytes of the scale output for T rows of G groups under `flags`. */
int64_t ora_sf_bytes(int64_t T, int64_t G, int flags);

/* The row cast of an fp32 [T, C] matrix with scale options: codes of
 * fl32(y / s) with s from ora_group_scale, rounded up to a power of two when
 * asked; scales written in the layout `flags` selects (sf is raw bytes). */
int ora_cast_rows_f32_ex(const float* y, int64_t T, int64_t C, int64_t group, int fmt,
                         int flags, uint8_t* out, void* sf);

/* Per-channel cast of a bf16 [T, C] matrix ([P1] §2 per_channel_cast
 * (+transpose)): groups of `group` consecutive tokens of one channel.
 * transpose == 0: out [T, C] codes in place, sf fp32 [T/group, C];
 * transpose != 0: out [C, T] (the column-major copy), sf fp32 [C, T/group].
 * T must be a multiple of group. */
int ora_per_channel_cast(const uint16_t* x, int64_t T, int64_t C, int64_t group, int fmt,
                         int transpose, uint8_t* out, float* sf);

/* Per-block cast of a bf16 [T, C] matrix ([P1] §2 per_block_cast): one scale
 * per block of `block` x `block` elements (the last row block may be short:
 * its amax covers the rows that exist).  out [T, C] codes, sf fp32
 * [ceil(T/block), C/block]. */
int ora_per_block_cast(const uint16_t* x, int64_t T, int64_t C, int64_t block, int fmt,
                       uint8_t* out, float* sf);

/* Cast back ([P1] §2 cast_back): y = fl32(decode(code) * s) for codes [T, C]
 * with scales of groups of gr rows x gc columns, sf row-major
 * [ceil(T/gr), C/gc] (gr, gc = 1 x 128 per-token, 128 x 1 per-channel,
 * 128 x 128 per-block).  out fp32 [T, C]. */
int ora_cast_back(const uint8_t* codes, const float* sf, int64_t T, int64_t C, int64_t gr,
                  int64_t gc, int fmt, float* out);

/* Gradient of y = silu(g) * u [* w] for a bf16 [T, 2H] gate|up input and a
 * bf16 [T, H] upstream gradient dy, written as the fp32 [T, 2H] matrix
 * [dg | du]:
 *   dg = dy * u * sigma(g) * (1 + g * (1 - sigma(g))) [* w]
 *   du = dy * silu(g) [* w],   sigma(g) = 1 / (1 + exp(-g)), silu = g sigma(g).
 * The pages name swiglu_backward_and_per_token_cast but give no formula and
 * no precision, so this is the textbook derivative evaluated in binary64 and
 * rounded once to binary32. */
int ora_swiglu_backward_values(const uint16_t* x, const uint16_t* dy, const float* w,
                               int64_t T, int64_t H, float* grad);

/* The gradient above followed by the per-token cast of [dg | du]:
 * out [T, 2H] codes, sf [T, 2H/group]. */
int ora_swiglu_backward_cast(const uint16_t* x, const uint16_t* dy, const float* w,
                             int64_t T, int64_t H, int64_t group, int fmt,
                             uint8_t* out, float* sf);

#ifdef __cplusplus
}
#endif
#endif /* TKQ_ORACLE_H */
