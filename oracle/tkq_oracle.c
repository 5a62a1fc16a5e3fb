/*
 * tkq_oracle.c -- plain single-threaded CPU oracle for per-token-group FP8
 * activation quantization.  TEST INFRASTRUCTURE ONLY (see tkq_oracle.h for
 * the sources, the arithmetic rules and who may use it).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared tkq_oracle.c -lm
 */
#include "tkq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* FP8 format descriptions, from the definitions of float8_e4m3fn / e5m2.     */
/* ------------------------------------------------------------------------ */

typedef struct {
    int mbits;       /* explicit mantissa bits                              */
    int ebits;       /* exponent bits                                       */
    int bias;        /* exponent bias                                       */
    double maxval;   /* largest finite magnitude                            */
    uint8_t maxcode; /* code of +maxval                                     */
} fp8_desc;

static int get_desc(int fmt, fp8_desc* d) {
    if (fmt == ORA_E4M3) {
        /* 1.75 * 2^8: exponent field 15 is finite except mantissa 111 (NaN). */
        d->mbits = 3; d->ebits = 4; d->bias = 7;
        d->maxval = 448.0; d->maxcode = 0x7E;
        return 0;
    }
    if (fmt == ORA_E5M2) {
        /* 1.75 * 2^15: exponent field 31 is reserved for inf / NaN. */
        d->mbits = 2; d->ebits = 5; d->bias = 15;
        d->maxval = 57344.0; d->maxcode = 0x7B;
        return 0;
    }
    return -1;
}

double ora_fp8_max(int fmt) {
    fp8_desc d;
    return get_desc(fmt, &d) ? 0.0 : d.maxval;
}

double ora_fp8_decode(uint8_t code, int fmt) {
    fp8_desc d;
    if (get_desc(fmt, &d)) return NAN;
    const int sign = code >> 7;
    const int efield = (code >> d.mbits) & ((1 << d.ebits) - 1);
    const int mfield = code & ((1 << d.mbits) - 1);
    const int emax_field = (1 << d.ebits) - 1;
    double v;
    if (fmt == ORA_E4M3 && efield == emax_field && mfield == (1 << d.mbits) - 1) {
        return NAN;                                   /* S.1111.111 */
    }
    if (fmt == ORA_E5M2 && efield == emax_field) {
        if (mfield != 0) return NAN;                  /* S.11111.xx, xx != 0 */
        return sign ? -INFINITY : INFINITY;           /* S.11111.00 */
    }
    if (efield == 0) {
        /* subnormal: m * 2^(1 - bias - mbits) */
        v = ldexp((double)mfield, 1 - d.bias - d.mbits);
    } else {
        /* normal: (1 + m / 2^mbits) * 2^(e - bias) */
        v = ldexp(1.0 + ldexp((double)mfield, -d.mbits), efield - d.bias);
    }
    return sign ? -v : v;
}

uint8_t ora_fp8_encode(float v, int fmt) {
    fp8_desc d;
    if (get_desc(fmt, &d)) return 0;
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= d.maxval) return (uint8_t)(sign | d.maxcode);   /* satfinite */
    if (a == 0.0) return sign;

    /* Exponent of the binade holding a, floored at the smallest normal
     * exponent so that the subnormal range shares one quantum. */
    const int emin = 1 - d.bias;
    int e2;
    (void)frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                  /* floor(log2(a)) */
    if (e < emin) e = emin;
    const double quantum = ldexp(1.0, e - d.mbits);

    /* a / quantum is exact in binary64 (a has 24 significant bits).  Round it
     * to an integer, ties to the even integer. */
    const double m = a / quantum;
    double r = floor(m);
    const double frac = m - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double val = r * quantum;
    if (val > d.maxval) val = d.maxval;         /* rounds past max: saturate */
    if (val == 0.0) return sign;

    if (val < ldexp(1.0, emin)) {
        /* subnormal code: exponent field 0, mantissa = val / 2^(emin - mbits) */
        const int mfield = (int)(val / ldexp(1.0, emin - d.mbits));
        return (uint8_t)(sign | mfield);
    }
    int f2;
    const double f = frexp(val, &f2);           /* val = f * 2^f2 */
    const int ev = f2 - 1;                      /* val in [2^ev, 2^(ev+1)) */
    const int mfield = (int)((2.0 * f - 1.0) * (double)(1 << d.mbits));
    return (uint8_t)(sign | ((ev + d.bias) << d.mbits) | mfield);
}

int ora_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out) {
    fp8_desc d;
    if (get_desc(fmt, &d) || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = ora_fp8_encode(v[i], fmt);
    return 0;
}

/* Scale rule: the clamp minimum is 1e-4 ([P2] §3.1, CastOutputConfig
 * .clamp_min_value for float8_e4m3fn; the E5M2 branch is lost from the page
 * and the same 1e-4 is used), and the scale is amax over the format maximum
 * ([P2] §3.2, get_sf_and_inv). */
float ora_group_scale(float amax, int fmt) {
    const float clamp_min = 1e-4f;
    const float a = (amax > clamp_min) ? amax : clamp_min;
    const float fmax = (float)ora_fp8_max(fmt);
    return a / fmax;
}

float ora_bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Casts                                                                     */
/* ------------------------------------------------------------------------ */

/* Largest |v| of n values at stride `stride` (in elements). */
static float group_absmax(const float* v, int64_t n, int64_t stride) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        const float a = fabsf(v[i * stride]);
        if (a > amax) amax = a;
    }
    return amax;
}

/* The code of each value is the code of the binary32 quotient v / s. */
static void encode_group(const float* v, int64_t n, int64_t stride, float s, int fmt,
                         uint8_t* codes, int64_t code_stride) {
    for (int64_t i = 0; i < n; ++i) {
        const float q = v[i * stride] / s;
        codes[i * code_stride] = ora_fp8_encode(q, fmt);
    }
}

/* The reciprocal-multiply reading: the code of each value is the code of the
 * binary32 product v * fl32(1 / s) ("DeepSeek开源TileKernels：用Python写的GPU算子
 * 逼近硬件性能上限" §3.2: the kernel multiplies by sf_inv; its computation is not
 * shown, read here as the correctly rounded reciprocal). */
static void encode_group_reciprocal(const float* v, int64_t n, float s, int fmt,
                                    uint8_t* codes) {
    const float inv = 1.0f / s;
    for (int64_t i = 0; i < n; ++i) {
        const float q = v[i] * inv;
        codes[i] = ora_fp8_encode(q, fmt);
    }
}

/* One group of n values at stride `stride` -> scale + codes. */
static float cast_group(const float* v, int64_t n, int64_t stride, int fmt,
                        uint8_t* codes, int64_t code_stride) {
    const float amax = group_absmax(v, n, stride);
    const float s = ora_group_scale(amax, fmt);
    encode_group(v, n, stride, s, fmt, codes, code_stride);
    return s;
}

int ora_cast_rows_f32(const float* y, int64_t T, int64_t C, int64_t group,
                      int fmt, uint8_t* out, float* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || group <= 0 || C % group) return -1;
    const int64_t G = C / group;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < G; ++j)
            sf[t * G + j] = cast_group(y + t * C + j * group, group, 1, fmt,
                                       out + t * C + j * group, 1);
    return 0;
}

int ora_per_token_cast(const uint16_t* x, int64_t T, int64_t C, int64_t group,
                       int fmt, uint8_t* out, float* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || group <= 0 || C % group) return -1;
    const int64_t G = C / group;
    float* v = (float*)malloc((size_t)(group > 0 ? group : 1) * sizeof(float));
    if (!v) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < G; ++j) {
            const uint16_t* xg = x + t * C + j * group;
            for (int64_t i = 0; i < group; ++i) v[i] = ora_bf16_to_f32(xg[i]);
            sf[t * G + j] = cast_group(v, group, 1, fmt, out + t * C + j * group, 1);
        }
    }
    free(v);
    return 0;
}

int ora_cast_cols_f32(const float* y, int64_t T, int64_t C, int64_t group,
                      int fmt, uint8_t* out_t, float* sf_t) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || group <= 0 || T % group) return -1;
    const int64_t B = T / group;
    for (int64_t c = 0; c < C; ++c)
        for (int64_t b = 0; b < B; ++b)
            /* values y[b*group + i, c], i.e. stride C; codes land contiguously
             * in row c of the [C, T] output */
            sf_t[c * B + b] = cast_group(y + (b * group) * C + c, group, C, fmt,
                                         out_t + c * T + b * group, 1);
    return 0;
}

/* SwiGLU: silu(g) * u with silu(g) = g / (1 + exp(-g)) ([P2] §3.3), then the
 * optional per-row routing weight, each step rounded to binary32. */
int ora_swiglu_values_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                            const float* clamp, float* y, int64_t* n_clamped) {
    if (T < 0 || H < 0 || (clamp && !(*clamp > 0.0f && *clamp < INFINITY))) return -1;
    int64_t n = 0;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* row = x + t * 2 * H;
        for (int64_t c = 0; c < H; ++c) {
            float g = ora_bf16_to_f32(row[c]);
            float u = ora_bf16_to_f32(row[H + c]);
            if (clamp) {
                /* [P2] §3.3: the gate is clamped from above only, the up
                 * projection on both sides; every value changed is counted */
                const float cv = *clamp;
                if (g > cv) { g = cv; ++n; }
                if (u > cv) { u = cv; ++n; }
                if (u < -cv) { u = -cv; ++n; }
            }
            const float e = (float)exp(-(double)g);
            const float den = 1.0f + e;
            const float silu = g / den;
            float val = silu * u;
            if (w) val = val * w[t];
            y[t * H + c] = val;
        }
    }
    if (n_clamped) *n_clamped = n;
    return 0;
}

int ora_swiglu_values(const uint16_t* x, const float* w, int64_t T, int64_t H,
                      float* y) {
    return ora_swiglu_values_clamp(x, w, T, H, NULL, y, NULL);
}

int ora_swiglu_cast_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                          int64_t group, int fmt, const float* clamp, uint8_t* out, float* sf,
                          int64_t* n_clamped) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || H < 0 || group <= 0 || H % group) return -1;
    float* y = (float*)malloc((size_t)(T * H > 0 ? T * H : 1) * sizeof(float));
    if (!y) return -1;
    int rc = ora_swiglu_values_clamp(x, w, T, H, clamp, y, n_clamped);
    if (!rc) rc = ora_cast_rows_f32(y, T, H, group, fmt, out, sf);
    free(y);
    return rc;
}

int ora_swiglu_cast(const uint16_t* x, const float* w, int64_t T, int64_t H,
                    int64_t group, int fmt, uint8_t* out, float* sf) {
    return ora_swiglu_cast_clamp(x, w, T, H, group, fmt, NULL, out, sf, NULL);
}

int ora_swiglu_cast_t_clamp(const uint16_t* x, const float* w, int64_t T, int64_t H,
                            int64_t group, int fmt, const float* clamp, uint8_t* out,
                            float* sf, uint8_t* out_t, float* sf_t, int64_t* n_clamped) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || H < 0 || group <= 0 || H % group || T % group)
        return -1;
    float* y = (float*)malloc((size_t)(T * H > 0 ? T * H : 1) * sizeof(float));
    if (!y) return -1;
    int rc = ora_swiglu_values_clamp(x, w, T, H, clamp, y, n_clamped);
    if (!rc) rc = ora_cast_rows_f32(y, T, H, group, fmt, out, sf);
    if (!rc) rc = ora_cast_cols_f32(y, T, H, group, fmt, out_t, sf_t);
    free(y);
    return rc;
}

int ora_swiglu_cast_t(const uint16_t* x, const float* w, int64_t T, int64_t H,
                      int64_t group, int fmt, uint8_t* out, float* sf,
                      uint8_t* out_t, float* sf_t) {
    return ora_swiglu_cast_t_clamp(x, w, T, H, group, fmt, NULL, out, sf, out_t, sf_t, NULL);
}

/* SwiGLU backward: the derivative of y = silu(g) * u [* w] ("TileKernels 与
 * DeepGEMM 的分界线" (chatdocs.ruinique.com) §2 and §6 step 13 name the
 * operator; no formula is given, so this is the textbook one), evaluated in
 * binary64 and rounded once to binary32. */
int ora_swiglu_backward_values(const uint16_t* x, const uint16_t* dy, const float* w,
                               int64_t T, int64_t H, float* grad) {
    if (T < 0 || H < 0) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const uint16_t* row = x + t * 2 * H;
        const double wt = w ? (double)w[t] : 1.0;
        for (int64_t c = 0; c < H; ++c) {
            const double g = (double)ora_bf16_to_f32(row[c]);
            const double u = (double)ora_bf16_to_f32(row[H + c]);
            const double d = (double)ora_bf16_to_f32(dy[t * H + c]);
            const double sig = 1.0 / (1.0 + exp(-g));
            const double silu = g * sig;
            const double dsilu = sig * (1.0 + g * (1.0 - sig));
            grad[t * 2 * H + c] = (float)(d * u * dsilu * wt);
            grad[t * 2 * H + H + c] = (float)(d * silu * wt);
        }
    }
    return 0;
}

int ora_swiglu_backward_cast(const uint16_t* x, const uint16_t* dy, const float* w,
                             int64_t T, int64_t H, int64_t group, int fmt,
                             uint8_t* out, float* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || H < 0 || group <= 0 || H % group) return -1;
    float* g = (float*)malloc((size_t)(T * 2 * H > 0 ? T * 2 * H : 1) * sizeof(float));
    if (!g) return -1;
    int rc = ora_swiglu_backward_values(x, dy, w, T, H, g);
    if (!rc) rc = ora_cast_rows_f32(g, T, 2 * H, group, fmt, out, sf);
    free(g);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout options ("DeepSeek开源TileKernels..." §3.1 round_sf,  */
/* use_packed_ue8m0, use_tma_aligned_col_major_sf; "TileKernels 与 DeepGEMM  */
/* 的分界线" §4C)                                                            */
/* ------------------------------------------------------------------------ */

float ora_pow2_ceil(float s) {
    int e;
    const double f = frexp((double)s, &e);  /* s = f * 2^e, f in [0.5, 1) */
    if (f == 0.5) return s;                 /* already a power of two */
    return (float)ldexp(1.0, e);            /* the next power of two above s */
}

int64_t ora_sf_bytes(int64_t T, int64_t G, int flags) {
    const int64_t T4 = (T + 3) / 4 * 4;
    const int64_t W = (G + 3) / 4;
    const int packed = (flags & ORA_SF_UE8M0_PACKED) != 0;
    const int cm = (flags & ORA_SF_COL_MAJOR) != 0;
    if (packed) return (cm ? W * T4 : T * W) * 4;
    return (cm ? G * T4 : T * G) * 4;
}

int ora_cast_rows_f32_ex(const float* y, int64_t T, int64_t C, int64_t group, int fmt,
                         int flags, uint8_t* out, void* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || group <= 0 || C % group || (flags & ~15))
        return -1;
    const int reciprocal = (flags & ORA_Q_RECIPROCAL) != 0;
    const int packed = (flags & ORA_SF_UE8M0_PACKED) != 0;
    const int pow2 = packed || (flags & ORA_SF_ROUND_POW2);
    const int cm = (flags & ORA_SF_COL_MAJOR) != 0;
    const int64_t G = C / group;
    const int64_t T4 = (T + 3) / 4 * 4;
    const int64_t W = (G + 3) / 4;
    memset(sf, 0, (size_t)ora_sf_bytes(T, G, flags));
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < G; ++j) {
            const float* v = y + t * C + j * group;
            float s = ora_group_scale(group_absmax(v, group, 1), fmt);
            if (pow2) s = ora_pow2_ceil(s);
            if (reciprocal)
                encode_group_reciprocal(v, group, s, fmt, out + t * C + j * group);
            else
                encode_group(v, group, 1, s, fmt, out + t * C + j * group, 1);
            if (packed) {
                uint32_t bits;
                memcpy(&bits, &s, sizeof bits);
                const int64_t word = cm ? (j / 4) * T4 + t : t * W + j / 4;
                ((uint8_t*)sf)[word * 4 + j % 4] = (uint8_t)((bits >> 23) & 0xFF);
            } else {
                ((float*)sf)[cm ? j * T4 + t : t * G + j] = s;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Per-channel and per-block casts, cast back ("TileKernels 与 DeepGEMM 的    */
/* 分界线" §2 operator table: per_channel_cast (+transpose), per_block_cast, */
/* cast_back)                                                                */
/* ------------------------------------------------------------------------ */

int ora_per_channel_cast(const uint16_t* x, int64_t T, int64_t C, int64_t group, int fmt,
                         int transpose, uint8_t* out, float* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || group <= 0 || T % group) return -1;
    const int64_t B = T / group;
    float* v = (float*)malloc((size_t)(group > 0 ? group : 1) * sizeof(float));
    if (!v) return -1;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t b = 0; b < B; ++b) {
            for (int64_t i = 0; i < group; ++i)
                v[i] = ora_bf16_to_f32(x[(b * group + i) * C + c]);
            if (transpose) {
                /* codes of channel c land contiguously in row c of [C, T] */
                sf[c * B + b] = cast_group(v, group, 1, fmt, out + c * T + b * group, 1);
            } else {
                /* codes stay at [t, c] */
                sf[b * C + c] = cast_group(v, group, 1, fmt, out + (b * group) * C + c, C);
            }
        }
    }
    free(v);
    return 0;
}

int ora_per_block_cast(const uint16_t* x, int64_t T, int64_t C, int64_t block, int fmt,
                       uint8_t* out, float* sf) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || block <= 0 || C % block) return -1;
    const int64_t RB = (T + block - 1) / block;
    const int64_t CB = C / block;
    float* v = (float*)malloc((size_t)(block * block > 0 ? block * block : 1) * sizeof(float));
    if (!v) return -1;
    for (int64_t rb = 0; rb < RB; ++rb) {
        const int64_t r0 = rb * block;
        const int64_t rows = (T - r0 < block) ? T - r0 : block;
        for (int64_t cb = 0; cb < CB; ++cb) {
            /* the block's rows, one after the other */
            for (int64_t r = 0; r < rows; ++r)
                for (int64_t c = 0; c < block; ++c)
                    v[r * block + c] = ora_bf16_to_f32(x[(r0 + r) * C + cb * block + c]);
            const float s = ora_group_scale(group_absmax(v, rows * block, 1), fmt);
            sf[rb * CB + cb] = s;
            for (int64_t r = 0; r < rows; ++r)
                encode_group(v + r * block, block, 1, s, fmt, out + (r0 + r) * C + cb * block, 1);
        }
    }
    free(v);
    return 0;
}

int ora_cast_back(const uint8_t* codes, const float* sf, int64_t T, int64_t C, int64_t gr,
                  int64_t gc, int fmt, float* out) {
    fp8_desc d;
    if (get_desc(fmt, &d) || T < 0 || C < 0 || gr <= 0 || gc <= 0 || C % gc) return -1;
    const int64_t G = C / gc;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            const double v = ora_fp8_decode(codes[t * C + c], fmt);
            const float s = sf[(t / gr) * G + c / gc];
            out[t * C + c] = (float)v * s;   /* decode is exact in binary32 */
        }
    return 0;
}
