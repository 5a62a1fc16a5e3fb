// tkq_device.cuh -- device building blocks shared by the quantization kernels.
//
// Everything here is per-element or per-group arithmetic of the per-token-group
// FP8 cast described in "DeepSeek开源TileKernels：用Python写的GPU算子逼近硬件
// 性能上限" (itsolotime.com) §3.1-§3.3:
//   scale  s = fl32(max(amax, 1e-4) / fmt_max)
//   code   = saturating RNE FP8 code of fl32(y / s)
//   SwiGLU y = (g / (1 + exp(-g))) * u [* w], binary32 steps.
#pragma once

#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tkq_internal.h"

namespace tkq {

constexpr int kFmtE4M3 = 0;
constexpr int kFmtE5M2 = 1;

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<kFmtE4M3> {
    static constexpr float kMax = 448.0f;
    static constexpr float kInvMax = 1.0f / 448.0f;  // rounded to nearest binary32
};
template <>
struct FmtTraits<kFmtE5M2> {
    static constexpr float kMax = 57344.0f;
    static constexpr float kInvMax = 1.0f / 57344.0f;
};

// ---------------------------------------------------------------------------
// access checking (checked build only)
// ---------------------------------------------------------------------------
// Built with -DTKQ_CHECKED, every global load and store of the kernels (all of
// them go through the helpers below; TMA loads are bounded by their tensor
// maps) first checks that the bytes it touches lie inside one of the buffers
// of the current call: its inputs for a load, its outputs for a store.  The
// ABI layer registers those buffers per call and each launcher copies the
// table to its translation unit's copy on the launch stream before the launch.
// An access not wholly inside them is skipped (no fault), sets
// kDeviceOutOfBounds in the device status word and records the first byte of
// the first such access that lies outside the buffers (bit 63 set for a
// store).  It stands in for a memory checker; the checked library is a test
// build, one launch at a time (the table is shared by a translation unit's
// launches).  In the release build the checks compile away.
#ifdef TKQ_CHECKED
static __device__ CheckTable g_check;  // this translation unit's copy

inline cudaError_t upload_checks(cudaStream_t s) {
    return cudaMemcpyToSymbolAsync(g_check, &host_check_table(), sizeof(CheckTable), 0,
                                   cudaMemcpyHostToDevice, s);
}
#else
inline cudaError_t upload_checks(cudaStream_t) { return cudaSuccess; }
#endif

__device__ __forceinline__ bool access_ok(const void* p, unsigned bytes, bool write) {
#ifdef TKQ_CHECKED
    const unsigned long long a = reinterpret_cast<unsigned long long>(p);
    unsigned long long first_out = a;   // first byte of the access outside the buffers
    for (int k = 0; k < g_check.n; ++k)
        if (a >= g_check.lo[k] && a < g_check.hi[k] &&
            (!write || ((g_check.writable >> k) & 1u))) {
            if (a + bytes <= g_check.hi[k]) return true;
            first_out = g_check.hi[k];
        }
    if (g_check.status) atomicOr(g_check.status, kDeviceOutOfBounds);
    if (g_check.bad) atomicCAS(g_check.bad, 0ull, first_out | (write ? (1ull << 63) : 0ull));
    return false;
#else
    (void)p;
    (void)bytes;
    (void)write;
    return true;
#endif
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// Every thread of a cast (launched by launch_pdl, tkq_internal.h) calls
// grid_dependency_launch at entry, which lets the next grid on the stream be
// scheduled (it waits in turn), and grid_dependency_wait before its first
// global load or store, which returns once the grid before it has completed
// and its memory operations are visible.  Between the two a cast issues only
// L2 prefetches (prefetch_l2, tma_prefetch_2d).  Without a preceding PDL
// launch the wait returns at once.
__device__ __forceinline__ void grid_dependency_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A bulk prefetch of `bytes` bytes at p into L2 (p 16-byte aligned, bytes a
// multiple of 16), issued by the calling thread alone.  A prefetch is a hint:
// it changes no value that any load returns, so a kernel may issue it between
// grid_dependency_launch and grid_dependency_wait, while the grid before it
// still runs and may still be writing those bytes (its writes land in L2,
// the point of coherence, after the prefetched lines or instead of them).
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned bytes) {
    if (!access_ok(p, bytes, false)) return;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// memory access
// ---------------------------------------------------------------------------

// 16-byte streaming load of read-only input: not kept in L1 (each byte is read
// once by this kernel).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r = make_uint4(0, 0, 0, 0);
    if (!access_ok(p, 16, false)) return r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Read-only loads through the non-coherent path (small per-row operands).
__device__ __forceinline__ float ld_ro(const float* p) {
    return access_ok(p, 4, false) ? __ldg(p) : 0.0f;
}
__device__ __forceinline__ float4 ld_ro(const float4* p) {
    return access_ok(p, 16, false) ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Streaming stores (.cs: the output is not read again by this kernel).
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) {
    if (!access_ok(p, 8, true)) return;
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
    if (!access_ok(p, 16, true)) return;
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream_u32(uint32_t* p, uint32_t v) {
    if (!access_ok(p, 4, true)) return;
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_stream(float* p, float v) {
    if (!access_ok(p, 4, true)) return;
    asm volatile("st.global.cs.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Plain stores and the counter update, checked the same way.
__device__ __forceinline__ void st_plain(uint8_t* p, uint8_t v) {
    if (access_ok(p, 1, true)) *p = v;
}
__device__ __forceinline__ void st_plain(float* p, float v) {
    if (access_ok(p, 4, true)) *p = v;
}
__device__ __forceinline__ void st_plain(float4* p, float4 v) {
    if (access_ok(p, 16, true)) *p = v;
}
__device__ __forceinline__ void atomic_add_count(unsigned long long* p, unsigned long long v) {
    if (access_ok(p, 8, true)) atomicAdd(p, v);
}

// ---------------------------------------------------------------------------
// bf16 -> fp32 (exact): a bf16 is the upper half of a binary32
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight bf16 packed in a uint4 -> eight floats, element order preserved.
__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x);
    v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z);
    v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

// ---------------------------------------------------------------------------
// scale and quotient
// ---------------------------------------------------------------------------

// s = fl32(max(amax, 1e-4) / fmt_max) and the correctly rounded reciprocal
// inv = fl32(1 / s).  The division is a product by c = fl32(1 / fmt_max) with
// one FMA residual correction (Markstein): q0 = a*c, r = a - q0*fmt_max,
// s = q0 + r*c.  For every binary32 a >= 1e-4 this equals the IEEE quotient
// (checked exhaustively for both formats: all 2.37e9 such a).
template <int FMT>
__device__ __forceinline__ void group_scale(float amax, float& s, float& inv) {
    const float a = fmaxf(amax, 1e-4f);
    const float q0 = __fmul_rn(a, FmtTraits<FMT>::kInvMax);
    const float r = __fmaf_rn(-q0, FmtTraits<FMT>::kMax, a);
    s = __fmaf_rn(r, FmtTraits<FMT>::kInvMax, q0);
    inv = __frcp_rn(s);
}

// fl32(y / s) from inv = fl32(1/s): the product y*inv is within one ulp of the
// quotient, and one Newton-Raphson residual step (Markstein's correction: the
// residual q0*s - y is exact with an FMA, and q0 - residual*inv rounds to the
// correctly rounded quotient) recovers the IEEE result.  It holds whenever the
// residual is a normal binary32, i.e. for every quotient large enough to give
// a non-zero FP8 code; smaller quotients encode to a signed zero either way.
// Taking the residual as q0*s - y (not y - q0*s) keeps the sign of zero: for
// y = -0, q0 = -0, the residual is +0 and -0 + -0 = -0.  (Checked on 8.8e7
// random pairs including signed zeros and subnormal y: same value and sign as
// the IEEE quotient.)
__device__ __forceinline__ float quotient(float y, float s, float inv) {
    const float q0 = __fmul_rn(y, inv);
    const float res = __fmaf_rn(q0, s, -y);
    return __fmaf_rn(-res, inv, q0);
}


// ---------------------------------------------------------------------------
// scale-factor layouts (the TKQ_SF_* flags of tkq.h)
// ---------------------------------------------------------------------------

// Where the scales of a launch go: a [rows, groups] matrix of scales in the
// layout the flags select.
struct SfLayout {
    unsigned flags;  // TKQ_SF_ROUND_POW2 | TKQ_SF_UE8M0_PACKED | TKQ_SF_COL_MAJOR
                     // | TKQ_Q_RECIPROCAL
    int groups;      // groups per row (G)
    int words;       // ceil(G / 4), packed layouts
    int64_t rows4;   // rows rounded up to a multiple of 4, column-major layouts
};
constexpr unsigned kSfRoundPow2 = 1u, kSfPacked = 2u, kSfColMajor = 4u, kQReciprocal = 8u;

// Option sets a kernel instance may fix at compile time (its SFC template
// argument): none, the two scale layouts a TMA-fed FP8 GEMM reads (UE8M0
// packed column-major, fp32 column-major), the reciprocal reading alone, or
// kSfcRuntime for flags read from the launch.  A flag test that is a run-time
// branch inside a kernel's loop measurably slows the latency-bound ones.
constexpr unsigned kSfcNone = 0u;
constexpr unsigned kSfcUe8m0ColMajor = kSfRoundPow2 | kSfPacked | kSfColMajor;
constexpr unsigned kSfcF32ColMajor = kSfColMajor;
constexpr unsigned kSfcReciprocal = kQReciprocal;
constexpr unsigned kSfcRuntime = ~0u;

// The instance for sf_flags: packed scales are powers of two, and with
// power-of-two scales the reciprocal reading is the quotient; `recip` says
// whether the kernel distinguishes the reciprocal reading at all.
__host__ __device__ inline unsigned sfc_of(unsigned sf_flags, bool recip) {
    unsigned f = sf_flags & (kSfRoundPow2 | kSfPacked | kSfColMajor | kQReciprocal);
    if (!recip) f &= ~kQReciprocal;
    if (f & kSfPacked) f |= kSfRoundPow2;
    if (f & kSfRoundPow2) f &= ~kQReciprocal;
    if (f == kSfcNone || f == kSfcUe8m0ColMajor || f == kSfcF32ColMajor ||
        f == kSfcReciprocal)
        return f;
    return kSfcRuntime;
}

// The scale rounded up to a power of two, s = 2^ceil(log2 s) (the mantissa
// bits dropped and the exponent raised when any were set), and its reciprocal,
// exact: 2^-k has the biased exponent 254 minus that of 2^k.
__device__ __forceinline__ void pow2_scale(float& s, float& inv) {
    uint32_t b = __float_as_uint(s);
    if (b & 0x007FFFFFu) b = (b & 0x7F800000u) + 0x00800000u;
    s = __uint_as_float(b);
    inv = __uint_as_float((254u << 23) - b);
}

// Scale of group gj of `row` in the chosen layout.  Padding rows of the
// column-major layouts (rows <= row < rows4) get 0, and the unused bytes of a
// row's last packed word are zeroed by the lane of its last group.
__device__ __forceinline__ void store_scale(void* sf, const SfLayout& lay, int64_t row,
                                            bool live, int gj, float sc) {
    const bool cm = lay.flags & kSfColMajor;
    if (!live && !(cm && row < lay.rows4)) return;
    if (lay.flags & kSfPacked) {
        const uint8_t byte = live ? static_cast<uint8_t>(__float_as_uint(sc) >> 23) : 0;
        const int64_t word = cm ? static_cast<int64_t>(gj >> 2) * lay.rows4 + row
                                : row * lay.words + (gj >> 2);
        uint8_t* p = static_cast<uint8_t*>(sf) + word * 4;
        st_plain(p + (gj & 3), byte);
        if (gj == lay.groups - 1)
            for (int k = (gj & 3) + 1; k < 4; ++k) st_plain(p + k, uint8_t{0});
    } else {
        const int64_t idx = cm ? static_cast<int64_t>(gj) * lay.rows4 + row
                               : row * lay.groups + gj;
        st_plain(static_cast<float*>(sf) + idx, live ? sc : 0.0f);
    }
}

// ---------------------------------------------------------------------------
// Packed binary32 pairs: sm_100+ add / mul / fma .f32x2 perform two
// independent IEEE operations per instruction, each rounded to nearest even
// like the scalar one, so results are bit-identical to the scalar forms while
// half as many instructions issue.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// quotient() of two elements with the packed pair instructions: the product
// and the correction are packed, the residual stays scalar (it needs -y);
// fma(res, -inv, q0) is the scalar fma(-res, inv, q0) exactly.  Bit-identical.
__device__ __forceinline__ float2 quotient2(float2 y, float2 s, float2 inv) {
    const float2 q0 = mul2(y, inv);
    const float2 res = make_float2(__fmaf_rn(q0.x, s.x, -y.x), __fmaf_rn(q0.y, s.y, -y.y));
    return fma2(res, make_float2(-inv.x, -inv.y), q0);
}

// ---------------------------------------------------------------------------
// FP8 packing: cvt.rn.satfinite converts two binary32 values to two FP8 codes
// with round-to-nearest-even and saturation to the largest finite value.  The
// first source operand lands in the upper byte, so operands are swapped to
// keep element order in memory (byte 0 = first element).
// ---------------------------------------------------------------------------

template <int FMT>
__device__ __forceinline__ uint32_t pack4(float a0, float a1, float a2, float a3) {
    uint32_t r;
    if constexpr (FMT == kFmtE4M3) {
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r)
            : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    } else {
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r)
            : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    }
    return r;
}

// Codes of four values (exact quotients) with per-value scales, packed
// little-endian.
template <int FMT>
__device__ __forceinline__ uint32_t quantize4_each(const float* v, const float* s,
                                                   const float* inv) {
    const float2 a = quotient2(make_float2(v[0], v[1]), make_float2(s[0], s[1]),
                               make_float2(inv[0], inv[1]));
    const float2 b = quotient2(make_float2(v[2], v[3]), make_float2(s[2], s[3]),
                               make_float2(inv[2], inv[3]));
    return pack4<FMT>(a.x, a.y, b.x, b.y);
}

// Codes of eight values sharing one group scale, packed little-endian.
template <int FMT>
__device__ __forceinline__ uint2 quantize8(const float* v, float s, float inv) {
    const float2 s2 = make_float2(s, s), i2 = make_float2(inv, inv);
    float q[8];
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const float2 r = quotient2(make_float2(v[k], v[k + 1]), s2, i2);
        q[k] = r.x;
        q[k + 1] = r.y;
    }
    return make_uint2(pack4<FMT>(q[0], q[1], q[2], q[3]), pack4<FMT>(q[4], q[5], q[6], q[7]));
}

__device__ __forceinline__ float absmax8(const float* v) {
    float m = fabsf(v[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    return m;
}

// ---------------------------------------------------------------------------
// SwiGLU, y = silu(g) * u with silu(g) = g / (1 + exp(-g)), g the gate and u
// the up half ("DeepSeek开源TileKernels..." §3.3), with the SM's
// transcendental unit:
//   exp(-g) = 2^(-g * log2 e)      hardware base-2 exponential (ex2.approx)
//   g / (1 + exp(-g))              hardware reciprocal (rcp.approx) times g
// Error against exactly rounded binary32 steps: the product t = -g * log2 e is
// rounded (absolute error <= |t| 2^-24 with the rounded constant), which gives
// exp(-g) a relative error of about (1.04 |t| + 2) ulp; it enters the result
// scaled by exp(-g) / (1 + exp(-g)) < 1/2 for g > 0.  Rounded reciprocal and the
// two products add about 2 ulp.  So y is within a few ulp wherever |y| is not
// tiny relative to |g u| (g > -6 or so), which covers the element that sets a
// group's scale; the parity tolerance is 1e-6 relative on scales (about 16 ulp)
// and one FP8 step on codes.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// swiglu of two elements with the packed pair instructions (bit-identical).
__device__ __forceinline__ float2 swiglu2(float2 g, float2 u) {
    const float2 t = mul2(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    const float2 den = add2(make_float2(1.0f, 1.0f), make_float2(ex2_approx(t.x), ex2_approx(t.y)));
    return mul2(mul2(g, make_float2(rcp_approx(den.x), rcp_approx(den.y))), u);
}

// ---------------------------------------------------------------------------
// SwiGLU clamp (gate <= c, -c <= up <= c) on packed bf16 pairs
// ---------------------------------------------------------------------------
// When the bound c is itself a bf16 value the clamp can run on the raw input
// pairs before they are widened, two elements per instruction: min / max
// return one of their operands (the other one when an operand is NaN, as
// fminf / fmaxf do), so they give exactly the values the fp32 clamp gives on
// the exact widening; and an input differs from its clamped copy under the
// ordered compare (false for NaN, as g > c and |u| > c are) exactly when it
// lies beyond the bound.

// c in both halves of a word, or 0 when c (finite, > 0) is not a bf16 value.
__host__ __device__ inline uint32_t bf16x2_bound(float c) {
    uint32_t b;
    memcpy(&b, &c, sizeof b);
    return (b & 0xFFFFu) ? 0u : (b >> 16) * 0x00010001u;
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t w) {
    return *reinterpret_cast<const __nv_bfloat162*>(&w);
}
__device__ __forceinline__ uint32_t as_word(__nv_bfloat162 v) {
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Clamps the gate pair g and the up pair u in place (c2 = bf16x2_bound(c))
// and counts the values the clamp changed into n.  The up clamp is one
// min.xorsign.abs: magnitude min(|u|, c), sign of u xor sign of c (+), which
// is clamp(u, -c, c) for every u that is not NaN, signed zeros and infinities
// included.  The count: each not-equal compare gives a 32-bit mask with
// 0xFFFF in every half whose value changed, and n adds both masks (one
// three-input integer add).  Modulo 2^32 a low-half mask is 2^16 - 1 and a
// high-half mask -2^16, so n = 2^16 (L - H) - L for L low-half and H
// high-half changes; clamped_total recovers L + H while both stay below 2^15
// (callers convert n after at most 16 pairs).
__device__ __forceinline__ void clamp_pairs_bf16(uint32_t& g, uint32_t& u, uint32_t c2,
                                                 uint32_t& n) {
    const __nv_bfloat162 gc = __hmin2(as_bf162(g), as_bf162(c2));
    const uint32_t gw = as_word(gc);
    uint32_t uw, mg, mu;
    asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(uw) : "r"(u), "r"(c2));
    asm("set.ne.u32.bf16x2 %0, %1, %2;" : "=r"(mg) : "r"(g), "r"(gw));
    asm("set.ne.u32.bf16x2 %0, %1, %2;" : "=r"(mu) : "r"(u), "r"(uw));
    n += mg + mu;
    g = gw;
    u = uw;
}

// The same clamp with the count kept as two bf16 halves (each compare gives
// 1.0 or 0.0 per half, summed exactly up to 256); the transposed cast uses
// this form, measured faster there than the integer count.
__device__ __forceinline__ void clamp_pairs_bf16(uint32_t& g, uint32_t& u, uint32_t c2,
                                                 __nv_bfloat162& n) {
    const __nv_bfloat162 gb = as_bf162(g), ub = as_bf162(u);
    const __nv_bfloat162 gc = __hmin2(gb, as_bf162(c2));
    uint32_t uw;
    asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(uw) : "r"(u), "r"(c2));
    const __nv_bfloat162 uc = as_bf162(uw);
    g = as_word(gc);
    u = uw;
    n = __hadd2(n, __hne2(gb, gc));
    n = __hadd2(n, __hne2(ub, uc));
}
__device__ __forceinline__ uint32_t clamped_total(__nv_bfloat162 n) {
    return static_cast<uint32_t>(__low2float(n) + __high2float(n));
}

// The number of changes a clamp_pairs_bf16 count n holds: L = -n mod 2^16,
// L - H = (n + L) / 2^16 as a signed value, L + H = 2 L - (L - H).
__device__ __forceinline__ uint32_t clamped_total(uint32_t n) {
    const uint32_t lo = (0u - n) & 0xFFFFu;
    const int32_t diff = static_cast<int32_t>(n + lo) >> 16;
    return 2u * lo - static_cast<uint32_t>(diff);
}

// Gradient of y = silu(g) * u with respect to g and u, scaled by the upstream
// gradient d (the derivative of the SwiGLU of the same page; it gives no
// formula, this is the textbook one), for two elements at a time with the
// packed pair instructions (the transcendental steps and the bound below stay
// scalar):
//   sigma = 1 / (1 + e), e = exp(-g);  1 - sigma = e * sigma (no cancellation)
//   dg = d * u * sigma * (1 + g * (1 - sigma)),  du = d * g * sigma.
// e * sigma is bounded by 1.  Where e overflows (g < -88.7), sigma = 0 and
// e * sigma = inf * 0 is NaN, which fminf turns into 1; both gradients are
// then exactly 0, which is what sigma -> 0 makes them.  (Clamping the exponent
// instead would leave sigma at its smallest normal value, so that dg grew like
// 2^-126 * g for very negative g.)  Elsewhere the bound changes at most a
// product that rounded above 1.
__device__ __forceinline__ void swiglu_grad2(float2 g, float2 u, float2 d, float2& dg,
                                             float2& du) {
    const float2 t = mul2(g, make_float2(-1.4426950408889634f, -1.4426950408889634f));
    const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    const float2 den = add2(make_float2(1.0f, 1.0f), e);
    const float2 sig = make_float2(rcp_approx(den.x), rcp_approx(den.y));
    const float2 es = mul2(e, sig);
    const float2 one_minus_sig = make_float2(fminf(es.x, 1.0f), fminf(es.y, 1.0f));
    const float2 dsilu = mul2(sig, fma2(g, one_minus_sig, make_float2(1.0f, 1.0f)));
    dg = mul2(mul2(d, u), dsilu);
    du = mul2(d, mul2(g, sig));
}

// Four bf16 packed in a uint2 -> four floats, element order preserved.
__device__ __forceinline__ void unpack4(const uint2& q, float* v) {
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x);
    v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
}

// Codes of four values sharing one group scale, packed little-endian.
template <int FMT>
__device__ __forceinline__ uint32_t quantize4(const float* v, float s, float inv) {
    const float2 s2 = make_float2(s, s), i2 = make_float2(inv, inv);
    const float2 a = quotient2(make_float2(v[0], v[1]), s2, i2);
    const float2 b = quotient2(make_float2(v[2], v[3]), s2, i2);
    return pack4<FMT>(a.x, a.y, b.x, b.y);
}

// The SwiGLU kernels quantize y * inv, the product by the rounded reciprocal of
// the scale, as the TileKernels per-token kernel does (x * sf_inv, "DeepSeek开源
// TileKernels..." §3.2, step 4).  It is within one ulp of y / s, and y itself
// carries a few ulp of exp error.  The exact quotient (quotient2) was measured
// in all three SwiGLU kernels: free in the flat stream, +2 % in the TMA ring,
// +6 to +17 % in the transposed kernel, whose rows must equal the row cast's;
// the plain casts keep `quotient` and are bit-exact.
template <int FMT>
__device__ __forceinline__ uint32_t quantize4_mul(const float* v, float inv) {
    const float2 i2 = make_float2(inv, inv);
    const float2 a = mul2(make_float2(v[0], v[1]), i2);
    const float2 b = mul2(make_float2(v[2], v[3]), i2);
    return pack4<FMT>(a.x, a.y, b.x, b.y);
}

template <int FMT>
__device__ __forceinline__ uint2 quantize8_mul(const float* v, float inv) {
    return make_uint2(quantize4_mul<FMT>(v, inv), quantize4_mul<FMT>(v + 4, inv));
}

}  // namespace tkq
