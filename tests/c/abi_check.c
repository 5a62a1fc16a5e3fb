/*
 * A plain C client of libtkq.so (test infrastructure): it allocates device
 * buffers with the CUDA runtime, calls tkq_per_token_cast, tkq_swiglu_cast_t
 * and tkq_cast_back through the C ABI on a stream, and compares the plain
 * cast and the cast back bit for bit with the C oracle, and the SwiGLU row
 * scales with the oracle's within 1e-6 relative.  Exit status 0 = all checks
 * passed.  Built against include/tkq.h as strict C11, so it also shows the
 * header is usable from C.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "tkq.h"
#include "tkq_oracle.h"

#define CHECK_CUDA(x)                                                          \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
            return 2;                                                          \
        }                                                                      \
    } while (0)

/* xorshift64*: deterministic test input, bf16 bits of moderate magnitude */
static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint16_t next_bf16(void) {
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    const uint64_t r = rng_state * 0x2545F4914F6CDD1Dull;
    const uint16_t sign_mant = (uint16_t)(r & 0x807Fu);
    const uint16_t expo = (uint16_t)(127 - 12 + (int)((r >> 20) % 20));
    return (uint16_t)(sign_mant | (expo << 7));
}

int main(void) {
    const int64_t T = 257, C = 512, H = 256, G = C / 128;
    const size_t n = (size_t)(T * C);
    uint16_t* x = malloc(n * 2);
    uint8_t* codes = malloc(n);
    uint8_t* ref_codes = malloc(n);
    float* sf = malloc((size_t)(T * G) * 4);
    float* ref_sf = malloc((size_t)(T * G) * 4);
    float* y = malloc(n * 4);
    float* ref_y = malloc(n * 4);
    if (!x || !codes || !ref_codes || !sf || !ref_sf || !y || !ref_y) return 2;
    for (size_t i = 0; i < n; ++i) x[i] = next_bf16();

    void *dx, *dout, *dsf, *dy, *dout_t, *dsf_t;
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    CHECK_CUDA(cudaMalloc(&dx, n * 2));
    CHECK_CUDA(cudaMalloc(&dout, n));
    CHECK_CUDA(cudaMalloc(&dsf, (size_t)(T * G) * 4));
    CHECK_CUDA(cudaMalloc(&dy, n * 4));
    CHECK_CUDA(cudaMemcpyAsync(dx, x, n * 2, cudaMemcpyHostToDevice, stream));

    /* plain per-token cast: bit-exact */
    tkq_status st = tkq_per_token_cast(dx, dout, (float*)dsf, T, C, 128, TKQ_FMT_E4M3, stream);
    if (st != TKQ_OK) { fprintf(stderr, "per_token_cast: %s\n", tkq_status_string(st)); return 1; }
    CHECK_CUDA(cudaMemcpyAsync(codes, dout, n, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(sf, dsf, (size_t)(T * G) * 4, cudaMemcpyDeviceToHost, stream));

    /* cast back to fp32 with the same per-token scales: bit-exact */
    st = tkq_cast_back(dout, (const float*)dsf, dy, T, C, 1, 128, TKQ_FMT_E4M3, TKQ_OUT_F32, stream);
    if (st != TKQ_OK) { fprintf(stderr, "cast_back: %s\n", tkq_status_string(st)); return 1; }
    CHECK_CUDA(cudaMemcpyAsync(y, dy, n * 4, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));

    if (ora_per_token_cast(x, T, C, 128, ORA_E4M3, ref_codes, ref_sf)) return 2;
    if (memcmp(codes, ref_codes, n) || memcmp(sf, ref_sf, (size_t)(T * G) * 4)) {
        fprintf(stderr, "per_token_cast differs from the oracle\n");
        return 1;
    }
    if (ora_cast_back(ref_codes, ref_sf, T, C, 1, 128, ORA_E4M3, ref_y)) return 2;
    if (memcmp(y, ref_y, n * 4)) {
        fprintf(stderr, "cast_back differs from the oracle\n");
        return 1;
    }

    /* SwiGLU + transposed cast of the same bytes read as [T', 2H] (T' = 256):
     * row scales within 1e-6 of the oracle's */
    const int64_t Ts = 256;
    CHECK_CUDA(cudaMalloc(&dout_t, (size_t)(Ts * H)));
    CHECK_CUDA(cudaMalloc(&dsf_t, (size_t)(H * (Ts / 128)) * 4));
    st = tkq_swiglu_cast_t(dx, NULL, dout, (float*)dsf, dout_t, (float*)dsf_t, Ts, H, 128,
                           TKQ_FMT_E4M3, stream);
    if (st != TKQ_OK) { fprintf(stderr, "swiglu_cast_t: %s\n", tkq_status_string(st)); return 1; }
    CHECK_CUDA(cudaMemcpyAsync(sf, dsf, (size_t)(Ts * (H / 128)) * 4, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    if (ora_swiglu_cast(x, NULL, Ts, H, 128, ORA_E4M3, ref_codes, ref_sf)) return 2;
    for (int64_t i = 0; i < Ts * (H / 128); ++i)
        if (fabs((double)sf[i] - (double)ref_sf[i]) > 1e-6 * fabs((double)ref_sf[i])) {
            fprintf(stderr, "swiglu scale %lld: %g vs %g\n", (long long)i, sf[i], ref_sf[i]);
            return 1;
        }

    uint32_t flags = 0;
    if (tkq_read_device_status(&flags, 1) != TKQ_OK || flags) return 1;
    cudaFree(dx); cudaFree(dout); cudaFree(dsf); cudaFree(dy); cudaFree(dout_t); cudaFree(dsf_t);
    cudaStreamDestroy(stream);
    printf("abi_check: OK (tkq_version %d)\n", tkq_version());
    return 0;
}
