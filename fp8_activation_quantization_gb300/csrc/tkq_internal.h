// tkq_internal.h -- launchers behind the C ABI (include/tkq.h).  Arguments are
// validated by the ABI layer before these are called.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tkq {

// Tensor map of a row-major bf16 matrix [rows, cols] (row stride cols * 2
// bytes) for 2-D TMA boxes of box_rows x box_cols elements, no swizzle,
// out-of-range elements read as zero.  The driver entry point is looked up
// through the runtime once.  Returns false if the driver call is unavailable
// or rejects the arguments.
bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                    uint32_t box_cols, uint32_t box_rows);

// Number of SMs of the current device (cached per device; the environment
// variable TKQ_NUM_SMS overrides it for grid sizing experiments).
int num_sms();

// Address of the library's device status word on the current device (bit
// kDeviceTimeout: a bounded wait inside a kernel gave up).  Resolved once per
// device with cudaGetSymbolAddress.
unsigned int* device_status_word();

// Access checking of the checked build (-DTKQ_CHECKED; see tkq_device.cuh):
// the buffers of the current call, inputs and outputs, as address ranges.
constexpr uint32_t kDeviceOutOfBounds = 2u;  // status-word bit: an access was refused
constexpr int kCheckMax = 8;

struct CheckTable {
    unsigned long long lo[kCheckMax], hi[kCheckMax];  // [lo, hi) per buffer
    unsigned writable;                                // bit k: buffer k is an output
    int n;
    unsigned int* status;     // the library's device status word
    unsigned long long* bad;  // first refused address (bit 63: a store)
};

// The calling host thread's table for its current call (filled by the ABI
// layer, copied to the device by each launcher).  Checked build only.
CheckTable& host_check_table();

// Persistent grid: min(blocks needed, SMs x resident blocks per SM).
int persistent_grid(const void* kernel, int threads, size_t smem, int64_t blocks_needed);

// How many units of its walk each warp of a flat stream (token_cast.cu,
// swiglu_flat.cu), or each CTA of cast back, sends to L2 before it waits for
// the grid before it: a CTA of the next launch starts on an SM as soon as a
// CTA of the draining one exits there, so these prefetches fill the DRAM time
// the drain leaves idle.  Measured back to back on one GB300 (four CTAs per
// SM for the plain cast): one unit took the plain cast of [8192, 7168] from
// 29.44 to 29.15 us and the SwiGLU cast of [16384, 4096] from 27.07 to
// 26.38 us, two units less (29.26, 26.57 us); on an input of a few MB, where
// every warp has one or two units, prefetching them all took the plain cast of
// [1024, 4096] from 3.67 to 2.7-2.8 us.
inline int prologue_prefetch_units(int64_t input_bytes) {
    return input_bytes <= (int64_t{16} << 20) ? 4 : 1;
}

// Launch of one of the library's casts, with programmatic dependent launch
// allowed when `allow`: its grid may then be scheduled while the kernel before
// it on the stream is still draining, once every CTA of that kernel has
// started (the casts signal that at entry, grid_dependency_launch in
// tkq_device.cuh).  Each cast then waits (grid_dependency_wait) for the
// previous grid to complete, its memory visible, before any global load or
// store.  What overlaps is the launch, the CTAs' start-up and the L2
// prefetches the casts issue before that wait (prologue_prefetch_units and the
// rings' first boxes), which change no value any load returns.  After a kernel
// that does not signal, or after a copy, the launch is ordered as usual.
// Measured back to back, this takes 2.5-3.5 % off the ~30 us flat casts and,
// with the prefetches, 4.4 % off the transposed per-channel cast (56.5 to
// 54.0 us); it made the SwiGLU backward cast slower (152.0 against 154.5 us
// with the prefetches, 156.1 without), whose launcher passes allow = false.
// Returns the launch's error.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), int grid, int block, size_t smem,
                              cudaStream_t stream, bool allow, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = allow ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// sf_flags: TKQ_SF_* options of include/tkq.h (0 = row-major fp32 scales).
cudaError_t launch_per_token_cast(const void* x, void* out, void* sf, int64_t T, int64_t C,
                                  int fmt, unsigned sf_flags, cudaStream_t stream);

// The fp32 SwiGLU values y [T, H] the SwiGLU casts quantize (diagnostic).
cudaError_t launch_swiglu_values(const void* x, const float* w, float* y, int64_t T, int64_t H,
                                 cudaStream_t stream);

// The fp32 gradients [dg | du] ([T, 2H]) the SwiGLU backward cast quantizes
// (diagnostic).
cudaError_t launch_swiglu_backward_values(const void* x, const void* dy, const float* w, float* y,
                                          int64_t T, int64_t H, cudaStream_t stream);

// FP8 codes of n fp32 values, unscaled (diagnostic; n % 4 == 0).
cudaError_t launch_fp8_encode(const float* x, void* out, int64_t n, int fmt,
                              cudaStream_t stream);

// The per-token cast of a row-major fp32 [T, C] matrix.
cudaError_t launch_per_token_cast_f32(const float* x, void* out, void* sf, int64_t T, int64_t C,
                                      int fmt, unsigned sf_flags, cudaStream_t stream);

// clamp: null (no clamp) or the SwiGLU clamp bound c > 0; clamp_count (may be
// null) receives the number of clamped input values by atomic addition.
cudaError_t launch_swiglu_cast(const void* x, const float* w, void* out, void* sf, int64_t T,
                               int64_t H, int fmt, unsigned sf_flags, const float* clamp,
                               unsigned long long* clamp_count, cudaStream_t stream);

// The same operation as a flat stream (swiglu_flat.cu), bit-identical; the
// kernel for short launches.
cudaError_t launch_swiglu_cast_flat(const void* x, const float* w, void* out, void* sf, int64_t T,
                                    int64_t H, int fmt, unsigned sf_flags, const float* clamp,
                                    unsigned long long* clamp_count, cudaStream_t stream);

// Whether a SwiGLU forward cast of [T, 2H] runs as the flat stream: yes
// without a routing weight, and with one when its bf16 input is at most
// kSwigluFlatMaxBytes (measured: the flat stream is faster at every size
// without a weight, and with one up to 320 MiB of input; the two tie at
// 384 MiB and the ring is faster above).  The environment variable
// TKQ_SWIGLU_KERNEL ("flat" or "ring") overrides this for tests and
// measurements.
constexpr int64_t kSwigluFlatMaxBytes = int64_t{384} << 20;
bool swiglu_flat_chosen(int64_t T, int64_t H, bool weighted);

cudaError_t launch_swiglu_backward_cast(const void* x, const void* dy, const float* w, void* out,
                                        void* sf, int64_t T, int64_t H, int fmt,
                                        unsigned sf_flags, cudaStream_t stream);

// sf_flags: TKQ_SF_* layout of both the row scales [T, H/128] and the column
// scales [H, T/128] (0 = row-major fp32).
cudaError_t launch_swiglu_cast_t(const void* x, const float* w, void* out, float* sf,
                                 void* out_t, float* sf_t, int64_t T, int64_t H, int fmt,
                                 unsigned sf_flags, const float* clamp,
                                 unsigned long long* clamp_count, cudaStream_t stream);

// Per-channel cast (128-token groups; T % 128 == 0): codes [T, C] with sf
// [T/128, C], or codes [C, T] with sf [C, T/128] when transpose.
cudaError_t launch_per_channel_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                    int fmt, bool transpose, cudaStream_t stream);

// Per-block cast (128 x 128 blocks, ragged T): codes [T, C], sf [ceil(T/128), C/128].
cudaError_t launch_per_block_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                  int fmt, cudaStream_t stream);

// Cast back: out (fp32, or bf16 when out_bf16) = decode(code) * scale, with
// scales of gr x gc groups (1x128, 128x1 or 128x128).
cudaError_t launch_cast_back(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                             int gr, int gc, int fmt, bool out_bf16, cudaStream_t stream);

}  // namespace tkq
