// tkq_api.cu -- the C ABI of libtkq.so (declared in include/tkq.h): argument
// validation, status codes and dispatch to the kernel launchers.  Nothing here
// allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <initializer_list>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "../../include/tkq.h"
#include "tkq_async.cuh"
#include "tkq_internal.h"

// The library's device status word (one per device): kernels OR status bits
// into it (tkq::kDeviceTimeout when a bounded wait gave up); the host reads and
// clears it with tkq_read_device_status.
__device__ unsigned int g_tkq_device_status;
// First address an access check refused (checked build; bit 63: a store).
__device__ unsigned long long g_tkq_bad_address;

namespace tkq {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];  // 0 = not yet queried
std::atomic<unsigned int*> g_status_ptr[kMaxDevices];
std::atomic<unsigned long long*> g_bad_ptr[kMaxDevices];

// One CTA waits on an mbarrier that nothing ever arrives on, so its bounded
// wait must give up after limit_ns and record a timeout in the status word.
__global__ void selftest_wait_kernel(unsigned int* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort, status, limit_ns);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range span(const void* p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + static_cast<uintptr_t>(bytes)};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
}  // namespace

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (const char* env = std::getenv("TKQ_NUM_SMS")) {
        const int v = std::atoi(env);
        if (v > 0) return v;
    }
    if (dev < kMaxDevices) {
        int v = g_sms[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 1;
    if (dev < kMaxDevices) g_sms[dev].store(v, std::memory_order_relaxed);
    return v;
}

bool swiglu_flat_chosen(int64_t T, int64_t H, bool weighted) {
    if (const char* env = std::getenv("TKQ_SWIGLU_KERNEL")) {
        if (std::strcmp(env, "flat") == 0) return true;
        if (std::strcmp(env, "ring") == 0) return false;
    }
    return !weighted || T * 2 * H * 2 <= kSwigluFlatMaxBytes;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}
}  // namespace

namespace {
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, int64_t elem_bytes, const void* base,
               int64_t cols, int64_t rows, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * elem_bytes)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t cols, int64_t rows,
                    uint32_t box_cols, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, box_cols,
                     box_rows);
}


unsigned int* device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    if (dev < kMaxDevices) {
        unsigned int* p = g_status_ptr[dev].load(std::memory_order_acquire);
        if (p) return p;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tkq_device_status) != cudaSuccess) return nullptr;
    if (dev < kMaxDevices)
        g_status_ptr[dev].store(static_cast<unsigned int*>(p), std::memory_order_release);
    return static_cast<unsigned int*>(p);
}

CheckTable& host_check_table() {
    thread_local CheckTable table{};
    return table;
}

namespace {
unsigned long long* bad_address_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    if (dev < kMaxDevices) {
        unsigned long long* p = g_bad_ptr[dev].load(std::memory_order_acquire);
        if (p) return p;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tkq_bad_address) != cudaSuccess) return nullptr;
    if (dev < kMaxDevices)
        g_bad_ptr[dev].store(static_cast<unsigned long long*>(p), std::memory_order_release);
    return static_cast<unsigned long long*>(p);
}

// The buffers of the call about to launch, for the checked build's access
// checks (a no-op otherwise): inputs may be read, outputs read and written.
// Empty ranges (an absent optional buffer) are skipped.  The environment
// variable TKQ_CHECK_WITHHOLD=n (checked build only) leaves the last n bytes of
// every output out of the table, so that the kernels' stores there are refused
// and reported: the test of the checks themselves, with no access outside any
// allocation.
void register_call(std::initializer_list<Range> inputs, std::initializer_list<Range> outputs) {
#ifdef TKQ_CHECKED
    CheckTable& t = host_check_table();
    t = CheckTable{};
    uint64_t withhold = 0;
    if (const char* env = std::getenv("TKQ_CHECK_WITHHOLD"))
        withhold = std::strtoull(env, nullptr, 10);
    auto add = [&t](uintptr_t lo, uintptr_t hi, bool out) {
        if (hi <= lo || t.n >= kCheckMax) return;
        t.lo[t.n] = lo;
        t.hi[t.n] = hi;
        if (out) t.writable |= 1u << t.n;
        ++t.n;
    };
    for (const Range& r : inputs) add(r.lo, r.hi, false);
    for (const Range& r : outputs)
        add(r.lo, r.hi - r.lo > withhold ? r.hi - withhold : r.lo, true);
    t.status = device_status_word();
    t.bad = bad_address_word();
#else
    (void)inputs;
    (void)outputs;
#endif
}

// Per (kernel, device, threads, smem): resident blocks per SM.  The first
// launch on a device raises the kernel's dynamic shared-memory limit and asks
// the occupancy calculator; later launches reuse the answer, which keeps both
// calls off the per-launch host path.
struct OccKey {
    const void* kernel;
    int dev, threads;
    size_t smem;
    bool operator==(const OccKey& o) const {
        return kernel == o.kernel && dev == o.dev && threads == o.threads && smem == o.smem;
    }
};
struct OccKeyHash {
    size_t operator()(const OccKey& k) const {
        return std::hash<const void*>()(k.kernel) ^ (static_cast<size_t>(k.dev) << 1) ^
               (static_cast<size_t>(k.threads) << 8) ^ (k.smem << 20);
    }
};
std::mutex g_occ_mutex;
std::unordered_map<OccKey, int, OccKeyHash> g_occ;
}  // namespace

int persistent_grid(const void* kernel, int threads, size_t smem, int64_t blocks_needed) {
    int dev = 0;
    cudaGetDevice(&dev);
    const OccKey key{kernel, dev, threads, smem};
    int per_sm = 0;
    {
        std::lock_guard<std::mutex> lock(g_occ_mutex);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) per_sm = it->second;
    }
    if (per_sm == 0) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
                cudaSuccess ||
            per_sm <= 0)
            per_sm = 1;
        std::lock_guard<std::mutex> lock(g_occ_mutex);
        g_occ[key] = per_sm;
    }
    const int64_t cap = static_cast<int64_t>(num_sms()) * per_sm;
    const int64_t g = blocks_needed < cap ? blocks_needed : cap;
    return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace tkq

namespace {

tkq_status check_common(int64_t T, int64_t C, int group, int fmt) {
    if (T < 0 || C <= 0) return TKQ_ERR_SHAPE;
    if (group != 128) return TKQ_ERR_GROUP;
    if (C % group) return TKQ_ERR_SHAPE;
    if (fmt != TKQ_FMT_E4M3 && fmt != TKQ_FMT_E5M2) return TKQ_ERR_FMT;
    // TMA row coordinates are 32-bit; C beyond 2^30 is far beyond one GPU
    if (T > INT32_MAX || C > (int64_t{1} << 30)) return TKQ_ERR_SHAPE;
    return TKQ_OK;
}

tkq_status launch_status(cudaError_t e) { return e == cudaSuccess ? TKQ_OK : TKQ_ERR_CUDA; }

constexpr unsigned kSfAllFlags =
    TKQ_SF_ROUND_POW2 | TKQ_SF_UE8M0_PACKED | TKQ_SF_COL_MAJOR | TKQ_Q_RECIPROCAL;

}  // namespace

extern "C" {

int64_t tkq_sf_bytes(int64_t T, int64_t groups_per_row, unsigned sf_flags) {
    if (T < 0 || groups_per_row < 0 || (sf_flags & ~kSfAllFlags)) return -1;
    const int64_t T4 = (T + 3) / 4 * 4;
    const int64_t W = (groups_per_row + 3) / 4;
    const bool cm = sf_flags & TKQ_SF_COL_MAJOR;
    if (sf_flags & TKQ_SF_UE8M0_PACKED) return (cm ? W * T4 : T * W) * 4;
    return (cm ? groups_per_row * T4 : T * groups_per_row) * 4;
}

namespace {
// Checks shared by the row casts: scale flags, scale-buffer alignment.
tkq_status check_sf(const void* sf, unsigned sf_flags) {
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    const uintptr_t a = (sf_flags & TKQ_SF_COL_MAJOR) ? 16 : 4;
    return tkq::aligned(sf, a) ? TKQ_OK : TKQ_ERR_ALIGN;
}
}  // namespace

tkq_status tkq_per_token_cast_ex(const void* x, void* out, void* sf, int64_t T, int64_t C,
                                 int group, int fmt, unsigned sf_flags, tkq_stream_t stream) {
    tkq_status st = check_common(T, C, group, fmt);
    if (st != TKQ_OK) return st;
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    if (T == 0) return TKQ_OK;
    if (!x || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16)) return TKQ_ERR_ALIGN;
    if ((st = check_sf(sf, sf_flags)) != TKQ_OK) return st;
    const auto rx = tkq::span(x, T * C * 2), ro = tkq::span(out, T * C),
               rs = tkq::span(sf, tkq_sf_bytes(T, C / group, sf_flags));
    if (tkq::overlap(rx, ro) || tkq::overlap(rx, rs) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx}, {ro, rs});
    return launch_status(tkq::launch_per_token_cast(x, out, sf, T, C, fmt, sf_flags,
                                                    static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_per_token_cast_f32(const float* x, void* out, void* sf, int64_t T, int64_t C,
                                  int group, int fmt, unsigned sf_flags, tkq_stream_t stream) {
    tkq_status st = check_common(T, C, group, fmt);
    if (st != TKQ_OK) return st;
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    if (T == 0) return TKQ_OK;
    if (!x || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16)) return TKQ_ERR_ALIGN;
    if ((st = check_sf(sf, sf_flags)) != TKQ_OK) return st;
    const auto rx = tkq::span(x, T * C * 4), ro = tkq::span(out, T * C),
               rs = tkq::span(sf, tkq_sf_bytes(T, C / group, sf_flags));
    if (tkq::overlap(rx, ro) || tkq::overlap(rx, rs) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx}, {ro, rs});
    return launch_status(tkq::launch_per_token_cast_f32(x, out, sf, T, C, fmt, sf_flags,
                                                        static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_per_token_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                              int group, int fmt, tkq_stream_t stream) {
    return tkq_per_token_cast_ex(x, out, sf, T, C, group, fmt, 0u, stream);
}

namespace {
// The SwiGLU clamp arguments: a finite bound > 0 and, if given, an 8-byte
// aligned counter that overlaps none of the call's other buffers.
tkq_status check_clamp(float clamp, const uint64_t* count, const tkq::Range* others, int n) {
    if (!(clamp > 0.0f && clamp < INFINITY)) return TKQ_ERR_VALUE;
    if (!count) return TKQ_OK;
    if (!tkq::aligned(count, 8)) return TKQ_ERR_ALIGN;
    const auto rc = tkq::span(count, 8);
    for (int i = 0; i < n; ++i)
        if (tkq::overlap(rc, others[i])) return TKQ_ERR_ALIAS;
    return TKQ_OK;
}

tkq_status swiglu_cast_impl(const void* x, const float* w, void* out, void* sf, int64_t T,
                            int64_t H, int group, int fmt, unsigned sf_flags, const float* clamp,
                            uint64_t* clamp_count, tkq_stream_t stream) {
    tkq_status st = check_common(T, H, group, fmt);
    if (st != TKQ_OK) return st;
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    if (clamp && !(*clamp > 0.0f && *clamp < INFINITY)) return TKQ_ERR_VALUE;
    if (T == 0) return TKQ_OK;
    if (!x || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16) || (w && !tkq::aligned(w, 4)))
        return TKQ_ERR_ALIGN;
    if ((st = check_sf(sf, sf_flags)) != TKQ_OK) return st;
    const auto rx = tkq::span(x, T * H * 4), ro = tkq::span(out, T * H),
               rs = tkq::span(sf, tkq_sf_bytes(T, H / group, sf_flags));
    if (tkq::overlap(rx, ro) || tkq::overlap(rx, rs) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    const auto rw = w ? tkq::span(w, T * 4) : tkq::Range{0, 0};
    if (tkq::overlap(rw, ro) || tkq::overlap(rw, rs)) return TKQ_ERR_ALIAS;
    if (clamp) {
        const tkq::Range others[4] = {rx, ro, rs, rw};
        if ((st = check_clamp(*clamp, clamp_count, others, 4)) != TKQ_OK) return st;
    }
    const auto rc = clamp && clamp_count ? tkq::span(clamp_count, 8) : tkq::Range{0, 0};
    tkq::register_call({rx, rw}, {ro, rs, rc});
    return launch_status(tkq::launch_swiglu_cast(
        x, w, out, sf, T, H, fmt, sf_flags, clamp,
        reinterpret_cast<unsigned long long*>(clamp_count), static_cast<cudaStream_t>(stream)));
}
}  // namespace

tkq_status tkq_swiglu_cast_ex(const void* x, const float* w, void* out, void* sf, int64_t T,
                              int64_t H, int group, int fmt, unsigned sf_flags,
                              tkq_stream_t stream) {
    return swiglu_cast_impl(x, w, out, sf, T, H, group, fmt, sf_flags, nullptr, nullptr, stream);
}

tkq_status tkq_swiglu_cast(const void* x, const float* w, void* out, float* sf, int64_t T,
                           int64_t H, int group, int fmt, tkq_stream_t stream) {
    return swiglu_cast_impl(x, w, out, sf, T, H, group, fmt, 0u, nullptr, nullptr, stream);
}

tkq_status tkq_swiglu_cast_clamp(const void* x, const float* w, void* out, void* sf, int64_t T,
                                 int64_t H, int group, int fmt, unsigned sf_flags,
                                 float clamp_value, uint64_t* clamp_count, tkq_stream_t stream) {
    return swiglu_cast_impl(x, w, out, sf, T, H, group, fmt, sf_flags, &clamp_value,
                            clamp_count, stream);
}

tkq_status tkq_swiglu_backward_cast_ex(const void* x, const void* dy, const float* w, void* out,
                                       void* sf, int64_t T, int64_t H, int group, int fmt,
                                       unsigned sf_flags, tkq_stream_t stream) {
    tkq_status st = check_common(T, H, group, fmt);
    if (st != TKQ_OK) return st;
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    if (T == 0) return TKQ_OK;
    if (!x || !dy || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(dy, 16) || !tkq::aligned(out, 16) ||
        (w && !tkq::aligned(w, 4)))
        return TKQ_ERR_ALIGN;
    if ((st = check_sf(sf, sf_flags)) != TKQ_OK) return st;
    const auto ro = tkq::span(out, T * 2 * H),
               rs = tkq::span(sf, tkq_sf_bytes(T, 2 * H / group, sf_flags));
    const tkq::Range inputs[3] = {tkq::span(x, T * H * 4), tkq::span(dy, T * H * 2),
                                  w ? tkq::span(w, T * 4) : tkq::Range{0, 0}};
    if (tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    for (const auto& in : inputs)
        if (tkq::overlap(in, ro) || tkq::overlap(in, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({inputs[0], inputs[1], inputs[2]}, {ro, rs});
    return launch_status(tkq::launch_swiglu_backward_cast(x, dy, w, out, sf, T, H, fmt, sf_flags,
                                                          static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_swiglu_backward_cast(const void* x, const void* dy, const float* w, void* out,
                                    float* sf, int64_t T, int64_t H, int group, int fmt,
                                    tkq_stream_t stream) {
    return tkq_swiglu_backward_cast_ex(x, dy, w, out, sf, T, H, group, fmt, 0u, stream);
}

namespace {
tkq_status swiglu_cast_t_impl(const void* x, const float* w, void* out, void* sf, void* out_t,
                              void* sf_t, int64_t T, int64_t H, int group, int fmt,
                              unsigned sf_flags, const float* clamp, uint64_t* clamp_count,
                              tkq_stream_t stream) {
    tkq_status st = check_common(T, H, group, fmt);
    if (st != TKQ_OK) return st;
    if (T % group) return TKQ_ERR_SHAPE;
    if (sf_flags & ~kSfAllFlags) return TKQ_ERR_FLAGS;
    if (clamp && !(*clamp > 0.0f && *clamp < INFINITY)) return TKQ_ERR_VALUE;
    if (T == 0) return TKQ_OK;
    // TMA box coordinates are 32-bit
    if (H > (int64_t{1} << 30) || T > INT32_MAX) return TKQ_ERR_SHAPE;
    if (!x || !out || !sf || !out_t || !sf_t) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16) || !tkq::aligned(out_t, 16) ||
        (w && !tkq::aligned(w, 4)))
        return TKQ_ERR_ALIGN;
    if ((st = check_sf(sf, sf_flags)) != TKQ_OK || (st = check_sf(sf_t, sf_flags)) != TKQ_OK)
        return st;
    const tkq::Range r[5] = {tkq::span(x, T * H * 4), tkq::span(out, T * H),
                             tkq::span(sf, tkq_sf_bytes(T, H / group, sf_flags)),
                             tkq::span(out_t, T * H),
                             tkq::span(sf_t, tkq_sf_bytes(H, T / group, sf_flags))};
    for (int i = 0; i < 5; ++i)
        for (int k = i + 1; k < 5; ++k)
            if (tkq::overlap(r[i], r[k])) return TKQ_ERR_ALIAS;
    const auto rw = w ? tkq::span(w, T * 4) : tkq::Range{0, 0};
    for (int i = 1; i < 5; ++i)
        if (tkq::overlap(rw, r[i])) return TKQ_ERR_ALIAS;
    if (clamp) {
        const tkq::Range others[6] = {r[0], r[1], r[2], r[3], r[4], rw};
        if ((st = check_clamp(*clamp, clamp_count, others, 6)) != TKQ_OK) return st;
    }
    const auto rc = clamp && clamp_count ? tkq::span(clamp_count, 8) : tkq::Range{0, 0};
    tkq::register_call({r[0], rw}, {r[1], r[2], r[3], r[4], rc});
    return launch_status(tkq::launch_swiglu_cast_t(
        x, w, out, static_cast<float*>(sf), out_t, static_cast<float*>(sf_t), T, H, fmt, sf_flags,
        clamp, reinterpret_cast<unsigned long long*>(clamp_count),
        static_cast<cudaStream_t>(stream)));
}
}  // namespace

tkq_status tkq_swiglu_cast_t(const void* x, const float* w, void* out, float* sf, void* out_t,
                             float* sf_t, int64_t T, int64_t H, int group, int fmt,
                             tkq_stream_t stream) {
    return swiglu_cast_t_impl(x, w, out, sf, out_t, sf_t, T, H, group, fmt, 0u, nullptr,
                              nullptr, stream);
}

tkq_status tkq_swiglu_cast_t_ex(const void* x, const float* w, void* out, void* sf, void* out_t,
                                void* sf_t, int64_t T, int64_t H, int group, int fmt,
                                unsigned sf_flags, tkq_stream_t stream) {
    return swiglu_cast_t_impl(x, w, out, sf, out_t, sf_t, T, H, group, fmt, sf_flags, nullptr,
                              nullptr, stream);
}

tkq_status tkq_swiglu_cast_t_clamp(const void* x, const float* w, void* out, void* sf,
                                   void* out_t, void* sf_t, int64_t T, int64_t H, int group,
                                   int fmt, unsigned sf_flags, float clamp_value,
                                   uint64_t* clamp_count, tkq_stream_t stream) {
    return swiglu_cast_t_impl(x, w, out, sf, out_t, sf_t, T, H, group, fmt, sf_flags,
                              &clamp_value, clamp_count, stream);
}

tkq_status tkq_per_channel_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                                int group, int fmt, int transpose, tkq_stream_t stream) {
    tkq_status st = check_common(T, C, group, fmt);
    if (st != TKQ_OK) return st;
    if (T % group) return TKQ_ERR_SHAPE;
    if (T == 0) return TKQ_OK;
    if (!x || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16) || !tkq::aligned(sf, 4))
        return TKQ_ERR_ALIGN;
    const auto rx = tkq::span(x, T * C * 2), ro = tkq::span(out, T * C),
               rs = tkq::span(sf, (T / group) * C * 4);
    if (tkq::overlap(rx, ro) || tkq::overlap(rx, rs) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx}, {ro, rs});
    return launch_status(tkq::launch_per_channel_cast(x, out, sf, T, C, fmt, transpose != 0,
                                                      static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_per_block_cast(const void* x, void* out, float* sf, int64_t T, int64_t C,
                              int block, int fmt, tkq_stream_t stream) {
    tkq_status st = check_common(T, C, block, fmt);
    if (st != TKQ_OK) return st;
    if (T == 0) return TKQ_OK;
    if (!x || !out || !sf) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 16) || !tkq::aligned(sf, 4))
        return TKQ_ERR_ALIGN;
    const auto rx = tkq::span(x, T * C * 2), ro = tkq::span(out, T * C),
               rs = tkq::span(sf, (T + block - 1) / block * (C / block) * 4);
    if (tkq::overlap(rx, ro) || tkq::overlap(rx, rs) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx}, {ro, rs});
    return launch_status(
        tkq::launch_per_block_cast(x, out, sf, T, C, fmt, static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_cast_back(const void* codes, const float* sf, void* out, int64_t T, int64_t C,
                         int group_rows, int group_cols, int fmt, int out_dtype,
                         tkq_stream_t stream) {
    if (T < 0 || C <= 0 || C % 128 || T > INT32_MAX || C > (int64_t{1} << 30))
        return TKQ_ERR_SHAPE;
    const bool per_token = group_rows == 1 && group_cols == 128;
    const bool per_channel = group_rows == 128 && group_cols == 1;
    const bool per_block = group_rows == 128 && group_cols == 128;
    if (!per_token && !per_channel && !per_block) return TKQ_ERR_GROUP;
    if (fmt != TKQ_FMT_E4M3 && fmt != TKQ_FMT_E5M2) return TKQ_ERR_FMT;
    if (out_dtype != TKQ_OUT_F32 && out_dtype != TKQ_OUT_BF16) return TKQ_ERR_FMT;
    if (T == 0) return TKQ_OK;
    if (!codes || !sf || !out) return TKQ_ERR_NULL;
    if (!tkq::aligned(codes, 16) || !tkq::aligned(out, 16) ||
        !tkq::aligned(sf, group_cols == 1 ? 16 : 4))
        return TKQ_ERR_ALIGN;
    const int64_t out_bytes = T * C * (out_dtype == TKQ_OUT_F32 ? 4 : 2);
    const int64_t sf_bytes = (T + group_rows - 1) / group_rows * (C / group_cols) * 4;
    const auto ro = tkq::span(out, out_bytes), rq = tkq::span(codes, T * C),
               rs = tkq::span(sf, sf_bytes);
    if (tkq::overlap(ro, rq) || tkq::overlap(ro, rs)) return TKQ_ERR_ALIAS;
    tkq::register_call({rq, rs}, {ro});
    return launch_status(tkq::launch_cast_back(codes, sf, out, T, C, group_rows, group_cols, fmt,
                                               out_dtype == TKQ_OUT_BF16,
                                               static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_swiglu_values(const void* x, const float* w, float* y, int64_t T, int64_t H,
                             tkq_stream_t stream) {
    tkq_status st = check_common(T, H, 128, TKQ_FMT_E4M3);
    if (st != TKQ_OK) return st;
    if (T == 0) return TKQ_OK;
    if (!x || !y) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(y, 16) || (w && !tkq::aligned(w, 4)))
        return TKQ_ERR_ALIGN;
    const auto rx = tkq::span(x, T * H * 4), ry = tkq::span(y, T * H * 4);
    const auto rw = w ? tkq::span(w, T * 4) : tkq::Range{0, 0};
    if (tkq::overlap(rx, ry) || tkq::overlap(rw, ry)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx, rw}, {ry});
    return launch_status(
        tkq::launch_swiglu_values(x, w, y, T, H, static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_swiglu_backward_values(const void* x, const void* dy, const float* w, float* y,
                                      int64_t T, int64_t H, tkq_stream_t stream) {
    tkq_status st = check_common(T, H, 128, TKQ_FMT_E4M3);
    if (st != TKQ_OK) return st;
    if (T == 0) return TKQ_OK;
    if (!x || !dy || !y) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(dy, 16) || !tkq::aligned(y, 16) ||
        (w && !tkq::aligned(w, 4)))
        return TKQ_ERR_ALIGN;
    const auto rx = tkq::span(x, T * H * 4), rd = tkq::span(dy, T * H * 2),
               ry = tkq::span(y, T * H * 8);
    const auto rw = w ? tkq::span(w, T * 4) : tkq::Range{0, 0};
    if (tkq::overlap(rx, ry) || tkq::overlap(rd, ry) || tkq::overlap(rw, ry)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx, rd, rw}, {ry});
    return launch_status(tkq::launch_swiglu_backward_values(x, dy, w, y, T, H,
                                                            static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_fp8_encode(const float* x, void* out, int64_t n, int fmt, tkq_stream_t stream) {
    if (n < 0 || n % 4) return TKQ_ERR_SHAPE;
    if (fmt != TKQ_FMT_E4M3 && fmt != TKQ_FMT_E5M2) return TKQ_ERR_FMT;
    if (n == 0) return TKQ_OK;
    if (!x || !out) return TKQ_ERR_NULL;
    if (!tkq::aligned(x, 16) || !tkq::aligned(out, 4)) return TKQ_ERR_ALIGN;
    const auto rx = tkq::span(x, n * 4), ro = tkq::span(out, n);
    if (tkq::overlap(rx, ro)) return TKQ_ERR_ALIAS;
    tkq::register_call({rx}, {ro});
    return launch_status(
        tkq::launch_fp8_encode(x, out, n, fmt, static_cast<cudaStream_t>(stream)));
}

tkq_status tkq_read_device_status(uint32_t* flags, int clear) {
    if (!flags) return TKQ_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return TKQ_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tkq_device_status, sizeof v) != cudaSuccess)
        return TKQ_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_tkq_device_status, &zero, sizeof zero) != cudaSuccess)
            return TKQ_ERR_CUDA;
    }
    *flags = v;
    return (v & TKQ_DEVICE_TIMEOUT) ? TKQ_ERR_TIMEOUT : TKQ_OK;
}

tkq_status tkq_selftest_wait_timeout(int64_t limit_ns, tkq_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > int64_t{2000000000}) return TKQ_ERR_SHAPE;
    unsigned int* status = tkq::device_status_word();
    if (!status) return TKQ_ERR_CUDA;
    tkq::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        status, static_cast<uint64_t>(limit_ns));
    return launch_status(cudaGetLastError());
}

const char* tkq_status_string(int status) {
    switch (status) {
        case TKQ_OK: return "TKQ_OK";
        case TKQ_ERR_NULL: return "TKQ_ERR_NULL: a required pointer is NULL";
        case TKQ_ERR_SHAPE: return "TKQ_ERR_SHAPE: invalid or unsupported extents";
        case TKQ_ERR_GROUP: return "TKQ_ERR_GROUP: group must be 128";
        case TKQ_ERR_FMT: return "TKQ_ERR_FMT: unknown FP8 format";
        case TKQ_ERR_ALIGN: return "TKQ_ERR_ALIGN: misaligned pointer";
        case TKQ_ERR_CUDA: return "TKQ_ERR_CUDA: kernel launch failed";
        case TKQ_ERR_TIMEOUT:
            return "TKQ_ERR_TIMEOUT: a bounded wait inside a kernel gave up (outputs incomplete)";
        case TKQ_ERR_ALIAS: return "TKQ_ERR_ALIAS: buffers overlap";
        case TKQ_ERR_FLAGS: return "TKQ_ERR_FLAGS: unknown option flags";
        case TKQ_ERR_VALUE: return "TKQ_ERR_VALUE: invalid scalar argument";
        default: return "TKQ_ERR_UNKNOWN";
    }
}

int tkq_version(void) { return 200; }

int tkq_checked_build(void) {
#ifdef TKQ_CHECKED
    return 1;
#else
    return 0;
#endif
}

tkq_status tkq_read_check_address(uint64_t* addr, int clear) {
    if (!addr) return TKQ_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return TKQ_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tkq_bad_address, sizeof v) != cudaSuccess) return TKQ_ERR_CUDA;
    if (clear) {
        const unsigned long long zero = 0;
        if (cudaMemcpyToSymbol(g_tkq_bad_address, &zero, sizeof zero) != cudaSuccess)
            return TKQ_ERR_CUDA;
    }
    *addr = v;
    return TKQ_OK;
}

}  // extern "C"
