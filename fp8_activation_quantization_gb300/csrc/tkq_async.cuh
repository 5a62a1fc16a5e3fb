// tkq_async.cuh -- mbarrier, TMA and named-barrier helpers (inline PTX for
// sm_103a) and the bounded wait used by every pipelined kernel.
//
// Every wait on an mbarrier is bounded: after kWaitLimitNs of wall time
// (%globaltimer) it gives up, records kDeviceTimeout in the library's device
// status word and returns false, so a kernel whose copies never arrive ends
// with an error status the host can read instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tkq {

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // one second
constexpr uint32_t kDeviceTimeout = 1u;                        // status-word bit

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// (returning false) when *abort becomes non-zero (another thread of the CTA gave
// up) or after `limit_ns`; a timeout is recorded in *status.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  const volatile int* abort, unsigned int* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                if (status) atomicOr(status, kDeviceTimeout);
                return false;
            }
        }
    }
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
// x is the innermost coordinate (elements); x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// L2 prefetch of the box a tma_load_2d at (x, y) would copy.  A hint that
// changes no value any load returns, so, like prefetch_l2, it may be issued
// before grid_dependency_wait.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Walk of a persistent CTA over a [rows x cols] grid of tiles (cols fastest):
// tiles start, start + step, start + 2 step, ...  The row/column of each tile
// is updated incrementally, so the loop needs no integer division.
struct TileWalk {
    uint32_t row, col, step_row, step_col, cols;
    __device__ __forceinline__ TileWalk(uint32_t start, uint32_t step, uint32_t n_cols)
        : cols(n_cols) {
        row = start / n_cols;
        col = start - row * n_cols;
        step_row = step / n_cols;
        step_col = step - step_row * n_cols;
    }
    __device__ __forceinline__ void next() {
        row += step_row;
        col += step_col;
        if (col >= cols) {
            col -= cols;
            ++row;
        }
    }
};

// Position in a ring of S stages: the stage index and the parity of the
// current use of that stage.  A consumer waits for `full[stage]` with parity
// `phase`; the producer waits for `empty[stage]` with parity `phase ^ 1`, which
// completes at once on the first use (the barrier's preceding phase counts as
// complete), so neither side needs a first-round special case.
template <int S>
struct RingPos {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// Barrier over `n` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over `n` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

}  // namespace tkq
