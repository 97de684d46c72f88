// tc_sync.cuh -- bounded mbarrier waits and small TMEM helpers shared by the
// tensor-core kernels.
//
// Every wait is bounded: after kTimeoutNs the waiting thread records
// (1 + role) << 24 | tile in its translation unit's device error word, raises
// the CTA's abort flag (other waiters then give up at once) and returns false,
// so a CTA can always wind down (drain its copies, free TMEM, exit) instead of
// hanging the GPU.
#pragma once

#include "tc_ptx.cuh"

namespace psa {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

struct Sync {
    uint32_t bar0;          // shared address of barrier 0 (barriers are 8 bytes apart)
    volatile int* abort;    // CTA-wide abort flag in shared memory
    int* err;               // device error word of the calling translation unit
    __device__ uint32_t bar(int i) const { return bar0 + 8u * i; }
};

// Bounded wait on a barrier phase, by one thread.  Returns false on timeout or
// when another thread of the CTA has already aborted.  Polls with the plain
// try_wait (whose own suspension is short and system-defined), so the
// %globaltimer check below always runs and the wait is bounded.
static __device__ __noinline__ bool wait_slow(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile,
                                              uint64_t limit_ns = kTimeoutNs) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 15) {
            if (*s.abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                *s.abort = 1;
                atomicCAS(s.err, 0, ((1 + role) << 24) | (tile & 0xFFFFFF));
                return false;
            }
        }
    }
}
// Fast path first (the phase is often already complete), then the bounded loop.
__device__ __forceinline__ bool wait_bounded(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(s, bar, parity, role, tile);
}

// The same bounded wait with cluster-scope acquire, for barriers that the
// peer CTA of a pair arrives on.
static __device__ __noinline__ bool wait_slow_cluster(const Sync& s, uint32_t bar, uint32_t parity, int role,
                                                      int tile) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 15) == 15) {
            if (*s.abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kTimeoutNs) {
                *s.abort = 1;
                atomicCAS(s.err, 0, ((1 + role) << 24) | (tile & 0xFFFFFF));
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_bounded_cluster(const Sync& s, uint32_t bar, uint32_t parity, int role,
                                                     int tile) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return wait_slow_cluster(s, bar, parity, role, tile);
}

// Four barrier phases tested in one round trip: the try_waits issue back to
// back and only their combined result is waited for.  (Pass a phase twice to
// test fewer.)  The fast path of warp_wait_all.
__device__ __forceinline__ bool mbar_try_wait4(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, uint32_t b2,
                                               uint32_t p2, uint32_t b3, uint32_t p3) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2, q3;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q3, [%7], %8;\n\t"
        "and.pred q0, q0, q1;\n\tand.pred q2, q2, q3;\n\tand.pred q0, q0, q2;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t}"
        : "=r"(ok)
        : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2), "r"(b3), "r"(p3)
        : "memory");
    return ok != 0;
}

// Whole-warp wait: every lane waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(const Sync& s, uint32_t bar, uint32_t parity, int role, int tile) {
    const bool ok = wait_bounded(s, bar, parity, role, tile);
    return __all_sync(0xffffffffu, ok);
}

// Whole-warp wait on four barrier phases (b_i, p_i): one round trip when all
// are complete already, else each in turn with the bounded wait.
__device__ __forceinline__ bool warp_wait_all(const Sync& s, uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1,
                                              uint32_t b2, uint32_t p2, uint32_t b3, uint32_t p3, int role,
                                              int tile) {
    if (__all_sync(0xffffffffu, mbar_try_wait4(b0, p0, b1, p1, b2, p2, b3, p3))) return true;
    return warp_wait(s, b0, p0, role, tile) && warp_wait(s, b1, p1, role, tile) && warp_wait(s, b2, p2, role, tile) &&
           warp_wait(s, b3, p3, role, tile);
}

// Wait without the abort short-cut (used only to drain work after an abort).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kTimeoutNs) return false;
    return true;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One TMEM row segment of D 32-bit columns (this thread's lane) into v[D].
template <int D>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t* v) {
    if constexpr (D == 16) {
        tmem_ld_32x32b_x16(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32 * c, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[32 * c + e] = r[e];
        }
    }
}

}  // namespace tc
}  // namespace psa
