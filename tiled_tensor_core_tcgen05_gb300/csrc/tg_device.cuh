// Device helpers shared by the kernels: bounded mbarrier waits (the watchdog)
// and the fused epilogue  y = epi(acc + bias)  with one rounding to binary16.
#pragma once

#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {

// Per-CTA view of the watchdog: a shared abort flag plus the global status word.
struct WaitCtx {
    volatile int* abort;  // shared memory: set once any wait in this CTA expires
    int* status;
    uint64_t limit_ns;
};

// Wait for the phase of `bar` with parity `parity` to complete. Gives up (and
// returns false) when another wait of this CTA has already expired, or after
// limit_ns, recording `site` as the first expired wait. kCluster: the barrier
// receives arrives from another CTA of the cluster (acquire at cluster scope).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    auto try_once = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (try_once()) return true;
        if (*w.abort) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            atomicCAS(w.status, 0, site);
            return false;
        }
    }
}

// Wait used while draining at exit: ignores the abort flag (the point is to let
// copies or MMAs already in flight land before shared/tensor memory is
// released), but still bounded.
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > w.limit_ns) {
            atomicCAS(w.status, 0, kSiteDrain);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so a
// group takes one decision together (e.g. "some thread's wait gave up").
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// GELU with the exact Gaussian CDF, in fp32: 0.5 x (1 + erf(x / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float x) {
    return 0.5f * x * (1.0f + erff(x * 0.70710678118654752440f));
}

__device__ __forceinline__ float epi_value(float acc, float b, int gelu) {
    const float x = acc + b;
    return gelu ? gelu_erf(x) : x;
}

// 32 consecutive columns of one output row (col0..col0+31), held as fp32 bit
// patterns by one thread: add bias, apply GELU, round to binary16, store.
// Columns >= N are not written; rows are masked by the caller.
__device__ __forceinline__ void epilogue_row32(const uint32_t (&r)[32], __half* __restrict__ crow,
                                               const __half* __restrict__ bias, int col0, int N,
                                               int gelu, int c_vec, int bias_vec) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    const bool full = col0 + 32 <= N;
    if (bias != nullptr) {
        if (full && bias_vec) {
            const uint4* bp = reinterpret_cast<const uint4*>(bias + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 u = __ldg(bp + q);
                const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = __half22float2(h[e]);
                    v[q * 8 + 2 * e] += f.x;
                    v[q * 8 + 2 * e + 1] += f.y;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col0 + i < N) v[i] += __half2float(bias[col0 + i]);
        }
    }
    if (gelu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_erf(v[i]);
    }
    if (full && c_vec) {
        uint4* cp = reinterpret_cast<uint4*>(crow + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 u;
            __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
            cp[q] = u;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < N) crow[col0 + i] = __float2half_rn(v[i]);
    }
}

}  // namespace tg
