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
// The abort flag and the clock are read once every kWaitCheckEvery polls, so
// a phase that completes is noticed by the next poll rather than after a
// clock read; every poll returns within its own hardware time limit, so the
// wait stays bounded.
constexpr uint32_t kWaitCheckEvery = 16;

template <bool kCluster = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    auto try_once = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (try_once()) return true;
    uint64_t t0 = 0;
    for (uint32_t spin = 1;; ++spin) {
        if (try_once()) return true;
        if (spin % kWaitCheckEvery == 0) {
            if (*w.abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > w.limit_ns) {
                *w.abort = 1;
                atomicCAS(w.status, 0, site);
                return false;
            }
        }
    }
}

// wait_phase for waits whose latency matters little (a whole work unit, or a
// ring slot refilled by a slower stage): between polls the thread sleeps
// about sleep_ns, so a waiting warp takes few issue slots from the warps that
// work beside it on the same scheduler. Same bound and abort rules.
__device__ __forceinline__ bool wait_phase_sleep(uint32_t bar, uint32_t parity, const WaitCtx& w, int site,
                                                 uint32_t sleep_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
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

// Bounds check of debug builds: records kSiteBounds in the status word (the
// first failure of any kind wins) and returns false, so the caller skips the
// access; in normal builds it is compiled away and returns true.
__device__ __forceinline__ bool dbg_check(bool ok, const Watchdog& wd) {
#if TG_DEBUG
    if (!ok) atomicCAS(wd.status, 0, kSiteBounds);
    return ok;
#else
    (void)ok;
    (void)wd;
    return true;
#endif
}

// [first, first + count) inside [0, limit)
__device__ __forceinline__ bool dbg_in(int64_t first, int64_t count, int64_t limit) {
    return first >= 0 && count >= 0 && first + count <= limit;
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

// ---------------------------------------------------------------------------
// 4-bit weight decoding, shared by the two 4-bit GEMM kernels.

// INT4: one 32-bit word of packed weights (eight consecutive k of one column, byte
// p holding k = 2p in its low and 2p + 1 in its high nibble) into four fp16
// pairs (w[k] * scale, each product rounded once), in the order
// (k0, k4), (k1, k5), (k2, k6), (k3, k7): the order in which masks that keep
// one nibble of each 16-bit half deliver them. The kernels that use it pair
// the activations the same way, so the dot product over k is unchanged.
// A nibble masked under the exponent bits 0x64 and XORed with 8 (two's
// complement q -> q + 8) reads 1024 + (q + 8) in the low nibble position and
// 1024 + 16 (q + 8) in the high one; one fp16 fused multiply-add maps either
// exactly to q, and the scale multiply is the only rounding.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, uint32_t* out) {
    const __half2 one = __halves2half2(__ushort_as_half(0x3C00), __ushort_as_half(0x3C00));        // 1
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
    const __half2 off_lo = __halves2half2(__ushort_as_half(0xE408), __ushort_as_half(0xE408));     // -1032
    const __half2 off_hi = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));     // -72
    const uint32_t w8 = w >> 8;
    uint32_t x[4] = {(w & 0x000F000Fu) ^ 0x64086408u, (w & 0x00F000F0u) ^ 0x64806480u,
                     (w8 & 0x000F000Fu) ^ 0x64086408u, (w8 & 0x00F000F0u) ^ 0x64806480u};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        __half2 h = *reinterpret_cast<__half2*>(&x[p]);
        h = __hmul2((p & 1) ? __hfma2(h, sixteenth, off_hi) : __hfma2(h, one, off_lo), s2);
        out[p] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// FP4 (E2M1): the same word into four fp16 pairs in natural order (k0, k1),
// (k2, k3), (k4, k5), (k6, k7): each byte holds one pair, converted exactly by
// the hardware's e2m1x2 -> f16x2 conversion (every E2M1 value is exact in
// fp16); the scale multiply is the only rounding. In this order the
// activations need no reordering.
__device__ __forceinline__ void dequant_word_fp4(uint32_t w, __half2 s2, uint32_t* out) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        __half2 v = __hmul2(*reinterpret_cast<__half2*>(&h[p]), s2);
        out[p] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// GELU with the Gaussian CDF, in fp32: 0.5 x (1 + erf(x / sqrt 2)), the erf form
// (not the tanh approximation). With z = |x| / sqrt 2 it is x (1 - erfc(z) / 2) for
// x >= 0 and x erfc(z) / 2 for x < 0, so no term cancels. erfc is Abramowitz &
// Stegun, Handbook of Mathematical Functions, formula 7.1.26: with t = 1 / (1 + p z),
// erfc(z) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2), |error| <= 1.5e-7,
// one reciprocal and one exp2 on the special-function unit. Rounded to fp16 it
// meets the correctly rounded GELU on all but a few hundred of the 63,488 finite
// fp16 inputs, each within one ulp.
__device__ __forceinline__ float gelu_erf(float x) {
    const float z = fabsf(x) * 0.70710678118654752440f;
    const float t = rcp_approx(fmaf(0.3275911f, z, 1.0f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    // __fmul_rn keeps 1 - erfc/2 from contracting into an fma in some call sites
    // and not others, so every kernel's epilogue rounds the same way
    const float half_erfc = __fmul_rn(0.5f * (q * t), ex2_approx(-1.44269504088896341f * z * z));
    return x * (x >= 0.0f ? 1.0f - half_erfc : half_erfc);
}

__device__ __forceinline__ float epi_value(float acc, float b, int gelu) {
    const float x = acc + b;
    return gelu ? gelu_erf(x) : x;
}

// Bytes of shared memory each epilogue warp uses to stage one 32 x 32 chunk of
// C: 32 rows of 64 bytes at an 80-byte pitch, so the lanes' 16-byte writes of
// their own rows fall in distinct banks.
constexpr int kStagePitch = 80;
constexpr int kStageWarpBytes = 32 * kStagePitch;

// How a warp may write C: 16-byte units (row starts 16-byte aligned, N % 8 == 0),
// 4-byte units (4-byte aligned, N even) or single elements.
enum CStoreMode : int { kStore16 = 2, kStore4 = 1, kStore2 = 0 };

// The epilogue of one lane's 32 accumulator values (fp32 bits) of columns
// col0..col0+31: add the bias (columns >= N get none), apply GELU.
__device__ __forceinline__ void epilogue_values(const uint32_t (&r)[32], float (&v)[32],
                                                const __half* __restrict__ bias, int col0, int N, int gelu,
                                                int bias_vec) {
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
}

// One warp's 32 x 32 chunk of C, rows row0..row0+31 (lane l computed row
// row0 + l), columns col0..col0+31. Each lane holds its row's 32 accumulator
// values (fp32 bits): add bias, apply GELU, round once to binary16, stage the
// row in this warp's shared buffer, then write the chunk back row by row so
// each store instruction covers whole 64-byte row segments. Rows >= M and
// columns >= N are not written.
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&r)[32], uint8_t* stage, __half* __restrict__ C,
                                               const __half* __restrict__ bias, int row0, int col0, int M, int N,
                                               int gelu, int store_mode, int bias_vec) {
    const int lane = threadIdx.x & 31;
    float v[32];
    epilogue_values(r, v, bias, col0, N, gelu, bias_vec);
    const bool full = col0 + 32 <= N;
    // this lane's row into the staging buffer
    uint4* mine = reinterpret_cast<uint4*>(stage + lane * kStagePitch);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
        mine[q] = u;
    }
    __syncwarp();
    if (store_mode == kStore16 && full) {
        // 4 lanes per row, 8 rows per instruction
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int rr = pass * 8 + (lane >> 2);
            const int q = lane & 3;
            const int row = row0 + rr;
            if (row < M)
                *reinterpret_cast<uint4*>(C + static_cast<int64_t>(row) * N + col0 + q * 8) =
                    *reinterpret_cast<const uint4*>(stage + rr * kStagePitch + q * 16);
        }
    } else if (store_mode != kStore2) {
        // 16 lanes per row, 2 rows per instruction, one or two elements per lane
#pragma unroll 4
        for (int pass = 0; pass < 16; ++pass) {
            const int rr = pass * 2 + (lane >> 4);
            const int c = col0 + 2 * (lane & 15);
            const int row = row0 + rr;
            if (row < M && c < N) {
                __half* dst = C + static_cast<int64_t>(row) * N + c;
                const __half* src = reinterpret_cast<const __half*>(stage + rr * kStagePitch) + 2 * (lane & 15);
                if (c + 1 < N)
                    *reinterpret_cast<__half2*>(dst) = *reinterpret_cast<const __half2*>(src);
                else
                    dst[0] = src[0];
            }
        }
    } else {
        // one element per lane, one row per instruction
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
            const int row = row0 + rr;
            const int c = col0 + lane;
            if (row < M && c < N)
                C[static_cast<int64_t>(row) * N + c] =
                    reinterpret_cast<const __half*>(stage + rr * kStagePitch)[lane];
        }
    }
    __syncwarp();  // the buffer is rewritten by this warp's next chunk
}

// Bytes of one TMA-store staging buffer: a 32 x 32 fp16 box, 64-byte rows.
constexpr int kStoreBoxBytes = 32 * 32 * 2;

// The same chunk written back by a TMA store: the lanes stage their rows in a
// dense 32 x 64-byte box at shared address `buf` (1024-byte aligned) in the
// 64-byte swizzle the tensor map of C uses (16-byte unit q of row rr at unit
// q ^ ((rr >> 1) & 3), so the warp's writes fall in distinct banks), then lane
// 0 issues one store of the box at (col0, row0) and commits it as a bulk
// group; the store leaves out rows >= M and columns >= N. The caller lets lane
// 0 wait (bulk_wait_group_read) before `buf` is written again.
__device__ __forceinline__ void epilogue_chunk_tma(const uint32_t (&r)[32], uint32_t buf, const CUtensorMap* tmC,
                                                   const __half* __restrict__ bias, int row0, int col0, int N,
                                                   int gelu, int bias_vec, const Watchdog& wd) {
    const int lane = threadIdx.x & 31;
    float v[32];
    epilogue_values(r, v, bias, col0, N, gelu, bias_vec);
    const uint32_t row_base = buf + static_cast<uint32_t>(lane) * 64;
    const uint32_t swz = static_cast<uint32_t>((lane >> 1) & 3);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row_base + ((static_cast<uint32_t>(q) ^ swz) << 4)),
                     "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w)
                     : "memory");
    }
    fence_proxy_async_smem();  // the generic-proxy writes -> visible to the TMA unit
    __syncwarp();
    // a store's x must start on a 16-byte boundary and no store may start at a negative coordinate
    if (lane == 0 && dbg_check(row0 >= 0 && col0 >= 0 && col0 % 8 == 0, wd)) {
        tma_store_2d(tmC, buf, col0, row0);
        bulk_commit_group();
    }
}

}  // namespace tg
