// Epilogue shared by the skinny (swap-AB) kernels. The accumulator of one work
// unit holds C^T: TMEM lane n (one output column) times m_pad fp32 columns
// (the rows of C), as kHalves 128-lane halves. Four warps, one per TMEM lane
// quarter, read it back. With one K slice they apply bias and GELU and write
// C; with several, each unit stores its partial tile to scratch laid out
// [slice][n][m_pad], and the last unit of a column slice to finish adds the
// partials in slice order 0, 1, ... (so the result does not depend on which
// CTA finishes last), applies the epilogue, writes C and resets the slice's
// arrival counter to zero for the next launch.
//
// The epilogue is that of "Designing high-performance GPU kernels with
// TileLang ..." (section 3, GELU(MatMul + Bias)); the split-K reduction is
// this library's own design for skinny shapes.
#pragma once

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {

constexpr int kSkEpiThreads = 128;

// Runs the epilogue role for every unit this CTA owns (units blockIdx.x,
// blockIdx.x + gridDim.x, ...; unit u is column slice u % n_tiles of K slice
// u / n_tiles). Accumulator buffer b = (i-th unit of this CTA) & 1 starts at
// TMEM column b * kHalves * tmem_stride; half h at + h * tmem_stride.
// acc_full0 / acc_empty0: the first of two consecutive mbarriers each (8 bytes
// apart); acc_empty counts kSkEpiThreads arrivals. epi_thread0: the first
// thread of the four epilogue warps. Named barrier 1 is used.
template <int kHalves>
__device__ __forceinline__ void skinny_epilogue(const SplitArgs& args, uint32_t tmem_base, uint32_t acc_full0,
                                                uint32_t acc_empty0, volatile int* last_flag, const WaitCtx& wc,
                                                int epi_thread0) {
    constexpr int kUnitCols = 128 * kHalves;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int ept = threadIdx.x - epi_thread0;  // 0..127
    const int chunks = args.m_pad / 16;
    int it = 0;
    for (int u = blockIdx.x; u < args.num_units; u += gridDim.x, ++it) {
        const int sp = u / args.n_tiles;
        const int nt = u - sp * args.n_tiles;
        const int b = it & 1;
        const bool ok = wait_phase(acc_full0 + 8 * b, (it >> 1) & 1, wc, kSiteEpilogueAccFull);
        // all 128 epilogue threads stop together, so the named barriers below
        // never wait for a thread that has left
        if (named_barrier_or(1, kSkEpiThreads, !ok)) break;
        tc_fence_after_sync();
#pragma unroll 1
        for (int h = 0; h < kHalves; ++h) {
            const int n = nt * kUnitCols + h * 128 + quarter * 32 + lane;  // this thread's output column
            const bool n_ok = n < args.N;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   (b * kHalves + h) * args.tmem_stride;
            const float bias_n = (args.bias != nullptr && n_ok) ? __half2float(args.bias[n]) : 0.0f;
            for (int c = 0; c < chunks; ++c) {
                uint32_t r[16];
                __syncwarp();  // tcgen05.ld is warp-collective; lanes diverged on the column mask
                tmem_ld_32x32b_x16(taddr + c * 16, r);
                tmem_ld_wait();
                if (h == kHalves - 1 && c == chunks - 1) {
                    tc_fence_before_sync();
                    mbar_arrive(acc_empty0 + 8 * b);  // every accumulator of buffer b is read
                }
                if (!n_ok) continue;
                if (args.splits == 1) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = c * 16 + i;
                        if (m >= args.M) break;
                        args.C[static_cast<int64_t>(m) * args.N + n] =
                            __float2half_rn(epi_value(__uint_as_float(r[i]), bias_n, args.gelu));
                    }
                } else {
                    // partials as [slice][n][m_pad]: this thread's 16 rows are 64 contiguous bytes
                    const int64_t off = (static_cast<int64_t>(sp) * args.N + n) * args.m_pad + c * 16;
                    if (!dbg_check(dbg_in(off, 16, args.wd.ws_floats), args.wd)) continue;
                    uint4* wp = reinterpret_cast<uint4*>(args.ws + off);
#pragma unroll
                    for (int q = 0; q < 4; ++q) wp[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                }
            }
        }
        if (args.splits > 1 && !args.separate_reduce) {
            // publish this slice's partials, then count arrivals for column slice nt
            __threadfence();
            named_barrier_sync(1, kSkEpiThreads);
            if (ept == 0) {
                *last_flag = 0;
                if (dbg_check(dbg_in(nt, 1, args.wd.n_counters), args.wd)) {
                    const unsigned int prev = atomicAdd(args.counters + nt, 1u);
                    *last_flag = (prev == static_cast<unsigned int>(args.splits - 1)) ? 1 : 0;
                }
            }
            named_barrier_sync(1, kSkEpiThreads);
            if (*last_flag) {
                __threadfence();
#pragma unroll 1
                for (int h = 0; h < kHalves; ++h) {
                    const int n = nt * kUnitCols + h * 128 + quarter * 32 + lane;
                    if (n >= args.N) continue;
                    const float bias_n = args.bias != nullptr ? __half2float(args.bias[n]) : 0.0f;
                    for (int m0 = 0; m0 < args.M; m0 += 16) {
                        // this column's 16 rows m0..m0+15 of every slice: four 16-byte loads per
                        // slice; each row sums its slices in order 0, 1, ... (deterministic). The
                        // loads of kBatch slices are issued before any of them is added, so the
                        // reduction waits for one L2 round trip per kBatch slices, not per slice.
                        constexpr int kBatch = 4;
                        float s[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) s[i] = 0.0f;
                        auto add_slice = [&](const float4 (&p)[4]) {
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                s[4 * v4] += p[v4].x;
                                s[4 * v4 + 1] += p[v4].y;
                                s[4 * v4 + 2] += p[v4].z;
                                s[4 * v4 + 3] += p[v4].w;
                            }
                        };
                        int q = 0;
                        for (; q + kBatch <= args.splits; q += kBatch) {
                            float4 p[kBatch][4];
                            bool in[kBatch];
#pragma unroll
                            for (int j = 0; j < kBatch; ++j) {
                                const int64_t off = (static_cast<int64_t>(q + j) * args.N + n) * args.m_pad + m0;
                                in[j] = dbg_check(dbg_in(off, 16, args.wd.ws_floats), args.wd);
                                const float4* wq = reinterpret_cast<const float4*>(args.ws + (in[j] ? off : 0));
#pragma unroll
                                for (int v4 = 0; v4 < 4; ++v4) p[j][v4] = __ldcg(wq + v4);
                            }
#pragma unroll
                            for (int j = 0; j < kBatch; ++j)
                                if (in[j]) add_slice(p[j]);
                        }
                        for (; q < args.splits; ++q) {
                            const int64_t off = (static_cast<int64_t>(q) * args.N + n) * args.m_pad + m0;
                            if (!dbg_check(dbg_in(off, 16, args.wd.ws_floats), args.wd)) continue;
                            const float4* wq = reinterpret_cast<const float4*>(args.ws + off);
                            float4 p[4];
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) p[v4] = __ldcg(wq + v4);
                            add_slice(p);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (m0 + i < args.M)
                                args.C[static_cast<int64_t>(m0 + i) * args.N + n] =
                                    __float2half_rn(epi_value(s[i], bias_n, args.gelu));
                    }
                }
                if (ept == 0) atomicExch(args.counters + nt, 0u);
            }
        }
    }
}

}  // namespace tg
