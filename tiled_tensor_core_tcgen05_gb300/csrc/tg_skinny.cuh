// Epilogue shared by the skinny (swap-AB) kernels. The accumulator of one work
// unit holds C^T: TMEM lane n (one output column) times m_pad fp32 columns
// (the rows of C), as kHalves 128-lane halves. Four warps, one per TMEM lane
// quarter, read it back. With one K slice they apply bias and GELU and write
// C; with several, each unit stores its partial tile to scratch laid out
// [slice][n][m_pad], and a second kernel (launch_splitk_reduce) adds the
// partials over the whole GPU in slice order 0, 1, ..., applies the epilogue
// and writes C; or, in the cluster form, each CTA stages its tile in shared
// memory for an in-kernel sum across the cluster. (Reducing in the last CTA of each column slice to arrive left
// one CTA per 256 columns summing every slice alone: at 64 rows and eight
// slices that serial tail took longer than the product.)
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
// apart); acc_empty counts kSkEpiThreads arrivals. Named barrier 1 is used.
// Cluster form (kCl): the CTAs of a cluster are the K slices of one unit, one unit per CTA;
// each stages its fp32 tile transposed back to C's orientation, [m][256 columns] with a row
// pitch of kSkClPitch floats, at stage_base (its idle operand ring), for the in-kernel sum.
constexpr int kSkClPitch = 256 + 4;

template <int kHalves, bool kCl = false>
__device__ __forceinline__ void skinny_epilogue(const SplitArgs& args, uint32_t tmem_base, uint32_t acc_full0,
                                                uint32_t acc_empty0, const WaitCtx& wc, uint32_t stage_base = 0) {
    constexpr int kUnitCols = 128 * kHalves;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int chunks = args.m_pad / 16;
    int it = 0;
    for (int u = blockIdx.x; u < args.num_units; u += gridDim.x, ++it) {
        const int sp = kCl ? u % args.splits : u / args.n_tiles;
        const int nt = kCl ? u / args.splits : u - sp * args.n_tiles;
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
                if (kCl && args.splits > 1) {
                    // every lane stages its column (rows beyond M are zeros and are not stored)
                    const int nl = h * 128 + quarter * 32 + lane;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        st_shared_u32(stage_base + static_cast<uint32_t>(((c * 16 + i) * kSkClPitch + nl) * 4), r[i]);
                    continue;
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
    }
}

}  // namespace tg
