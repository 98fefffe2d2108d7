// Attention forward (FlashAttention): O = softmax(Q K^T / sqrt(d)) V, optional
// causal mask, on (batch, sequence, head, dim) fp16 tensors with d = 128.
//
// "TileLang: writing LLM GPU kernels by thinking in tiles" (section 5,
// FlashAttention) states the operation and the strategy: blocks of Q against
// blocks of K and V, intermediates kept on chip, the softmax built up
// incrementally. "TileLang: you write the dataflow, the compiler owns the
// schedule" (section "FlashAttention, in tiles") gives the online form used
// here: per key block, the running row maximum, the ratio of old to new
// maximum rescaling the accumulator and the running sum, exponentials in base
// 2 with log2(e) folded into the scale; 128 x 128 blocks with d = 128.
//
// GB300 mapping. One CTA per (batch, head, 128-query block).
//   warp 0      TMA producer: Q once (two 64-column boxes), then K and V
//               blocks of 128 keys into a two-stage ring;
//   warp 1      allocates TMEM; one thread issues S_j = Q K_j^T (M = N = 128,
//               K = d) into one of two TMEM score buffers, and O += P_j V_j
//               with P_j read from TMEM as the A operand. S_{j+1} is issued
//               before O += P_j V_j, so the tensor core works while the
//               softmax of block j runs;
//   warps 2-5   softmax, one thread per query row (its TMEM lane): read the
//               row of S_j, mask, row maximum, exponentials, running sum;
//               write P_j (fp16) to TMEM; rescale the O row when needed; at
//               the end divide by the sum and write O.
// The accumulator is only rescaled when a row's maximum grows by more than
// 2^8 (in the base-2 domain); otherwise the old maximum stays the reference,
// so the exponentials are at most 2^8 and the final O / sum is unchanged.
//
// TMEM columns: S buffers [0, 256), O [256, 384), P buffers [384, 512)
// (fp16 pairs of keys, 64 columns each).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kD = kAttnD;
constexpr int kBM = 128;                       // queries per CTA
constexpr int kBN = 128;                       // keys per block
constexpr int kStages = 2;
constexpr int kBoxBytes = 128 * 64 * 2;        // 128 rows x 64 columns fp16
constexpr int kTileBytes = 2 * kBoxBytes;      // 128 rows x 128 columns
constexpr int kThreads = 6 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr float kRescaleLog2 = 8.0f;           // lazy rescale threshold (base-2 exponent)
static_assert(kD == 128, "head dimension 128");

// shared memory: Q, then per stage K and V, then barriers
constexpr int kOffQ = 0;
constexpr int kOffKV = kTileBytes;
constexpr int kOffBar = kOffKV + kStages * 2 * kTileBytes;
constexpr int kBarQ = kOffBar;
constexpr int kBarKFull = kBarQ + 8;
constexpr int kBarVFull = kBarKFull + 8 * kStages;
constexpr int kBarKVEmpty = kBarVFull + 8 * kStages;
constexpr int kBarSFull = kBarKVEmpty + 8 * kStages;
constexpr int kBarSFree = kBarSFull + 16;
constexpr int kBarPFull = kBarSFree + 16;
constexpr int kBarPFree = kBarPFull + 16;
constexpr int kBarDrain = kBarPFree + 16;
constexpr int kTmemSlot = kBarDrain + 8;
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kSmemUsed = kAbortSlot + 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // block -> (query block, head, batch); the longest causal blocks first
    const int qt = args.n_qt - 1 - static_cast<int>(blockIdx.x % args.n_qt);
    const int bh = static_cast<int>(blockIdx.x / args.n_qt);
    const int h = bh % args.H;
    const int b = bh / args.H;
    const int n_kt = (args.S + kBN - 1) / kBN;
    const int j_last = args.causal ? min(qt, n_kt - 1) : n_kt - 1;  // key blocks 0..j_last

    const uint32_t bar_q = sbase + kBarQ;
    auto k_full = [&](int s) { return sbase + kBarKFull + 8 * s; };
    auto v_full = [&](int s) { return sbase + kBarVFull + 8 * s; };
    auto kv_empty = [&](int s) { return sbase + kBarKVEmpty + 8 * s; };
    auto s_full = [&](int i) { return sbase + kBarSFull + 8 * i; };
    auto s_free = [&](int i) { return sbase + kBarSFree + 8 * i; };
    auto p_full = [&](int i) { return sbase + kBarPFull + 8 * i; };
    auto p_free = [&](int i) { return sbase + kBarPFree + 8 * i; };
    auto k_tile = [&](int s) { return sbase + kOffKV + s * 2 * kTileBytes; };
    auto v_tile = [&](int s) { return sbase + kOffKV + s * 2 * kTileBytes + kTileBytes; };
    const uint32_t drain_bar = sbase + kBarDrain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(s_free(i), 4);  // one arrival per softmax warp
            mbar_init(p_full(i), 4);
            mbar_init(p_free(i), 1);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wc{abort_flag, args.wd.status, args.wd.limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, kTileBytes);
            for (int i = 0; i < 2; ++i)
                tma_load_4d(sbase + kOffQ + i * kBoxBytes, &tmQ, bar_q, 64 * i, h, qt * kBM, b);
            uint32_t issued = 0, parity = 0;
            for (int j = 0; j <= j_last; ++j) {
                const int s = j % kStages;
                const uint32_t ph = static_cast<uint32_t>(j / kStages) & 1u;
                if (!wait_phase_sleep(kv_empty(s), ph ^ 1, wc, kSiteProducerEmpty, 64)) break;
                mbar_arrive_expect_tx(k_full(s), kTileBytes);
                for (int i = 0; i < 2; ++i)
                    tma_load_4d(k_tile(s) + i * kBoxBytes, &tmK, k_full(s), 64 * i, h, j * kBN, b);
                mbar_arrive_expect_tx(v_full(s), kTileBytes);
                for (int i = 0; i < 2; ++i)
                    tma_load_4d(v_tile(s) + i * kBoxBytes, &tmV, v_full(s), 64 * i, h, j * kBN, b);
                issued |= 1u << s;
                parity = (parity & ~(1u << s)) | (ph << s);
            }
            wait_phase_drain(bar_q, 0, wc);
            for (int s = 0; s < kStages; ++s)
                if (issued & (1u << s)) {
                    wait_phase_drain(k_full(s), (parity >> s) & 1, wc);
                    wait_phase_drain(v_full(s), (parity >> s) & 1, wc);
                }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16_f32(kBM, kBN, /*a_mn_major=*/false, /*b_mn_major=*/false);
            const uint32_t idesc_o = idesc_f16_f32(kBM, kD, /*a_mn_major=*/false, /*b_mn_major=*/true);
            bool ok = wait_phase(bar_q, 0, wc, kSiteMmaFull);
            tc_fence_after_sync();
            // S_j = Q K_j^T: both operands K-major (d contiguous), two 64-column boxes
            auto issue_s = [&](int j) -> bool {
                const int s = j % kStages;
                const int sb = j & 1;
                if (!wait_phase(k_full(s), static_cast<uint32_t>(j / kStages) & 1u, wc, kSiteMmaFull)) return false;
                if (j >= 2 && !wait_phase(s_free(sb), static_cast<uint32_t>((j >> 1) - 1) & 1u, wc, kSiteMmaAccEmpty))
                    return false;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(sbase + kOffQ + (kk >> 2) * kBoxBytes, 16, 1024) +
                                       static_cast<uint64_t>(((kk & 3) * 32) >> 4);
                    const uint64_t bd = smem_desc_sw128(k_tile(s) + (kk >> 2) * kBoxBytes, 16, 1024) +
                                        static_cast<uint64_t>(((kk & 3) * 32) >> 4);
                    mma_f16(tmem_base + kColS + sb * kBN, a, bd, idesc_s, kk != 0);
                }
                mma_commit(s_full(sb));
                return true;
            };
            // O += P_j V_j: P from TMEM (8 columns per 16 keys), V N-major (d contiguous)
            auto issue_o = [&](int j) -> bool {
                const int s = j % kStages;
                const int sb = j & 1;
                if (!wait_phase(v_full(s), static_cast<uint32_t>(j / kStages) & 1u, wc, kSiteMmaFull)) return false;
                if (!wait_phase(p_full(sb), static_cast<uint32_t>(j >> 1) & 1u, wc, kSiteMmaFull)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(v_tile(s), kBoxBytes, 1024) +
                                        static_cast<uint64_t>((kk * 2048) >> 4);
                    mma_f16_tmem_a(tmem_base + kColO, tmem_base + kColP + sb * (kBN / 2) + kk * 8, bd, idesc_o,
                                   (j != 0) || (kk != 0));
                }
                mma_commit(p_free(sb));
                mma_commit(kv_empty(s));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 1; ok && j <= j_last; ++j) ok = issue_s(j) && issue_o(j - 1);
            if (ok) issue_o(j_last);
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // query row within the block = TMEM lane
        const int q_pos = qt * kBM + row;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const float scale = args.scale_log2;
        float m_run = 0.0f, l_run = 0.0f;
        bool ok = true;
        for (int j = 0; j <= j_last; ++j) {
            const int sb = j & 1;
            const uint32_t use = static_cast<uint32_t>(j >> 1);
            ok = __all_sync(0xFFFFFFFFu, wait_phase(s_full(sb), use & 1u, wc, kSiteEpilogueAccFull));
            if (!ok) break;
            tc_fence_after_sync();
            uint32_t r[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                tmem_ld_32x32b_x32(lane_base + kColS + sb * kBN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(sb));  // the MMA may now write S_{j+2} here

            // mask (keys past the sequence, keys after the query when causal) and row maximum
            const int key0 = j * kBN;
            const int limit = args.causal ? min(args.S, q_pos + 1) : args.S;  // visible keys: < limit
            float mx = -INFINITY;
            if (key0 + kBN > limit) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    if (key0 + c >= limit) r[c] = __float_as_uint(-INFINITY);
                    mx = fmaxf(mx, __uint_as_float(r[c]));
                }
            } else {
#pragma unroll
                for (int c = 0; c < kBN; ++c) mx = fmaxf(mx, __uint_as_float(r[c]));
            }
            const float m_tile = mx * scale;
            float alpha = 1.0f;
            bool rescale = false;
            if (j == 0) {
                m_run = m_tile;
            } else if (m_tile > m_run + kRescaleLog2) {
                alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
                rescale = true;
            }
            // P buffer sb was last read by O += P_{j-2} V_{j-2}
            if (j >= 2) {
                ok = __all_sync(0xFFFFFFFFu, wait_phase(p_free(sb), (use - 1) & 1u, wc, kSiteEpilogueAccFull));
                if (!ok) break;
                tc_fence_after_sync();
            }
            // exponentials, running sum, P (fp16 pairs) into TMEM, 32 keys at a time
            float sum = 0.0f;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(r[32 * c + 2 * e]), scale, -m_run));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(r[32 * c + 2 * e + 1]), scale, -m_run));
                    sum += p0 + p1;
                    pk[e] = pack_half2(p0, p1);
                }
                tmem_st_32x32b_x16(lane_base + kColP + sb * (kBN / 2) + c * 16, pk);
            }
            l_run = l_run * alpha + sum;
            // O row *= alpha once O += P_{j-1} V_{j-1} has landed (any lane of the warp needing it)
            if (j >= 1 && __any_sync(0xFFFFFFFFu, rescale)) {
                ok = __all_sync(0xFFFFFFFFu,
                                wait_phase(p_free((j - 1) & 1), static_cast<uint32_t>((j - 1) >> 1) & 1u, wc,
                                           kSiteEpilogueAccFull));
                if (!ok) break;
                tc_fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < kD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(lane_base + kColO + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_32x32b_x32(lane_base + kColO + c * 32, o);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(sb));
        }
        // O / sum, written as fp16 once the last O += P V has landed
        if (ok && __all_sync(0xFFFFFFFFu, wait_phase(p_free(j_last & 1), static_cast<uint32_t>(j_last >> 1) & 1u, wc,
                                                     kSiteEpilogueAccFull))) {
            tc_fence_after_sync();
            const float inv = 1.0f / l_run;
            __half* dst = args.O + ((static_cast<int64_t>(b) * args.S + q_pos) * args.H + h) * kD;
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(lane_base + kColO + c * 32, o);
                tmem_ld_wait();
                if (q_pos < args.S) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<uint4*>(dst + c * 32)[q] =
                            make_uint4(pack_half2(__uint_as_float(o[8 * q]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                                       pack_half2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                                       pack_half2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                                       pack_half2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

int attn_smem_bytes() { return kSmemAlloc; }

cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        int grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    attn_fwd_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(tmQ, tmK, tmV, a);
    return cudaGetLastError();
}

}  // namespace tg
