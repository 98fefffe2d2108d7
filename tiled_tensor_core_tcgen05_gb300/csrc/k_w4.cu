// Weight-only 4-bit GEMM for skinny M (decode): C = epi(A @ W + bias), where
// W is stored as 4-bit two's-complement integers q with one fp16 scale per
// column and per 128 rows of K, W[k][n] = fp16(q[k][n] * scale[k/128][n]).
//
// "TileLang: writing LLM GPU kernels by thinking in tiles" (section
// "Quantized LLM inference") lays out the shape of such a kernel. The packed
// weights are brought on chip as a tile, converted there, and the converted
// tile feeds the tensor-core product, so no fp16 copy of W ever goes through
// memory. Here the converted tile lives in tensor memory, as the MMA's A
// operand. The swap-AB schedule of the fp16 skinny kernel is kept:
// C^T = W^T A^T, N on the 128-row side of the MMA and M (padded to 16) as its
// N. With the weights stored as N rows of K/2 bytes, the thread that owns
// TMEM lane n decodes row n's own contiguous bytes.
//
// One work unit is a 128-column slice of N times a range of 256-wide K
// blocks. Roles, per CTA:
//   warp 0      TMA producer: per stage, the slice's packed weights
//               (128 x 128 bytes, 128-byte swizzle), A's 256 columns
//               (four 64-wide K-major boxes) and the two scale rows;
//   warp 1      allocates TMEM; one thread issues the MMAs (A from TMEM,
//               A^T from shared memory) and the commits. Consecutive K steps
//               go to up to four accumulators in turn, so an MMA need not
//               wait for the one before it; the epilogue adds them;
//   warps 2-5   epilogue (the skinny kernels' shared epilogue);
//   warps 6-13  converters, two groups of four taking stages in turn. Warp w
//               owns TMEM lanes 32 (w % 4) .. +31. Each thread reads its row's
//               128 bytes and two scales, frees the raw stage, waits for a
//               free TMEM slot, and writes 128 columns of fp16 pairs with
//               tcgen05.st.
// Barriers: raw_full (TMA bytes), raw_empty (4 converter warps + the MMA
// commit), tfull (4 converter warps), tempty (MMA commit), plus the
// accumulator pair of the skinny epilogue.
#include "tg_device.cuh"
#include "tg_internal.h"
#include "tg_skinny.cuh"

namespace tg {
namespace {

constexpr int kRawBytes = kW4BN * (kW4BK / 2);          // 16 KB of packed weights per stage
constexpr int kScaleBytes = 2 * kW4BN * 2;              // two scale rows of 128 fp16
constexpr int kConvWarps = 4 * kW4ConvGroups;
constexpr int kThreads = (6 + kConvWarps) * 32;
constexpr int kMaxSlots = 3;
constexpr uint32_t kTmemCols = 512;
static_assert(kW4BK == 2 * kW4Group, "a stage spans two scale groups");

struct Layout {
    int stage_bytes, act_off, scale_off, ring, bar_raw_full, bar_raw_empty, bar_tfull, bar_tempty, bar_acc_full,
        bar_acc_empty, bar_drain, tmem_slot, abort_slot, flag_slot, used, alloc;
};

__host__ __device__ inline Layout layout_for(int m_pad, int stages) {
    Layout L;
    L.act_off = kRawBytes;                    // 1024-aligned
    L.scale_off = kRawBytes + m_pad * 512;    // m_pad * 512 is a multiple of 8 KB
    L.stage_bytes = (L.scale_off + kScaleBytes + 1023) / 1024 * 1024;
    L.ring = stages * L.stage_bytes;
    L.bar_raw_full = L.ring;
    L.bar_raw_empty = L.bar_raw_full + 8 * stages;
    L.bar_tfull = L.bar_raw_empty + 8 * stages;
    L.bar_tempty = L.bar_tfull + 8 * kMaxSlots;
    L.bar_acc_full = L.bar_tempty + 8 * kMaxSlots;
    L.bar_acc_empty = L.bar_acc_full + 16;
    L.bar_drain = L.bar_acc_empty + 16;
    L.tmem_slot = L.bar_drain + 8;
    L.abort_slot = L.tmem_slot + 4;
    L.flag_slot = L.abort_slot + 4;
    L.used = L.flag_slot + 4;
    L.alloc = L.used + 1024;
    return L;
}

// One 32-bit word of packed weights (eight consecutive k of one column, byte
// p holding k = 2p in its low and 2p + 1 in its high nibble) into four fp16
// pairs, pair p = (w[2p], w[2p+1]) * scale, each product rounded once.
// Byte p is copied under the exponent byte 0x64 in both halves; the masks keep
// the low nibble in the low half and the high nibble (times 16) in the high
// half, and the XOR with 8 maps the two's-complement value q to q + 8. The
// halves then read 1024 + (q_lo + 8) and 1024 + 16 (q_hi + 8), which one fp16
// fused multiply-add maps exactly to (q_lo, q_hi); the scale multiply is the
// only rounding.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, uint32_t* out) {
    const __half2 mul = __halves2half2(__ushort_as_half(0x3C00), __ushort_as_half(0x2C00));  // (1, 1/16)
    const __half2 add = __halves2half2(__ushort_as_half(0xE408), __ushort_as_half(0xD480));  // (-1032, -72)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        uint32_t x = __byte_perm(w, 0x64u, 0x4040u | (0x101u * p));
        x = (x & 0xFFF0FF0Fu) ^ 0x00800008u;
        __half2 h = *reinterpret_cast<__half2*>(&x);
        h = __hmul2(__hfma2(h, mul, add), s2);
        out[p] = *reinterpret_cast<uint32_t*>(&h);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    w4_gemm_kernel(const __grid_constant__ CUtensorMap tmBq, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmS, const W4Args wa) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const SplitArgs& args = wa.s;
    const Layout L = layout_for(args.m_pad, args.stages);
    const int R = args.stages;
    const int T = wa.a_slots;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto raw_full = [&](int s) { return sbase + L.bar_raw_full + 8 * s; };
    auto raw_empty = [&](int s) { return sbase + L.bar_raw_empty + 8 * s; };
    auto tfull = [&](int t) { return sbase + L.bar_tfull + 8 * t; };
    auto tempty = [&](int t) { return sbase + L.bar_tempty + 8 * t; };
    auto acc_full = [&](int b) { return sbase + L.bar_acc_full + 8 * b; };
    auto acc_empty = [&](int b) { return sbase + L.bar_acc_empty + 8 * b; };
    const uint32_t drain_bar = sbase + L.bar_drain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_slot);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L.flag_slot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), 4 + 1);
        }
        for (int t = 0; t < T; ++t) {
            mbar_init(tfull(t), 4);
            mbar_init(tempty(t), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kSkEpiThreads);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmBq);
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmS);
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
            const uint64_t pol_stream = l2_policy_evict_first();  // weights and scales: read once
            const uint64_t pol_keep = l2_policy_evict_last();     // A: re-read by every unit
            const uint32_t tx = static_cast<uint32_t>(kRawBytes + args.m_pad * 512 + kScaleBytes);
            int slot = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int sp = u / args.n_tiles;
                const int nt = u - sp * args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(raw_empty(slot), phase ^ 1, wc, kSiteProducerEmpty)) { ok = false; break; }
                    const uint32_t st = sbase + slot * L.stage_bytes;
                    mbar_arrive_expect_tx(raw_full(slot), tx);
                    tma_load_2d_hint(st, &tmBq, raw_full(slot), kb * (kW4BK / 2), nt * kW4BN, pol_stream);
#pragma unroll
                    for (int j = 0; j < kW4BK / 64; ++j)
                        tma_load_2d_hint(st + L.act_off + j * args.m_pad * 128, &tmA, raw_full(slot),
                                         kb * kW4BK + j * 64, 0, pol_keep);
                    tma_load_2d_hint(st + L.scale_off, &tmS, raw_full(slot), nt * kW4BN, kb * (kW4BK / kW4Group),
                                     pol_stream);
                    issued_mask |= 1u << slot;
                    issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
                    if (++slot == R) { slot = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < R; ++s)
                if (issued_mask & (1u << s)) wait_phase_drain(raw_full(s), (issued_parity >> s) & 1, wc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, args.m_pad, /*a_mn_major=*/false, /*b_mn_major=*/false);
            int slot = 0, ts = 0, ui = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x, ++ui) {
                const int sp = u / args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                const int b = ui & 1;
                if (!wait_phase(acc_empty(b), ((ui >> 1) & 1) ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * args.n_acc * args.tmem_stride;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(raw_full(slot), phase, wc, kSiteMmaFull) ||
                        !wait_phase(tfull(ts), tphase, wc, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t act = sbase + slot * L.stage_bytes + L.act_off;
                    const uint32_t a_tmem = tmem_base + wa.a_col0 + ts * 128;
                    const int nk = min(kW4BK, args.K - kb * kW4BK) / 16;
                    // K step j goes to accumulator j % n_acc: consecutive MMAs are independent
                    for (int j = 0, acc = 0; j < nk; ++j, acc = (acc + 1 == args.n_acc) ? 0 : acc + 1) {
                        const uint64_t b_desc = smem_desc_sw128(act + (j >> 2) * args.m_pad * 128, 16, 1024) +
                                                static_cast<uint64_t>(((j & 3) * 32) >> 4);
                        mma_f16_tmem_a(d_tmem + acc * args.tmem_stride, a_tmem + j * 8, b_desc, idesc,
                                       (kb != kb0) || (j >= args.n_acc));
                    }
                    mma_commit(raw_empty(slot));
                    mma_commit(tempty(ts));
                    if (++slot == R) { slot = 0; phase ^= 1; }
                    if (++ts == T) { ts = 0; tphase ^= 1; }
                }
                if (!ok) break;
                mma_commit(acc_full(b));
            }
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue
        skinny_epilogue<1>(args, tmem_base, acc_full(0), acc_empty(0), last_flag, wc, 64);
    } else {
        // ------------------------------------------------------------ converters
        const int group = (warp - 6) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;  // TMEM lane = output column within the slice
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + wa.a_col0;
        int slot = 0, ts = 0, it = 0;
        uint32_t phase = 0, tphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
            const int sp = u / args.n_tiles;
            const int kb0 = sp * args.kb_per_split;
            const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                if (it % kW4ConvGroups == group) {
                    ok = __all_sync(0xFFFFFFFFu, wait_phase(raw_full(slot), phase, wc, kSiteConvFull));
                    if (!ok) break;
                    const uint32_t st = sbase + slot * L.stage_bytes;
                    // this row's 128 bytes: 16-byte chunk j sits at chunk j ^ (row % 8) (128-byte swizzle)
                    uint4 w[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) w[j] = lds_v4(st + row * 128 + ((j ^ (row & 7)) << 4));
                    const __half2 s_lo = __half2half2(__ushort_as_half(lds_u16(st + L.scale_off + 2 * row)));
                    const __half2 s_hi = __half2half2(__ushort_as_half(lds_u16(st + L.scale_off + 2 * (kW4BN + row))));
                    __syncwarp();
                    if (lane == 0) mbar_arrive(raw_empty(slot));
                    ok = __all_sync(0xFFFFFFFFu, wait_phase(tempty(ts), tphase ^ 1, wc, kSiteConvEmpty));
                    if (!ok) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {  // 64 k per chunk: 32 TMEM columns
                        const __half2 s2 = c < 2 ? s_lo : s_hi;
                        uint32_t r[32];
                        const uint32_t* words = reinterpret_cast<const uint32_t*>(&w[2 * c]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) dequant_word(words[i], s2, &r[4 * i]);
                        tmem_st_32x32b_x32(lane_addr + ts * 128 + c * 32, r);
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tfull(ts));
                }
                if (++slot == R) { slot = 0; phase ^= 1; }
                if (++ts == T) { ts = 0; tphase ^= 1; }
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

int w4_stage_bytes(int m_pad) { return layout_for(m_pad, 1).stage_bytes; }

int w4_stages_for(int m_pad) {
    int s = kW4SmemBudget / w4_stage_bytes(m_pad);
    if (s > 16) s = 16;
    s -= s % kW4ConvGroups;  // each converter group keeps the same ring slots
    if (s < kW4ConvGroups) s = kW4ConvGroups;
    return s;
}

int w4_smem_bytes(int m_pad, int stages) { return layout_for(m_pad, stages).alloc; }

cudaError_t launch_w4(const W4Args& a, const CUtensorMap& tmBq, const CUtensorMap& tmA, const CUtensorMap& tmS,
                      int grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_done[dev]) {
        e = cudaFuncSetAttribute(w4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    w4_gemm_kernel<<<grid, kThreads, w4_smem_bytes(a.s.m_pad, a.s.stages), stream>>>(tmBq, tmA, tmS, a);
    return cudaGetLastError();
}

}  // namespace tg
