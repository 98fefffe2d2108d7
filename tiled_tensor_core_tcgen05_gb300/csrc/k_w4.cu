// Weight-only 4-bit GEMM for skinny M (decode): C = epi(A @ W + bias), where
// W is stored as 4-bit fields with one fp16 scale per column and per 128 rows
// of K, W[k][n] = fp16(v(q[k][n]) * scale[k/128][n]); v is the field's value
// as a two's-complement integer (INT4) or as an FP4 E2M1 number.
//
// "TileLang: writing LLM GPU kernels by thinking in tiles" (section
// "Quantized LLM inference") lays out the shape of such a kernel: the packed
// weights are brought on chip, converted there, and the converted tile feeds
// the tensor-core product, so no fp16 copy of W ever goes through memory.
//
// Orientation. A tcgen05 MMA costs about the same for any N up to 256 but
// grows with its M rows, so the weights sit on the N side: each MMA is
// 128 (tokens, M padded) x 256 (weight columns) x 16. The tokens are the A
// operand, read from tensor memory; the converted weights are the B operand,
// written to shared memory by converter warps as a K-major tile (each weight
// column's 64 k contiguous, 128-byte swizzle). Only M <= 64 runs per launch;
// the host runs larger M as row blocks. The MMA's rows beyond the real tokens
// read whatever tensor memory holds there and land in accumulator rows that
// are never read.
//
// Shared-memory traffic is what bounds this kernel, so each byte crosses it
// as few times as possible: the packed weights go from global memory straight
// into the converters' registers (one stage ahead), and the activations go
// once through shared memory into tensor memory, so per converted weight
// shared memory carries only its fp16 write and the MMA's read of it.
//
// One work unit is a 256-column slice of N times a range of 256-wide K
// blocks (stages). Per CTA:
//   warps 0-1   A loaders, one per tensor-memory lane quarter (rows 0-31 and
//               32-63): per sub-tile, read the activation rows from shared
//               memory, put them in the order of the converted weights, and
//               store them into an A slot of tensor memory as soon as the MMAs
//               that last read that slot are done;
//   warp 2      lane 0: TMA of each stage's activations (four 64-wide boxes
//               of m_pad rows), several stages ahead;
//   warp 3      allocates tensor memory (one 256-column accumulator and eight
//               32-column A slots, one 64-k sub-tile each); lane 0 issues four
//               MMAs per sub-tile and the commits;
//   warps 4-7   epilogue: bias, GELU, C, or fp32 partials plus the
//               deterministic last-arrival reduction for split K;
//   warps 8-23  converters, two groups of 256 threads (one thread per weight
//               column) taking alternate 64-k sub-tiles.
// Barriers: act_full (TMA bytes) / act_empty (A loader warps) for the
// shared-memory activation ring, which the producer keeps several stages
// ahead; a_full (A loader warps) / a_empty (MMA commit) for the eight
// tensor-memory A slots; b_full (the 8 warps of one
// converter group) / b_empty (MMA commit); acc_full / acc_empty (MMA commit /
// the two epilogue warps that read tensor memory).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kSubK = 64;                        // k per B sub-tile (one 128-byte row per column)
constexpr int kSubs = kW4BK / kSubK;             // sub-tiles per stage
constexpr int kSlotBytes = kW4BN * kSubK * 2;    // 32 KB of fp16 per B slot
constexpr int kMmaM = 128;
constexpr int kConvGroups = 2;                   // converter groups, taking alternate sub-tiles
constexpr int kSubsPerGroup = kSubs / kConvGroups;
constexpr int kConvWarps = kConvGroups * kW4BN / 32;
constexpr int kLoadWarps = 2;                    // tensor-memory lane quarters 0 and 1: rows 0..63
constexpr int kProdWarp = 2;
constexpr int kMmaWarp = 3;
constexpr int kEpiWarp0 = 4;                     // warps 4..7 = lane quarters 0..3
constexpr int kEpiThreads = 128;
constexpr int kConvWarp0 = 8;
constexpr int kThreads = (kConvWarp0 + kConvWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc = 0;                  // accumulator, 256 columns
constexpr uint32_t kColA = 256;                  // A slots: 32 columns = one 64-k sub-tile each
constexpr int kASlots = 8;                       // tensor-memory A slots
constexpr int kMaxActStages = 6;                 // shared-memory activation stages (TMA ahead of the loaders)
constexpr int kMaxBSlots = 6;
constexpr uint32_t kEpiSleepNs = 256;   // epilogue: waits about one work unit
constexpr uint32_t kConvSleepNs = 32;   // converters: wait for a free B slot
constexpr uint32_t kLoadSleepNs = 32;   // A loaders
constexpr uint32_t kProdSleepNs = 64;
constexpr uint32_t kMmaSleepNs = 20;
static_assert(kW4BK == 2 * kW4Group, "a stage spans two scale groups");
static_assert(kW4MaxM <= 32 * kLoadWarps, "A loaders cover the rows of one launch");

struct Layout {
    int act_bytes, bring, bar_act_full, bar_act_empty, bar_a_full, bar_a_empty, bar_bfull, bar_bempty,
        bar_acc_full, bar_acc_empty, bar_drain, tmem_slot, abort_slot, flag_slot, used, alloc;
};

// [activation stages][B slots][barriers]. An activation stage holds four
// 64-k boxes of m_pad rows (128-byte swizzle).
__host__ __device__ inline Layout layout_for(int m_pad, int act_stages, int slots) {
    Layout L;
    L.act_bytes = kSubs * m_pad * 128;  // multiple of 8 KB
    L.bring = act_stages * L.act_bytes;
    L.bar_act_full = L.bring + slots * kSlotBytes;
    L.bar_act_empty = L.bar_act_full + 8 * act_stages;
    L.bar_a_full = L.bar_act_empty + 8 * act_stages;
    L.bar_a_empty = L.bar_a_full + 8 * kASlots;
    L.bar_bfull = L.bar_a_empty + 8 * kASlots;
    L.bar_bempty = L.bar_bfull + 8 * slots;
    L.bar_acc_full = L.bar_bempty + 8 * slots;
    L.bar_acc_empty = L.bar_acc_full + 8;
    L.bar_drain = L.bar_acc_empty + 8;
    L.tmem_slot = L.bar_drain + 8;
    L.abort_slot = L.tmem_slot + 4;
    L.flag_slot = L.abort_slot + 4;
    L.used = L.flag_slot + 4;
    L.alloc = L.used + 1024;
    return L;
}

// INT4: one 32-bit word of packed weights (eight consecutive k of one column,
// byte p holding k = 2p in its low and 2p + 1 in its high nibble) into four
// fp16 pairs (value * scale, each product rounded once), in the order
// (k0, k4), (k1, k5), (k2, k6), (k3, k7): the order in which masks that keep
// one nibble of each 16-bit half deliver them. The A loaders put the
// activations in the same order, so the dot product over k is unchanged.
// A nibble masked under the exponent bits 0x64 and XORed with 8 (two's
// complement q -> q + 8) reads 1024 + (q + 8) in the low nibble position and
// 1024 + 16 (q + 8) in the high one; one fp16 fused multiply-add maps either
// exactly to q, and the scale multiply is the only rounding.
__device__ __forceinline__ void dequant_word_int4(uint32_t w, __half2 s2, uint32_t* out) {
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
// fp16); the scale multiply is the only rounding.
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

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 32 bytes of packed weights (64 k of one column) from global memory, read
// once: two 16-byte loads, or one 32-byte load when the base is 32-byte
// aligned.
template <bool kV8>
__device__ __forceinline__ void ldg_weights(const uint8_t* p, uint4& a, uint4& b) {
    if (kV8) {
        asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                     : "l"(p));
    } else {
        asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w)
                     : "l"(p));
        asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                     : "l"(p + 16));
    }
}

// The packed weights and scales one converter thread needs for one stage:
// its column's bytes of its group's two sub-tiles and the stage's two scales.
struct ConvData {
    uint4 w[2 * kSubsPerGroup];
    unsigned short s_lo, s_hi;
};

template <bool kV8>
__device__ __forceinline__ void load_stage(const W4Args& wa, int n, int kb, int group, ConvData& d) {
    const SplitArgs& a = wa.s;
    const bool col_ok = n < a.N;
    const uint8_t* row = wa.Bq + static_cast<int64_t>(n) * (a.K / 2);
#pragma unroll
    for (int jj = 0; jj < kSubsPerGroup; ++jj) {
        const int c = group + kConvGroups * jj;
        const int k0 = kb * kW4BK + c * kSubK;
        if (col_ok && k0 < a.K) {
            ldg_weights<kV8>(row + k0 / 2, d.w[2 * jj], d.w[2 * jj + 1]);
        } else {
            d.w[2 * jj] = make_uint4(0, 0, 0, 0);
            d.w[2 * jj + 1] = make_uint4(0, 0, 0, 0);
        }
    }
    const int g0 = 2 * kb;
    const int groups = a.K / kW4Group;
    const unsigned short* sc = reinterpret_cast<const unsigned short*>(wa.scales);
    d.s_lo = col_ok ? __ldg(sc + static_cast<int64_t>(g0) * a.N + n) : static_cast<unsigned short>(0);
    d.s_hi = (col_ok && g0 + 1 < groups) ? __ldg(sc + static_cast<int64_t>(g0 + 1) * a.N + n)
                                         : static_cast<unsigned short>(0);
}

// The (unit, K block) stage that follows (u, kb) in this CTA's sequence.
__device__ __forceinline__ bool next_stage(const SplitArgs& a, int& u, int& kb, int& kb1) {
    if (++kb < kb1) return true;
    u += gridDim.x;
    if (u >= a.num_units) return false;
    const int sp = u / a.n_tiles;
    kb = sp * a.kb_per_split;
    kb1 = min(a.kb_total, kb + a.kb_per_split);
    return true;
}

template <int kFmt, bool kV8>
__global__ void __launch_bounds__(kThreads, 1)
    w4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const W4Args wa) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const SplitArgs& args = wa.s;
    const int T = wa.b_slots;
    const int NA = wa.act_stages;
    const Layout L = layout_for(args.m_pad, NA, T);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int loaders = args.m_pad > 32 ? 2 : 1;  // A loader warps with rows to store

    auto act_full = [&](int s) { return sbase + L.bar_act_full + 8 * s; };
    auto act_empty = [&](int s) { return sbase + L.bar_act_empty + 8 * s; };
    auto a_full = [&](int s) { return sbase + L.bar_a_full + 8 * s; };
    auto a_empty = [&](int s) { return sbase + L.bar_a_empty + 8 * s; };
    auto bfull = [&](int t) { return sbase + L.bar_bfull + 8 * t; };
    auto bempty = [&](int t) { return sbase + L.bar_bempty + 8 * t; };
    const uint32_t acc_full = sbase + L.bar_acc_full, acc_empty = sbase + L.bar_acc_empty;
    const uint32_t drain_bar = sbase + L.bar_drain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_slot);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L.flag_slot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NA; ++s) {
            mbar_init(act_full(s), 1);
            mbar_init(act_empty(s), loaders);
        }
        for (int s = 0; s < kASlots; ++s) {
            mbar_init(a_full(s), loaders);
            mbar_init(a_empty(s), 1);
        }
        for (int t = 0; t < T; ++t) {
            mbar_init(bfull(t), kConvWarps / kConvGroups);
            mbar_init(bempty(t), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2);  // epilogue warps 4 and 5 (lane quarters 0 and 1)
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wc{abort_flag, args.wd.status, args.wd.limit_ns};

    if (warp < kLoadWarps) {
        // ------------------------------------------------------------ A loaders
        // thread = row (warp * 32 + lane) = its tensor-memory lane; per stage its 256 k
        // become 128 columns of the A slot, two fp16 per column
        if (warp < loaders) {
            const int row = warp * 32 + lane;
            const bool has_row = row < args.m_pad;
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
            const uint32_t swz = static_cast<uint32_t>(row & 7);
            int as = 0, ts = 0;
            uint32_t aphase = 0, tphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int sp = u / args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    // the stage's activations have landed in shared memory
                    ok = __all_sync(0xFFFFFFFFu, wait_phase_sleep(act_full(as), aphase, wc, kSiteConvFull,
                                                                  kLoadSleepNs));
                    if (!ok) break;
                    const uint32_t sa = sbase + as * L.act_bytes;
#pragma unroll 1
                    for (int c = 0; c < kSubs; ++c) {
                        // the MMAs that last read this sub-tile slot are done
                        ok = __all_sync(0xFFFFFFFFu, wait_phase(a_empty(ts), tphase ^ 1, wc, kSiteConvEmpty));
                        if (!ok) break;
                        tc_fence_after_sync();
                        uint32_t r[32];
                        if (has_row) {
                            const uint32_t box = sa + c * args.m_pad * 128 + row * 128;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {  // 16-byte chunk i: k = 8i .. 8i+7
                                const uint4 v = lds_v4(box + ((static_cast<uint32_t>(i) ^ swz) << 4));
                                if (kFmt == 0) {  // (a0, a4), (a1, a5), (a2, a6), (a3, a7)
                                    r[4 * i + 0] = __byte_perm(v.x, v.z, 0x5410);
                                    r[4 * i + 1] = __byte_perm(v.x, v.z, 0x7632);
                                    r[4 * i + 2] = __byte_perm(v.y, v.w, 0x5410);
                                    r[4 * i + 3] = __byte_perm(v.y, v.w, 0x7632);
                                } else {  // natural order
                                    r[4 * i + 0] = v.x;
                                    r[4 * i + 1] = v.y;
                                    r[4 * i + 2] = v.z;
                                    r[4 * i + 3] = v.w;
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) r[i] = 0u;
                        }
                        tmem_st_32x32b_x32(lane_addr + kColA + ts * 32, r);
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(a_full(ts));
                        if (++ts == kASlots) { ts = 0; tphase ^= 1; }
                    }
                    if (!ok) break;
                    if (lane == 0) mbar_arrive(act_empty(as));  // every sub-tile of the stage was read
                    if (++as == NA) { as = 0; aphase ^= 1; }
                }
            }
        }
    } else if (warp == kProdWarp) {
        // ------------------------------------------------------------ activations + L2 prefetch
        if (lane == 0) {
            const uint64_t pol_keep = l2_policy_evict_last();  // A: re-read by every unit
            int as = 0;
            uint32_t aphase = 0, a_mask = 0, a_parity = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int sp = u / args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase_sleep(act_empty(as), aphase ^ 1, wc, kSiteProducerEmpty, kProdSleepNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + as * L.act_bytes;
                    mbar_arrive_expect_tx(act_full(as), L.act_bytes);
#pragma unroll
                    for (int j = 0; j < kSubs; ++j)
                        tma_load_2d_hint(sa + j * args.m_pad * 128, &tmA, act_full(as), kb * kW4BK + j * kSubK, 0,
                                         pol_keep);
                    a_mask |= 1u << as;
                    a_parity = (a_parity & ~(1u << as)) | (aphase << as);
                    if (++as == NA) { as = 0; aphase ^= 1; }
                }
            }
            for (int s = 0; s < NA; ++s)
                if (a_mask & (1u << s)) wait_phase_drain(act_full(s), (a_parity >> s) & 1, wc);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kMmaM, kW4BN, /*a_mn_major=*/false, /*b_mn_major=*/false);
            int as = 0, ts = 0, ui = 0;
            uint32_t aphase = 0, tphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x, ++ui) {
                const int sp = u / args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                // one accumulator: the previous unit's epilogue must have read it
                if (!wait_phase(acc_empty, (ui & 1) ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + kColAcc;
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    const int subs = min(kW4BK, args.K - kb * kW4BK) / kSubK;  // K % 128 == 0: 2 or 4
                    for (int c = 0; c < kSubs; ++c) {
                        if (!wait_phase(a_full(as), aphase, wc, kSiteMmaFull) ||
                            !wait_phase_sleep(bfull(ts), tphase, wc, kSiteMmaFull, kMmaSleepNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        if (c < subs) {
                            const uint32_t a_tmem = tmem_base + kColA + as * 32;
                            const uint64_t b_desc = smem_desc_sw128(sbase + L.bring + ts * kSlotBytes, 16, 1024);
#pragma unroll
                            for (int k = 0; k < kSubK / 16; ++k)
                                mma_f16_tmem_a(d_tmem, a_tmem + k * 8, b_desc + static_cast<uint64_t>((k * 32) >> 4),
                                               idesc, (kb != kb0) || (c != 0) || (k != 0));
                        }
                        mma_commit(bempty(ts));
                        mma_commit(a_empty(as));
                        if (++ts == T) { ts = 0; tphase ^= 1; }
                        if (++as == kASlots) { as = 0; aphase ^= 1; }
                    }
                }
                if (!ok) break;
                mma_commit(acc_full);
            }
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else if (warp < kConvWarp0) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;         // warps 4..7: lane quarters 0..3
        const int ept = threadIdx.x - kEpiWarp0 * 32;
        const int row = quarter * 32 + lane;  // accumulator row = tensor-memory lane
        const bool reads_tmem = quarter < 2;  // rows 0..63
        const bool row_ok = reads_tmem && row < args.M;
        const bool vec = wa.c_vec != 0;
        int it = 0;
        for (int u = blockIdx.x; u < args.num_units; u += gridDim.x, ++it) {
            const int sp = u / args.n_tiles;
            const int nt = u - sp * args.n_tiles;
            const int n0 = nt * kW4BN;
            const bool ok = wait_phase_sleep(acc_full, it & 1, wc, kSiteEpilogueAccFull, kEpiSleepNs);
            if (named_barrier_or(1, kEpiThreads, !ok)) break;
            tc_fence_after_sync();
            if (reads_tmem) {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + kColAcc;
#pragma unroll 1
                for (int c = 0; c < kW4BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + c * 32, r);
                    tmem_ld_wait();
                    if (c == kW4BN / 32 - 1) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(acc_empty);
                    }
                    const int col0 = n0 + c * 32;
                    if (!row_ok || col0 >= args.N) continue;
                    if (args.splits == 1) {
                        __half* dst = args.C + static_cast<int64_t>(row) * args.N + col0;
                        const bool whole = vec && col0 + 32 <= args.N;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // eight columns at a time
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int n = col0 + 8 * q + e;
                                const float bi =
                                    (args.bias != nullptr && n < args.N) ? __half2float(args.bias[n]) : 0.0f;
                                v[e] = epi_value(__uint_as_float(r[8 * q + e]), bi, args.gelu);
                            }
                            if (whole) {
                                uint4 o;
                                __half2* h = reinterpret_cast<__half2*>(&o);
#pragma unroll
                                for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
                                reinterpret_cast<uint4*>(dst)[q] = o;
                            } else {
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    if (col0 + 8 * q + e < args.N) dst[8 * q + e] = __float2half_rn(v[e]);
                            }
                        }
                    } else {
                        // partials as [slice][m_pad][N] fp32: this thread's 32 columns are 128 contiguous bytes
                        float* wp = args.ws + (static_cast<int64_t>(sp) * args.m_pad + row) * args.N + col0;
                        if (col0 + 32 <= args.N) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                reinterpret_cast<uint4*>(wp)[q] =
                                    make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (col0 + i < args.N) wp[i] = __uint_as_float(r[i]);
                        }
                    }
                }
            }
            if (args.splits > 1) {
                // publish this slice's partials, then count arrivals for column slice nt
                __threadfence();
                named_barrier_sync(1, kEpiThreads);
                if (ept == 0) {
                    const unsigned int prev = atomicAdd(args.counters + nt, 1u);
                    *last_flag = (prev == static_cast<unsigned int>(args.splits - 1)) ? 1 : 0;
                }
                named_barrier_sync(1, kEpiThreads);
                if (*last_flag) {
                    __threadfence();
                    // every (row, column) of the slice: thread t takes four adjacent
                    // columns (float4) of rows t/64, t/64 + 2, ...; per batch of four rows
                    // all slices' loads are issued before the sums, which run in slice
                    // order 0, 1, ... (deterministic); then bias, GELU and C
                    const int cq = ept & 63;
                    const int n = n0 + 4 * cq;
                    const int64_t slice_stride = static_cast<int64_t>(args.m_pad) * args.N;
                    if (n < args.N) {
                        float bi[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            bi[e] = (args.bias != nullptr && n + e < args.N) ? __half2float(args.bias[n + e]) : 0.0f;
                        for (int m0 = ept >> 6; m0 < args.M; m0 += 8) {
                            float4 acc[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int q0 = 0; q0 < args.splits; q0 += 2) {
                                float4 p[2][4];
#pragma unroll
                                for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                                    for (int i = 0; i < 4; ++i) {
                                        const int m = m0 + 2 * i;
                                        p[qq][i] = (q0 + qq < args.splits && m < args.M)
                                                       ? __ldcg(reinterpret_cast<const float4*>(
                                                             args.ws + (q0 + qq) * slice_stride +
                                                             static_cast<int64_t>(m) * args.N + n))
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                                    }
#pragma unroll
                                for (int qq = 0; qq < 2; ++qq)
#pragma unroll
                                    for (int i = 0; i < 4; ++i)
                                        if (q0 + qq < args.splits) {
                                            acc[i].x += p[qq][i].x;
                                            acc[i].y += p[qq][i].y;
                                            acc[i].z += p[qq][i].z;
                                            acc[i].w += p[qq][i].w;
                                        }
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int m = m0 + 2 * i;
                                if (m >= args.M) break;
                                __half* dst = args.C + static_cast<int64_t>(m) * args.N + n;
                                const float v[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (n + e < args.N) dst[e] = __float2half_rn(epi_value(v[e], bi[e], args.gelu));
                            }
                        }
                    }
                    if (ept == 0) atomicExch(args.counters + nt, 0u);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ converters
        // kConvGroups groups of kW4BN threads; group g converts sub-tiles
        // c = g, g + kConvGroups, ... of every stage. Sub-tile c of the CTA's
        // stage number it is the (4 it + c)-th B slot use, so with
        // T % kConvGroups == 0 each slot is only ever filled by one group. Each
        // thread holds the next stage's packed weights in registers while it
        // converts the current one.
        const int cidx = threadIdx.x - kConvWarp0 * 32;
        const int group = cidx / kW4BN;
        const int col = cidx - group * kW4BN;  // weight column within the unit's slice (0..255)
        const uint32_t swz = static_cast<uint32_t>(col & 7);
        // converts stage number `it` from `d` into this group's B slots; false once a wait gave up
        auto convert = [&](const ConvData& d, int it) -> bool {
            const __half2 s_lo = __half2half2(__ushort_as_half(d.s_lo));
            const __half2 s_hi = __half2half2(__ushort_as_half(d.s_hi));
            bool ok = true;
            // fully unrolled (no exit inside), so the weights stay in registers
#pragma unroll
            for (int jj = 0; jj < kSubsPerGroup; ++jj) {  // 64 k per sub-tile: this column's 128-byte row of B
                const int c = group + kConvGroups * jj;
                const int use = it * kSubs + c;  // B slot use number
                const int ts = use % T;
                const uint32_t tphase = static_cast<uint32_t>(use / T) & 1u;
                if (ok)
                    ok = __all_sync(0xFFFFFFFFu,
                                    wait_phase_sleep(bempty(ts), tphase ^ 1, wc, kSiteConvEmpty, kConvSleepNs));
                if (ok) {
                    const __half2 s2 = (c * kSubK < kW4Group) ? s_lo : s_hi;
                    const uint32_t dst = sbase + L.bring + ts * kSlotBytes + col * 128;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {  // word i: k = 8i .. 8i+7 -> 16-byte chunk i
                        const uint4& q4 = d.w[2 * jj + (i >> 2)];
                        const uint32_t word = (i & 3) == 0 ? q4.x : (i & 3) == 1 ? q4.y : (i & 3) == 2 ? q4.z : q4.w;
                        uint32_t o[4];
                        if (kFmt == 0)
                            dequant_word_int4(word, s2, o);
                        else
                            dequant_word_fp4(word, s2, o);
                        sts_v4(dst + ((static_cast<uint32_t>(i) ^ swz) << 4), o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bfull(ts));
                }
            }
            return ok;
        };
        // two register buffers used in turn: the next stage's packed weights load into one while
        // the other is converted
        int u = blockIdx.x;
        if (u < args.num_units) {
            int kb = (u / args.n_tiles) * args.kb_per_split;
            int kb1 = min(args.kb_total, kb + args.kb_per_split);
            ConvData b0, b1;
            load_stage<kV8>(wa, (u % args.n_tiles) * kW4BN + col, kb, group, b0);
            for (int it = 0;; it += 2) {
                bool more = next_stage(args, u, kb, kb1);
                if (more) load_stage<kV8>(wa, (u % args.n_tiles) * kW4BN + col, kb, group, b1);
                if (!convert(b0, it) || !more) break;
                more = next_stage(args, u, kb, kb1);
                if (more) load_stage<kV8>(wa, (u % args.n_tiles) * kW4BN + col, kb, group, b0);
                if (!convert(b1, it + 1) || !more) break;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int kFmt, bool kV8>
cudaError_t launch_w4_t(const W4Args& a, const CUtensorMap& tmA, int grid, cudaStream_t stream) {
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(w4_gemm_kernel<kFmt, kV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_gen[dev] = g_generation;
    }
    w4_gemm_kernel<kFmt, kV8>
        <<<grid, kThreads, layout_for(a.s.m_pad, a.act_stages, a.b_slots).alloc, stream>>>(tmA, a);
    return cudaGetLastError();
}

}  // namespace

// Ring depths for a padded M within the shared-memory budget: the deepest
// converted-weight ring (a multiple of the converter groups) that leaves room
// for at least three activation stages (two for the largest M), then as many
// activation stages as fit, up to kMaxActStages.
void w4_pipeline(int m_pad, int* act_stages, int* slots) {
    const int min_act = m_pad > 32 ? 2 : 3;
    int t = kMaxBSlots;
    while (t > kConvGroups && layout_for(m_pad, min_act, t).alloc > kW4SmemBudget) t -= kConvGroups;
    int na = min_act;
    while (na < kMaxActStages && layout_for(m_pad, na + 1, t).alloc <= kW4SmemBudget) ++na;
    *act_stages = na;
    *slots = t;
}

int w4_smem_bytes(int m_pad, int act_stages, int slots) { return layout_for(m_pad, act_stages, slots).alloc; }

cudaError_t launch_w4(const W4Args& a, const CUtensorMap& tmA, int grid, cudaStream_t stream) {
    if (a.fmt == 1)
        return a.bq_v8 ? launch_w4_t<1, true>(a, tmA, grid, stream) : launch_w4_t<1, false>(a, tmA, grid, stream);
    return a.bq_v8 ? launch_w4_t<0, true>(a, tmA, grid, stream) : launch_w4_t<0, false>(a, tmA, grid, stream);
}

}  // namespace tg
