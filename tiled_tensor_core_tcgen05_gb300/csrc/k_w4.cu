// Weight-only 4-bit GEMM for skinny M (decode): C = epi(A @ W + bias), where
// W is stored as 4-bit fields with one fp16 scale per column and per 128 rows
// of K, W[k][n] = fp16(v(q[k][n]) * scale[k/128][n]); v is the field's value
// as a two's-complement integer (INT4) or as an FP4 E2M1 number.
//
// "TileLang: writing LLM GPU kernels by thinking in tiles" (section
// "Quantized LLM inference") lays out the shape of such a kernel. The packed
// weights are brought on chip as a tile, converted there, and the converted
// tile feeds the tensor-core product, so no fp16 copy of W ever goes through
// memory.
//
// Orientation. A tcgen05 MMA costs about the same for any N up to 256 but
// grows with its M rows, so the weights sit on the N side: the MMA is
// 64 (tokens, M padded) x 256 (weight columns) x 16, A = the activations from
// shared memory, B = the converted weights, written to shared memory by the
// converter warps as a K-major tile (each weight column's 64 k contiguous,
// 128-byte swizzle). Only M <= 64 runs per launch; the host runs larger M as
// several row blocks. The activation boxes hold only the m_pad real rows; the
// MMA's remaining rows read whatever follows in shared memory and land in
// accumulator rows that are never stored.
//
// One work unit is a 256-column slice of N times a range of 256-wide K
// blocks. Per CTA:
//   warp 0      TMA producer, per 256-k stage: the slice's packed weights
//               (256 rows x 128 bytes, 128-byte swizzle) and the two scale
//               rows into a raw stage, A's 256 columns (four 64-wide boxes
//               of m_pad rows) into an activation slot;
//   warp 1      allocates TMEM (two 256-column accumulators); one thread
//               issues four MMAs per 64-k sub-tile and the commits;
//   warps 2-5   epilogue: TMEM lane 32q + i (i < 16) holds accumulator row
//               16q + i; bias, GELU, C, or fp32 partials plus the
//               deterministic last-arrival reduction for split K;
//   warps 6-21  converters, two groups of 256 threads (one thread per weight
//               column) taking alternate 64-k sub-tiles: read the column's
//               bytes of its sub-tiles and two scales once per stage, then
//               write the sub-tiles as fp16 into a ring of B slots (for INT4
//               in the pair order of dequant_word, with the group's activation
//               chunks reordered to match; for FP4 in natural order).
// Barriers: raw_full (TMA bytes), raw_empty (16 converter warps), afull (TMA
// bytes), aempty (MMA commit after the stage's last sub-tile), bfull (the 8
// warps of one converter group), bempty (MMA commit), acc_full / acc_empty
// (MMA commit / 128 epilogue threads).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kRawBytes = kW4BN * (kW4BK / 2);   // 32 KB of packed weights per stage
constexpr int kScaleBytes = 2 * kW4BN * 2;       // two scale rows of 256 fp16
constexpr int kSubK = 64;                        // k per B sub-tile (one 128-byte row per column)
constexpr int kSubs = kW4BK / kSubK;             // sub-tiles per stage
constexpr int kSlotBytes = kW4BN * kSubK * 2;    // 32 KB of fp16 per B slot
constexpr int kMmaM = 64;
constexpr int kConvGroups = 2;                   // converter groups, taking alternate sub-tiles
constexpr int kSubsPerGroup = 4 / kConvGroups;
constexpr int kConvWarps = kConvGroups * kW4BN / 32;
constexpr int kEpiThreads = 128;
constexpr int kThreads = (6 + kConvWarps) * 32;
constexpr uint32_t kTmemCols = 512;              // two 256-column accumulators
constexpr int kMaxStages = 8;
constexpr uint32_t kEpiSleepNs = 256;   // epilogue: waits about one work unit
constexpr uint32_t kConvSleepNs = 32;   // converters: wait for a TMA stage or a free B slot
constexpr int kPrefetchStages = 2;      // packed-weight boxes requested into L2 ahead of their load
// The producer and MMA threads share schedulers with converter warps, so
// their waits sleep too (briefly) instead of taking issue slots.
constexpr uint32_t kProdSleepNs = 64;
constexpr uint32_t kMmaSleepNs = 20;
static_assert(kW4BK == 2 * kW4Group, "a stage spans two scale groups");

struct Layout {
    int stage_bytes, scale_off, act_bytes, aring, bring, bar_raw_full, bar_raw_empty, bar_afull, bar_aempty,
        bar_bfull, bar_bempty, bar_acc_full, bar_acc_empty, bar_drain, tmem_slot, abort_slot, flag_slot, used,
        alloc;
};

// [raw stages][activation slots][B slots][barriers]. Raw stages (packed
// weights + scales) are freed as soon as the converters have read them;
// activation slots (four 64-k boxes of m_pad rows) when the stage's MMAs are
// done. A box's 64-row MMA window (8 KB) may run past its slot; the B ring
// behind the activation slots keeps it inside the CTA's shared memory.
__host__ __device__ inline Layout layout_for(int m_pad, int stages, int act_slots, int slots) {
    Layout L;
    L.scale_off = kRawBytes;
    L.stage_bytes = kRawBytes + kScaleBytes;  // multiple of 1024
    L.act_bytes = kSubs * m_pad * 128;       // multiple of 8 KB
    L.aring = stages * L.stage_bytes;
    L.bring = L.aring + act_slots * L.act_bytes;
    L.bar_raw_full = L.bring + slots * kSlotBytes;
    L.bar_raw_empty = L.bar_raw_full + 8 * stages;
    L.bar_afull = L.bar_raw_empty + 8 * stages;
    L.bar_aempty = L.bar_afull + 8 * act_slots;
    L.bar_bfull = L.bar_aempty + 8 * act_slots;
    L.bar_bempty = L.bar_bfull + 8 * slots;
    L.bar_acc_full = L.bar_bempty + 8 * slots;
    L.bar_acc_empty = L.bar_acc_full + 16;
    L.bar_drain = L.bar_acc_empty + 16;
    L.tmem_slot = L.bar_drain + 8;
    L.abort_slot = L.tmem_slot + 4;
    L.flag_slot = L.abort_slot + 4;
    L.used = L.flag_slot + 4;
    L.alloc = L.used + 1024;
    return L;
}

// In-place reorder of one 16-byte chunk of activations (eight consecutive k)
// to the order dequant_word gives the weights: (a0, a4, a1, a5, a2, a6, a3, a7).
__device__ __forceinline__ void permute_chunk(uint32_t addr) {
    const uint4 v = lds_v4(addr);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(__byte_perm(v.x, v.z, 0x5410)),
                 "r"(__byte_perm(v.x, v.z, 0x7632)), "r"(__byte_perm(v.y, v.w, 0x5410)),
                 "r"(__byte_perm(v.y, v.w, 0x7632))
                 : "memory");
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Accumulator row of TMEM lane (32 q + i) for a 64-row MMA: row 16 q + i for
// i < 16; lanes 16..31 of each quarter hold no row (-1).
__device__ __forceinline__ int acc_row(int quarter, int lane) { return lane < 16 ? quarter * 16 + lane : -1; }

template <int kFmt>
__global__ void __launch_bounds__(kThreads, 1)
    w4_gemm_kernel(const __grid_constant__ CUtensorMap tmBq, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmS, const W4Args wa) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const SplitArgs& args = wa.s;
    const int R = args.stages;
    const int RA = wa.a_slots;
    const int T = wa.b_slots;
    const Layout L = layout_for(args.m_pad, R, RA, T);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto raw_full = [&](int s) { return sbase + L.bar_raw_full + 8 * s; };
    auto raw_empty = [&](int s) { return sbase + L.bar_raw_empty + 8 * s; };
    auto afull = [&](int s) { return sbase + L.bar_afull + 8 * s; };
    auto aempty = [&](int s) { return sbase + L.bar_aempty + 8 * s; };
    auto bfull = [&](int t) { return sbase + L.bar_bfull + 8 * t; };
    auto bempty = [&](int t) { return sbase + L.bar_bempty + 8 * t; };
    auto acc_full = [&](int b) { return sbase + L.bar_acc_full + 8 * b; };
    auto acc_empty = [&](int b) { return sbase + L.bar_acc_empty + 8 * b; };
    const uint32_t drain_bar = sbase + L.bar_drain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_slot);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L.flag_slot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(raw_full(s), 1);
            mbar_init(raw_empty(s), kConvWarps);
        }
        for (int s = 0; s < RA; ++s) {
            mbar_init(afull(s), 1);
            mbar_init(aempty(s), 1);
        }
        for (int t = 0; t < T; ++t) {
            mbar_init(bfull(t), kConvWarps / kConvGroups);
            mbar_init(bempty(t), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), kEpiThreads);
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
            int slot = 0, as = 0;
            uint32_t phase = 0, aphase = 0;
            uint32_t issued_mask = 0, issued_parity = 0, a_mask = 0, a_parity = 0;
            bool ok = true;
            // L2 prefetch cursor, kPrefetchStages stages ahead of the loads in
            // this CTA's sequence of (unit, K block) stages: the SMEM ring holds
            // few stages, so HBM requests are issued earlier through L2
            int pu = blockIdx.x, pkb = 0, pkb1 = 0;
            auto pf_unit = [&](int u) {
                const int sp = u / args.n_tiles;
                pkb = sp * args.kb_per_split;
                pkb1 = min(args.kb_total, pkb + args.kb_per_split);
            };
            auto pf_issue = [&]() {
                if (pu >= args.num_units) return;
                tma_prefetch_l2_2d(&tmBq, pkb * (kW4BK / 2), (pu % args.n_tiles) * kW4BN);
                if (++pkb == pkb1) {
                    pu += gridDim.x;
                    if (pu < args.num_units) pf_unit(pu);
                }
            };
            if (pu < args.num_units) pf_unit(pu);
            for (int i = 0; i < kPrefetchStages; ++i) pf_issue();
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int sp = u / args.n_tiles;
                const int nt = u - sp * args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase_sleep(raw_empty(slot), phase ^ 1, wc, kSiteProducerEmpty, kProdSleepNs)) {
                        ok = false;
                        break;
                    }
                    pf_issue();
                    const uint32_t st = sbase + slot * L.stage_bytes;
                    mbar_arrive_expect_tx(raw_full(slot), kRawBytes + kScaleBytes);
                    tma_load_2d_hint(st, &tmBq, raw_full(slot), kb * (kW4BK / 2), nt * kW4BN, pol_stream);
                    tma_load_2d_hint(st + L.scale_off, &tmS, raw_full(slot), nt * kW4BN, kb * (kW4BK / kW4Group),
                                     pol_stream);
                    issued_mask |= 1u << slot;
                    issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
                    if (++slot == R) { slot = 0; phase ^= 1; }
                    if (!wait_phase_sleep(aempty(as), aphase ^ 1, wc, kSiteProducerEmpty, kProdSleepNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = sbase + L.aring + as * L.act_bytes;
                    mbar_arrive_expect_tx(afull(as), L.act_bytes);
#pragma unroll
                    for (int j = 0; j < kSubs; ++j)
                        tma_load_2d_hint(sa + j * args.m_pad * 128, &tmA, afull(as), kb * kW4BK + j * kSubK, 0, pol_keep);
                    a_mask |= 1u << as;
                    a_parity = (a_parity & ~(1u << as)) | (aphase << as);
                    if (++as == RA) { as = 0; aphase ^= 1; }
                }
            }
            for (int s = 0; s < R; ++s)
                if (issued_mask & (1u << s)) wait_phase_drain(raw_full(s), (issued_parity >> s) & 1, wc);
            for (int s = 0; s < RA; ++s)
                if (a_mask & (1u << s)) wait_phase_drain(afull(s), (a_parity >> s) & 1, wc);
        }
    } else if (warp == 1) {
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
                const int b = ui & 1;
                if (!wait_phase(acc_empty(b), ((ui >> 1) & 1) ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kW4BN;
                for (int kb = kb0; kb < kb1 && ok; ++kb) {
                    if (!wait_phase(afull(as), aphase, wc, kSiteMmaFull)) { ok = false; break; }
                    const uint32_t act = sbase + L.aring + as * L.act_bytes;
                    const int subs = min(kW4BK, args.K - kb * kW4BK) / kSubK;  // K % 128 == 0: 2 or 4
                    for (int c = 0; c < kSubs; ++c) {
                        if (!wait_phase_sleep(bfull(ts), tphase, wc, kSiteMmaFull, kMmaSleepNs)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        if (c < subs) {
                            const uint64_t a_desc = smem_desc_sw128(act + c * args.m_pad * 128, 16, 1024);
                            const uint64_t b_desc = smem_desc_sw128(sbase + L.bring + ts * kSlotBytes, 16, 1024);
#pragma unroll
                            for (int k = 0; k < kSubK / 16; ++k)
                                mma_f16(d_tmem, a_desc + static_cast<uint64_t>((k * 32) >> 4),
                                        b_desc + static_cast<uint64_t>((k * 32) >> 4), idesc,
                                        (kb != kb0) || (c != 0) || (k != 0));
                        }
                        mma_commit(bempty(ts));
                        if (++ts == T) { ts = 0; tphase ^= 1; }
                    }
                    if (!ok) break;
                    mma_commit(aempty(as));
                    if (++as == RA) { as = 0; aphase ^= 1; }
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
        const int quarter = warp & 3;
        const int ept = threadIdx.x - 64;
        const int row = acc_row(quarter, lane);
        const bool row_ok = row >= 0 && row < args.M;
        const bool vec = wa.c_vec != 0;
        int it = 0;
        for (int u = blockIdx.x; u < args.num_units; u += gridDim.x, ++it) {
            const int sp = u / args.n_tiles;
            const int nt = u - sp * args.n_tiles;
            const int n0 = nt * kW4BN;
            const int b = it & 1;
            const bool ok = wait_phase_sleep(acc_full(b), (it >> 1) & 1, wc, kSiteEpilogueAccFull, kEpiSleepNs);
            if (named_barrier_or(1, kEpiThreads, !ok)) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kW4BN;
#pragma unroll 1
            for (int c = 0; c < kW4BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_ld_wait();
                if (c == kW4BN / 32 - 1) {
                    tc_fence_before_sync();
                    mbar_arrive(acc_empty(b));
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
                            const float bi = (args.bias != nullptr && n < args.N) ? __half2float(args.bias[n]) : 0.0f;
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
                    const int64_t off = (static_cast<int64_t>(sp) * args.m_pad + row) * args.N + col0;
                    if (!dbg_check(dbg_in(off, min(32, args.N - col0), args.wd.ws_floats), args.wd)) continue;
                    float* wp = args.ws + off;
                    if (col0 + 32 <= args.N) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<uint4*>(wp)[q] = make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + i < args.N) wp[i] = __uint_as_float(r[i]);
                    }
                }
            }
            if (args.splits > 1) {
                // publish this slice's partials, then count arrivals for column slice nt
                __threadfence();
                named_barrier_sync(1, kEpiThreads);
                if (ept == 0) {
                    *last_flag = 0;
                    if (dbg_check(dbg_in(nt, 1, args.wd.n_counters), args.wd)) {
                        const unsigned int prev = atomicAdd(args.counters + nt, 1u);
                        *last_flag = (prev == static_cast<unsigned int>(args.splits - 1)) ? 1 : 0;
                    }
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
                                        const int64_t off =
                                            (q0 + qq) * slice_stride + static_cast<int64_t>(m) * args.N + n;
                                        p[qq][i] = (q0 + qq < args.splits && m < args.M &&
                                                    dbg_check(dbg_in(off, 4, args.wd.ws_floats), args.wd))
                                                       ? __ldcg(reinterpret_cast<const float4*>(args.ws + off))
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
        // T % kConvGroups == 0 each slot is only ever filled by one group.
        const int cidx = threadIdx.x - 6 * 32;
        const int group = cidx / kW4BN;
        const int col = cidx - group * kW4BN;  // weight column within the unit's slice (0..255)
        const uint32_t swz = static_cast<uint32_t>(col & 7);
        int slot = 0, it = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
            const int sp = u / args.n_tiles;
            const int kb0 = sp * args.kb_per_split;
            const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                ok = __all_sync(0xFFFFFFFFu, wait_phase_sleep(raw_full(slot), phase, wc, kSiteConvFull, kConvSleepNs));
                if (!ok) break;
                const uint32_t st = sbase + slot * L.stage_bytes;
                // this column's bytes of this group's sub-tiles: 16-byte chunk j of the
                // 128-byte row sits at chunk j ^ (col % 8) (128-byte swizzle)
                uint4 w[2 * kSubsPerGroup];
#pragma unroll
                for (int jj = 0; jj < kSubsPerGroup; ++jj)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t chunk = static_cast<uint32_t>(2 * (group + kConvGroups * jj) + h);
                        w[2 * jj + h] = lds_v4(st + col * 128 + ((chunk ^ swz) << 4));
                    }
                const __half2 s_lo = __half2half2(__ushort_as_half(lds_u16(st + L.scale_off + 2 * col)));
                const __half2 s_hi = __half2half2(__ushort_as_half(lds_u16(st + L.scale_off + 2 * (kW4BN + col))));
                // the next TMA write into this stage is an async-proxy write after these
                // generic-proxy reads: without the proxy fence it can land before them
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(raw_empty(slot));
                // INT4: this group's activation boxes of the stage, permuted like the weights; the
                // MMA reads a box only after this group's bfull arrive for its sub-tile
                if (kFmt == 0) {
                    const int as = it % RA;
                    ok = __all_sync(0xFFFFFFFFu, wait_phase_sleep(afull(as), static_cast<uint32_t>(it / RA) & 1u, wc,
                                                                  kSiteConvFull, kConvSleepNs));
                    if (!ok) break;
                    const uint32_t sa = sbase + L.aring + as * L.act_bytes;
                    const int chunks = args.m_pad * 8;  // 16-byte chunks per 64-k box
#pragma unroll
                    for (int jj = 0; jj < kSubsPerGroup; ++jj) {
                        const uint32_t box = sa + (group + kConvGroups * jj) * args.m_pad * 128;
                        for (int t = col; t < chunks; t += kW4BN) permute_chunk(box + 16 * t);
                    }
                }
                // fully unrolled (no exit inside), so w[] stays in registers
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
                            const uint4& q4 = w[2 * jj + (i >> 2)];
                            const uint32_t word = (i & 3) == 0 ? q4.x : (i & 3) == 1 ? q4.y : (i & 3) == 2 ? q4.z : q4.w;
                            uint32_t o[4];
                            if (kFmt == 0)
                                dequant_word(word, s2, o);
                            else
                                dequant_word_fp4(word, s2, o);
                            sts_v4(dst + ((static_cast<uint32_t>(i) ^ swz) << 4), o[0], o[1], o[2], o[3]);
                        }
                        fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bfull(ts));
                    }
                }
                if (!ok) break;
                if (++slot == R) { slot = 0; phase ^= 1; }
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

// Ring depths for a padded M within the shared-memory budget: B slots a
// multiple of the converter groups (four when they fit: measured faster than
// more raw stages), then the most raw stages, then activation slots; each
// ring at least two deep.
void w4_pipeline(int m_pad, int* stages, int* act_slots, int* slots) {
    int best = -1;
    for (int s = 2; s <= kMaxStages; ++s)
        for (int t = kConvGroups; t <= 4; t += kConvGroups)
            for (int a = 2; a <= 3; ++a) {
                if (layout_for(m_pad, s, a, t).alloc > kW4SmemBudget) continue;
                const int score = t * 100 + s * 10 + a;
                if (score > best) {
                    best = score;
                    *stages = s;
                    *slots = t;
                    *act_slots = a;
                }
            }
}

int w4_smem_bytes(int m_pad, int stages, int act_slots, int slots) {
    return layout_for(m_pad, stages, act_slots, slots).alloc;
}

template <int kFmt>
static cudaError_t launch_w4_t(const W4Args& a, const CUtensorMap& tmBq, const CUtensorMap& tmA,
                               const CUtensorMap& tmS, int grid, cudaStream_t stream) {
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(w4_gemm_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_gen[dev] = g_generation;
    }
    w4_gemm_kernel<kFmt><<<grid, kThreads, w4_smem_bytes(a.s.m_pad, a.s.stages, a.a_slots, a.b_slots), stream>>>(
        tmBq, tmA, tmS, a);
    return cudaGetLastError();
}

cudaError_t launch_w4(const W4Args& a, const CUtensorMap& tmBq, const CUtensorMap& tmA, const CUtensorMap& tmS,
                      int grid, cudaStream_t stream) {
    return a.fmt == 1 ? launch_w4_t<1>(a, tmBq, tmA, tmS, grid, stream)
                      : launch_w4_t<0>(a, tmBq, tmA, tmS, grid, stream);
}

}  // namespace tg
