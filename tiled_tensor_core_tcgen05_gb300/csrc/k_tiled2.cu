// Persistent tiled GEMM C = epi(A @ B + bias) on CTA pairs: each cluster of two
// CTAs (two SMs) computes a 256 x 256 tile of C with the pair form of the
// Blackwell tensor-core MMA.
//
// Same computation as the single-CTA kernel (the tile program of "TileLang:
// writing LLM GPU kernels by thinking in tiles", section 3, with the
// GELU(MatMul + Bias) epilogue of "Designing high-performance GPU kernels with
// TileLang ...", section 3). What the pair buys on GB300: one MMA of
// M=256 x N=256 x K=16 reads A's 256 rows from the two SMs (128 each) and B's
// 256 columns from the two SMs (128 each), so per SM and per MMA the shared
// memory delivers 8 KB instead of the 12 KB a single-CTA 128 x 256 MMA needs,
// and each SM streams half as much of B from L2.
//
// Roles, in both CTAs: warp 0 lane 0 loads this CTA's 128 rows of A and 128
// columns of B for each K block by TMA into its own 6-stage ring; the copies
// of BOTH CTAs complete on the even CTA's "full" barrier (the pair form of the
// TMA copy), which the even CTA arms with the bytes of both halves. Warp 1
// lane 0 of the even CTA issues the pair MMAs; warps 2..5 are the epilogue,
// each CTA reading its own 128 accumulator rows from its own tensor memory (one
// warp per quarter of the rows; with eight epilogue warps, two per quarter, each
// taking half of the columns). A warp reaches only the tensor-memory lanes of its
// scheduler (warp % 4), so the rows of quarter 1 are read on the scheduler that
// also runs the MMA-issuing warp; measured, bias + GELU there slowed the MMA issue
// by ~8%. So with four epilogue warps, warp 5 only moves its chunks from tensor
// memory into a two-slot shared-memory hand-off buffer, and a helper, warp 6
// (scheduler 2), applies bias and GELU and stores them.
// MMA completion is committed to both CTAs at once (multicast), freeing the
// stage in both rings and publishing the accumulator to both epilogues; both
// epilogues release the accumulator to the issuer with one arrive per warp.
#include "tg_device.cuh"
#include "tg_internal.h"

#ifndef TG_PAIR_ACC_BUFS
#define TG_PAIR_ACC_BUFS 2
#endif

namespace tg {
namespace {

constexpr int kHalfM = kBM;                 // 128 rows of A per CTA
constexpr int kHalfN = kBN / 2;             // 128 columns of B per CTA
constexpr int kPairBM = 2 * kHalfM;         // 256 rows of C per cluster tile
constexpr int kPairBN = kBN;                // 256 columns of C per cluster tile
constexpr int kStageA = kHalfM * kBK * 2;   // 16 KB
constexpr int kStageB = kBK * kHalfN * 2;   // 16 KB: two 64x64 N-major boxes
constexpr int kStageBytes = kStageA + kStageB;
#ifndef TG_PAIR_STAGES
#define TG_PAIR_STAGES 6
#endif
constexpr int kPairStages = TG_PAIR_STAGES;
constexpr int kRingBytes = kPairStages * kStageBytes;
constexpr int kBoxB = kBK * 64 * 2;
constexpr int kAccBufs = TG_PAIR_ACC_BUFS;  // accumulators per CTA (256 fp32 columns each)
constexpr int kTmemCols = kAccBufs * kPairBN;
constexpr int kEpiWarp0 = 2;
// hand-off of quarter 1 (the MMA warp's scheduler) to a helper warp; four epilogue warps only
constexpr bool kHandoff = kEpiWarps == 4;
constexpr int kHandQuarter = 1;                    // warp 1 (MMA issue) % 4
constexpr int kHelpWarp = kEpiWarp0 + kEpiWarps;   // warp 6: scheduler 2
constexpr int kHandSlots = 2;
constexpr int kHandSlotBytes = 32 * 32 * 4;        // one 32-row x 32-column fp32 chunk
constexpr int kThreads = (kEpiWarp0 + kEpiWarps + (kHandoff ? 1 : 0)) * 32;

constexpr int kBarFull = kRingBytes;
constexpr int kBarEmpty = kBarFull + 8 * kPairStages;
constexpr int kBarAccFull = kBarEmpty + 8 * kPairStages;
constexpr int kBarAccEmpty = kBarAccFull + 16;
constexpr int kBarDrain = kBarAccEmpty + 16;
constexpr int kTmemSlot = kBarDrain + 8;
constexpr int kAbortSlot = kTmemSlot + 4;
// per-warp output staging: two TMA-store boxes (or one padded st.global chunk)
constexpr int kEpiWarpBytes = 2 * kStoreBoxBytes;
static_assert(kEpiWarpBytes >= kStageWarpBytes, "staging covers both store paths");
constexpr int kBarHandFull = kAbortSlot + 4;
constexpr int kBarHandEmpty = kBarHandFull + 8 * kHandSlots;
static_assert(kBarHandFull % 8 == 0, "mbarriers are 8-byte aligned");
constexpr int kEpiStage = (kBarHandEmpty + 8 * kHandSlots + 1023) / 1024 * 1024;
constexpr int kStoreWarps = kEpiWarps + (kHandoff ? 1 : 0);  // warps that stage and store C
constexpr int kHandBuf = kEpiStage + kStoreWarps * kEpiWarpBytes;
constexpr int kSmemUsed = kHandBuf + (kHandoff ? kHandSlots * kHandSlotBytes : 0);
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 227 * 1024, "one CTA's dynamic shared memory");

// M=256 (pair), N=256, A K-major, B N-major; and the half-width form (N=128)
// used for the split tiles of the last wave.
constexpr uint32_t kIdesc = idesc_f16_f32(kPairBM, kPairBN, /*a_mn_major=*/false, /*b_mn_major=*/true);
constexpr uint32_t kIdescHalf = idesc_f16_f32(kPairBM, kPairBN / 2, /*a_mn_major=*/false, /*b_mn_major=*/true);

// Work unit u -> tile and column range. Units below split_from are whole
// 256x256 tiles; the rest are the two 256x128 halves of the last wave's tiles,
// so that wave takes half as long when it would otherwise leave clusters idle.
struct Unit {
    int tile;
    int col0;   // first column of the unit within the tile (0 or 128)
    int width;  // 256 or 128
};

__device__ __forceinline__ Unit unit_of(int u, int split_from) {
    if (u < split_from) return Unit{u, 0, kPairBN};
    const int j = u - split_from;
    return Unit{split_from + (j >> 1), (j & 1) * (kPairBN / 2), kPairBN / 2};
}

// K order: a CTA's odd work units walk K backwards, so a wave starts on the k-blocks the
// previous wave read last (most likely still in L2)
#ifndef TG_PAIR_KSERP
#define TG_PAIR_KSERP 1
#endif
#ifndef TG_PAIR_SERPENTINE
#define TG_PAIR_SERPENTINE 1
#endif
__device__ __forceinline__ void tile_coords(int tile, int m_blocks, int n_blocks, int group_m, int& mb, int& nb) {
    const int per_group = group_m * n_blocks;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gsize = min(m_blocks - first_m, group_m);
    const int local = tile - g * per_group;
    mb = first_m + local % gsize;
    nb = local / gsize;
    // serpentine: odd groups walk the columns backwards, so a group starts on the B strips the
    // previous group used last
    if (TG_PAIR_SERPENTINE && (g & 1)) nb = n_blocks - 1 - nb;
}

// kTmaStore: C is written by TMA stores from swizzled staging boxes (C 16-byte
// aligned with N % 8 == 0), otherwise by ordinary stores of staged row segments.
template <bool kTmaStore>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tiled_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const TiledArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs; 1: its peer
    const int cluster = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;

    auto full_bar = [&](int s) { return sbase + kBarFull + 8 * s; };
    auto empty_bar = [&](int s) { return sbase + kBarEmpty + 8 * s; };
    auto acc_full_bar = [&](int b) { return sbase + kBarAccFull + 8 * b; };
    auto acc_empty_bar = [&](int b) { return sbase + kBarAccEmpty + 8 * b; };
    const uint32_t drain_bar = sbase + kBarDrain;
    auto hand_full_bar = [&](int h) { return sbase + kBarHandFull + 8 * h; };
    auto hand_empty_bar = [&](int h) { return sbase + kBarHandEmpty + 8 * h; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(full_bar(s), 1);  // even CTA: armed with both halves' bytes
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full_bar(b), 1);
            mbar_init(acc_empty_bar(b), 2 * kEpiWarps);  // one arrive per epilogue warp, both CTAs
        }
        mbar_init(drain_bar, 1);
        for (int h = 0; h < kHandSlots; ++h) {
            mbar_init(hand_full_bar(h), 32);   // every lane of the quarter-1 warp, after its writes
            mbar_init(hand_empty_bar(h), 32);  // every lane of the helper, after its reads
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync();  // barriers of both CTAs initialised before any remote arrive
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wc{abort_flag, args.wd.status, args.wd.limit_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            const uint32_t leader_full0 = mapa_shared(full_bar(0), 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            int it = 0;
            for (int u = cluster; u < args.num_units && ok; u += num_clusters, ++it) {
                const Unit un = unit_of(u, args.split_from);
                int mb, nb;
                tile_coords(un.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
                const bool backwards = TG_PAIR_KSERP && (it & 1);
                const int m0 = mb * kPairBM + rank * kHalfM;
                // this CTA's half of the unit's columns: 128 of a whole tile, 64 of a half tile
                const int n0 = nb * kPairBN + un.col0 + rank * (un.width / 2);
                const bool whole = un.width == kPairBN;
                const uint32_t bytes = kStageA + (whole ? kStageB : kStageB / 2);
                for (int i = 0; i < args.num_kb; ++i) {
                    const int kb = backwards ? args.num_kb - 1 - i : i;
                    if (!wait_phase(empty_bar(stage), phase ^ 1, wc, kSiteProducerEmpty)) { ok = false; break; }
                    // test hook (watchdog tests): the first stage of each cluster's first unit is
                    // never armed or filled, so every bounded wait behind it must expire
                    const bool skip = args.wd.skip_first_arrive && u == cluster && i == 0;
                    if (!skip) {
                        const uint32_t sA = sbase + stage * kStageBytes;
                        const uint32_t sB = sA + kStageA;
                        const uint32_t fb = leader_full0 + 8 * stage;
                        if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * bytes);
                        tma_load_2d_pair(sA, &tmA, fb, kb * kBK, m0);
                        tma_load_2d_pair(sB, &tmB, fb, n0, kb * kBK);
                        if (whole) tma_load_2d_pair(sB + kBoxB, &tmB, fb, n0 + 64, kb * kBK);
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == kPairStages) { stage = 0; phase ^= 1; }
                }
            }
            // Before the CTA can leave: in the even CTA, every armed stage has
            // landed (its barrier counts both halves); in both CTAs, the MMA's last
            // commit to each stage of this ring (which follows the MMA's wait for
            // that stage's copies) has arrived.
            for (int s = 0; s < kPairStages; ++s)
                if (issued_mask & (1u << s)) {
                    if (rank == 0) wait_phase_drain(full_bar(s), (issued_parity >> s) & 1, wc);
                    if (!*abort_flag) wait_phase_drain(empty_bar(s), (issued_parity >> s) & 1, wc);
                }
        }
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            // -------------------------------------------------------- MMA issue (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = cluster; u < args.num_units && ok; u += num_clusters, ++it) {
                const uint32_t idesc = unit_of(u, args.split_from).width == kPairBN ? kIdesc : kIdescHalf;
                const int b = kAccBufs == 2 ? (it & 1) : 0;
                const uint32_t acc_phase = kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
                if (!wait_phase<true>(acc_empty_bar(b), acc_phase ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kPairBN;
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, wc, kSiteMmaFull)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t sA = sbase + stage * kStageBytes;
                    const uint32_t sB = sA + kStageA;
                    const uint64_t a_desc = smem_desc_sw128(sA, 16, 1024);
                    const uint64_t b_desc = smem_desc_sw128(sB, kBoxB, 1024);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_f16_pair(d_tmem, a_desc + (uint64_t)((k * 32) >> 4), b_desc + (uint64_t)((k * 2048) >> 4),
                                     idesc, (kb | k) != 0);
                    mma_commit_pair(empty_bar(stage), 0x3);  // stage free in both CTAs
                    if (++stage == kPairStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit_pair(acc_full_bar(b), 0x3);  // accumulator ready in both CTAs
            }
            // every pair MMA issued here completes before tensor memory is freed
            mma_commit_pair(drain_bar, 0x1);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else if (kHandoff && warp == kHelpWarp) {
        // ------------------------------------------------------------ helper: quarter 1's math
        // Walks the same units and chunks as the quarter-1 warp, taking each chunk from the
        // hand-off buffer instead of tensor memory.
        const int row_in_tile = rank * kHalfM + kHandQuarter * 32 + lane;
        uint8_t* stage = smem + kEpiStage + kEpiWarps * kEpiWarpBytes;
        int nstore = 0, hc = 0;
        bool ok = true;
        for (int u = cluster; u < args.num_units && ok; u += num_clusters) {
            const Unit un = unit_of(u, args.split_from);
            int mb, nb;
            tile_coords(un.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
            const int row = mb * kPairBM + row_in_tile;
            const int n0 = nb * kPairBN + un.col0;
            const int chunks = max(0, min(un.width / 32, (args.N - n0 + 31) / 32));
            for (int c = 0; c < chunks; ++c, ++hc) {
                const int slot = hc % kHandSlots;
                if (!__all_sync(0xFFFFFFFFu,
                                wait_phase(hand_full_bar(slot), (hc / kHandSlots) & 1, wc, kSiteEpilogueAccFull))) {
                    ok = false;
                    break;
                }
                const uint32_t src = sbase + kHandBuf + slot * kHandSlotBytes + lane * 128;
                uint32_t r[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint4 v = lds_v4(src + 16 * (q ^ (lane & 7)));
                    r[4 * q] = v.x, r[4 * q + 1] = v.y, r[4 * q + 2] = v.z, r[4 * q + 3] = v.w;
                }
                mbar_arrive(hand_empty_bar(slot));
                if (kTmaStore) {
                    if (lane == 0 && nstore >= 2) bulk_wait_group_read<1>();
                    __syncwarp();
                    epilogue_chunk_tma(r, smem_u32(stage) + (nstore & 1) * kStoreBoxBytes, &tmC, args.bias,
                                       row - lane, n0 + c * 32, args.N, args.gelu, args.bias_vec, args.wd);
                    ++nstore;
                } else {
                    epilogue_chunk(r, stage, args.C, args.bias, row - lane, n0 + c * 32, args.M, args.N, args.gelu,
                                   args.c_store, args.bias_vec);
                }
            }
        }
        if (kTmaStore && lane == 0) bulk_wait_group_all();  // every store of this warp has completed
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int quarter = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const bool hand_src = kHandoff && quarter == kHandQuarter;  // this warp's math runs on the helper
        const int row_in_tile = rank * kHalfM + quarter * 32 + lane;
        uint8_t* stage = smem + kEpiStage + (warp - kEpiWarp0) * kEpiWarpBytes;
        const uint32_t leader_acc_empty0 = mapa_shared(acc_empty_bar(0), 0);
        int it = 0, nstore = 0, hc = 0;
        bool ok = true;
        for (int u = cluster; u < args.num_units && ok; u += num_clusters, ++it) {
            const Unit un = unit_of(u, args.split_from);
            int mb, nb;
            tile_coords(un.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
            const int b = kAccBufs == 2 ? (it & 1) : 0;
            const uint32_t acc_phase = kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
            if (!wait_phase(acc_full_bar(b), acc_phase, wc, kSiteEpilogueAccFull)) break;
            tc_fence_after_sync();
            const int row = mb * kPairBM + row_in_tile;
            const int n0 = nb * kPairBN + un.col0;
            const int chunks = max(0, min(un.width / 32, (args.N - n0 + 31) / 32));
            constexpr int kChunksPerWarp = (kPairBN / 32) / (kEpiWarps / 4);
            const int c_begin = half * kChunksPerWarp;
            const int c_end = min(c_begin + kChunksPerWarp, chunks);
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kPairBN;
            if (c_begin >= c_end) {  // no columns of this tile for this warp
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(leader_acc_empty0 + 8 * b);
            }
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_ld_wait();
                if (c == c_end - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(leader_acc_empty0 + 8 * b);
                }
                if (hand_src) {
                    // the chunk goes to the helper: row `lane` of the slot, 16-byte units
                    // rotated by lane % 8 (conflict-free for both sides' 16-byte accesses)
                    const int slot = hc % kHandSlots;
                    if (!__all_sync(0xFFFFFFFFu, wait_phase(hand_empty_bar(slot), ((hc / kHandSlots) & 1) ^ 1, wc,
                                                            kSiteEpilogueAccFull))) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + kHandBuf + slot * kHandSlotBytes + lane * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        sts_v4(dst + 16 * (q ^ (lane & 7)), make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]));
                    mbar_arrive(hand_full_bar(slot));
                    ++hc;
                } else if (kTmaStore) {
                    // this warp's two staging boxes alternate: the store issued two chunks ago
                    // must have read its box before the box is written again
                    if (lane == 0 && nstore >= 2) bulk_wait_group_read<1>();
                    __syncwarp();
                    epilogue_chunk_tma(r, smem_u32(stage) + (nstore & 1) * kStoreBoxBytes, &tmC, args.bias,
                                       row - lane, n0 + c * 32, args.N, args.gelu, args.bias_vec, args.wd);
                    ++nstore;
                } else {
                    epilogue_chunk(r, stage, args.C, args.bias, row - lane, n0 + c * 32, args.M, args.N, args.gelu,
                                   args.c_store, args.bias_vec);
                }
            }
        }
        if (kTmaStore && lane == 0) bulk_wait_group_all();  // every store of this warp has completed
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace

int tiled_pair_smem_bytes() { return kSmemAlloc; }

template <bool kTmaStore>
static cudaError_t launch_pair_t(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 const CUtensorMap& tmC, int max_clusters, cudaStream_t stream) {
    static int attr_gen[64] = {};
    static int active_clusters[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(tiled_pair_kernel<kTmaStore>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemAlloc);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * max_clusters);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemAlloc;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, tiled_pair_kernel<kTmaStore>, &cfg);
        if (e != cudaSuccess) return e;
        active_clusters[dev] = n > 0 ? n : 1;
        attr_gen[dev] = g_generation;
    }
    int clusters = dev < 64 ? active_clusters[dev] : 1;
    if (clusters > max_clusters) clusters = max_clusters;
    if (clusters > a.num_tiles) clusters = a.num_tiles;
    if (clusters < 1) clusters = 1;
    TiledArgs args = a;
    // a last wave of R < clusters tiles leaves clusters idle; when the halves
    // of those tiles still fit in one wave (2R <= clusters), run them as halves
    const int full_waves = a.num_tiles / clusters;
    const int rest = a.num_tiles - full_waves * clusters;
    args.split_from = (full_waves > 0 && rest > 0 && 2 * rest <= clusters) ? full_waves * clusters : a.num_tiles;
    args.num_units = args.split_from + 2 * (a.num_tiles - args.split_from);
    tiled_pair_kernel<kTmaStore><<<2 * clusters, kThreads, kSmemAlloc, stream>>>(tmA, tmB, tmC, args);
    return cudaGetLastError();
}

cudaError_t launch_tiled_pair(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap* tmC, int max_clusters, cudaStream_t stream) {
    if (tmC != nullptr) return launch_pair_t<true>(a, tmA, tmB, *tmC, max_clusters, stream);
    return launch_pair_t<false>(a, tmA, tmB, tmA, max_clusters, stream);
}

}  // namespace tg
