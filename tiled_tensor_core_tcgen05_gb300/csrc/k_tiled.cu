// Persistent tiled GEMM C = epi(A @ B + bias) on the Blackwell tensor core.
//
// The tile program of "TileLang: writing LLM GPU kernels by thinking in tiles"
// (section 3: a C tile per thread block, A/B tiles staged in shared memory,
// T.gemm on the tiles, a pipelined K loop, the fragment written back) and of
// "TileLang: you write the dataflow, the compiler owns the schedule" (section
// "The tile program"), with the epilogue GELU(MatMul + Bias) applied on chip as
// in "Designing high-performance GPU kernels with TileLang ...", section 3.
//
// GB300 design (not the pages' Ampere/Hopper schedule):
//   * one CTA per SM, persistent over 128 x BN output tiles in grouped order
//     (BN = 256; 128 or 64 when 256-wide tiles would leave most SMs idle);
//   * warp roles: a producer (one TMA-issuing lane, or four warps of ordinary
//     loads when TMA cannot describe the operands), one MMA-issuing lane, and
//     four epilogue warps (one per quarter of the accumulator's rows);
//   * a ~192 KB ring (4 stages of A 128x64 K-major + B 64x256 N-major, or 6 / 8
//     of the narrower stages, all in the 128-byte swizzled layout) guarded by
//     full/empty mbarriers;
//   * tcgen05.mma (M=128, N=BN, K=16) accumulating in tensor memory; two
//     BN-column accumulators so the epilogue of one tile overlaps the
//     mainloop of the next;
//   * the epilogue reads TMEM with tcgen05.ld, adds bias, applies GELU in fp32,
//     rounds once to binary16 and stores with masking for ragged M/N;
//   * when the tiles alone cannot fill the SMs (few rows, long K), K is split:
//     a work unit is one K slice of one tile. Up to 8 slices run as one
//     thread-block cluster (one CTA per slice, one unit each): every CTA stages
//     its fp32 tile in its own shared memory, and after a cluster barrier each
//     sums its share of the tile's rows over all slices (distributed shared
//     memory, slices in order) and applies the epilogue. Otherwise each unit
//     writes its fp32 tile to scratch and the reduction kernel of the skinny
//     path sums the slices in order and applies the epilogue.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kBoxB = kBK * 64 * 2;  // one 64 (k) x 64 (n) box, 8 KB

// Geometry for a tile width BN (256, or 128 / 64 for problems with few tiles):
// a ring of ~192 KB (4, 6 or 8 stages), two BN-column fp32 accumulators in
// TMEM, and the barrier block after the ring: full[S], empty[S], acc_full[2],
// acc_empty[2], drain; then the per-warp output staging.
template <int BN>
struct Geom {
    static constexpr int kStageA = kBM * kBK * 2;  // 16 KB: 128 rows x 128 B
    static constexpr int kStageB = kBK * BN * 2;   // BN / 64 N-major boxes of 8 KB
    static constexpr int kStageBytes = kStageA + kStageB;
    static constexpr int kStagesN = (kStages * (kBM * kBK + kBK * kBN) * 2) / kStageBytes;
    static constexpr int kRingBytes = kStagesN * kStageBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kBarFull = kRingBytes;
    static constexpr int kBarEmpty = kBarFull + 8 * kStagesN;
    static constexpr int kBarAccFull = kBarEmpty + 8 * kStagesN;
    static constexpr int kBarAccEmpty = kBarAccFull + 16;
    static constexpr int kBarDrain = kBarAccEmpty + 16;
    static constexpr int kTmemSlot = kBarDrain + 8;
    static constexpr int kAbortSlot = kTmemSlot + 4;
    static constexpr int kEpiStage = (kAbortSlot + 4 + 127) / 128 * 128;
    static constexpr int kSmemUsed = kEpiStage + kEpiWarps * kStageWarpBytes;
    static constexpr int kSmemAlloc = kSmemUsed + 1024;  // slack to align the ring to 1024 B
    // Operand descriptors: A is K-major (8-row groups 1024 B apart); B is N-major
    // with 64-column atoms 8 KB apart (one TMA box each) and 8-row K groups 1024 B
    // apart. One K=16 step advances A by 32 B within the swizzled row and B by 16
    // rows (2048 B).
    static constexpr uint32_t kIdesc = idesc_f16_f32(kBM, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);
    static_assert(kStagesN >= 4 && kStagesN <= 8, "ring depth");
};

template <bool kTma>
struct Roles {
    static constexpr int kProducerWarps = kTma ? 1 : 4;
    static constexpr int kMmaWarp = kProducerWarps;
    static constexpr int kEpiWarp0 = kProducerWarps + 1;
    static constexpr int kThreads = (kProducerWarps + 1 + kEpiWarps) * 32;
};

// Work unit u: K slice u / num_tiles of tile u % num_tiles (the tiles' first slices first, so
// the CTAs of one wave share the K range of the strips they read), K blocks [kb0, kb1). In a
// cluster launch the CTAs of one cluster are the slices of one tile: slice u % splits.
struct Unit {
    int tile, slice, kb0, kb1;
};
template <bool kCl>
__device__ __forceinline__ Unit unit_of(const TiledArgs& a, int u) {
    Unit w;
    if (kCl) {
        const int t = u / a.splits;
        w.slice = u - t * a.splits;
        w.tile = a.tile0 + t;
    } else {
        w.slice = u / a.num_tiles;
        w.tile = u - w.slice * a.num_tiles;
    }
    w.kb0 = w.slice * a.kb_per_split;
    w.kb1 = min(a.num_kb, w.kb0 + a.kb_per_split);
    return w;
}

__device__ __forceinline__ void tile_coords(int tile, int m_blocks, int n_blocks, int group_m,
                                            int& mb, int& nb) {
    const int per_group = group_m * n_blocks;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gsize = min(m_blocks - first_m, group_m);
    const int local = tile - g * per_group;
    mb = first_m + local % gsize;
    nb = local / gsize;
}

// ---- ordinary-load staging into the same swizzled layout TMA produces ----
//
// 16- and 4-byte units go through cp.async (asynchronous, zero-filled when out
// of range), so a producer thread issues a whole stage and moves on; operands
// aligned to 2 bytes only are copied with ordinary loads and stores.

template <int VEC>
struct VecT;
template <> struct VecT<8> { using T = uint4; };
template <> struct VecT<2> { using T = uint32_t; };
template <> struct VecT<1> { using T = uint16_t; };

template <int VEC>
__device__ __forceinline__ void copy_unit(uint8_t* dst, const __half* src, bool valid, const __half* any_valid) {
    if constexpr (VEC == 8) {
        cp_async_16(smem_u32(dst), valid ? src : any_valid, valid ? 16u : 0u);
    } else if constexpr (VEC == 2) {
        cp_async_4(smem_u32(dst), valid ? src : any_valid, valid ? 4u : 0u);
    } else {
        *reinterpret_cast<uint16_t*>(dst) = valid ? *reinterpret_cast<const uint16_t*>(src) : uint16_t(0);
    }
}

// A tile: rows m0..m0+127, k0..k0+63; byte (r, k) = r*128 + ((k/8) ^ (r%8))*16 + (k%8)*2.
template <int VEC>
__device__ __forceinline__ void stage_A(uint8_t* sA, const __half* __restrict__ A, int M, int K,
                                        int m0, int k0, int ptid) {
    constexpr int kUnitsPerRow = kBK / VEC;
    constexpr int kPerThread = kBM * kUnitsPerRow / 128;
#pragma unroll 8
    for (int i = 0; i < kPerThread; ++i) {
        const int u = ptid + 128 * i;
        const int r = u / kUnitsPerRow;
        const int k = (u % kUnitsPerRow) * VEC;
        const int gm = m0 + r, gk = k0 + k;
        const int off = r * 128 + ((((k * 2) >> 4) ^ (r & 7)) << 4) + ((k * 2) & 15);
        const bool valid = gm < M && gk < K;
        copy_unit<VEC>(sA + off, A + (valid ? static_cast<int64_t>(gm) * K + gk : 0), valid, A);
    }
}

// B tile: k0..k0+63, n0..n0+BN-1; byte (k, n) = (n/64)*8192 + k*128 + (((n%64)/8) ^ (k%8))*16 + (n%8)*2.
template <int BN, int VEC>
__device__ __forceinline__ void stage_B(uint8_t* sB, const __half* __restrict__ B, int N, int K,
                                        int n0, int k0, int ptid) {
    constexpr int kUnitsPerRow = BN / VEC;
    constexpr int kPerThread = kBK * kUnitsPerRow / 128;
#pragma unroll 8
    for (int i = 0; i < kPerThread; ++i) {
        const int u = ptid + 128 * i;
        const int k = u / kUnitsPerRow;
        const int n = (u % kUnitsPerRow) * VEC;
        const int gk = k0 + k, gn = n0 + n;
        const int nn = n & 63;
        const int off = (n >> 6) * kBoxB + k * 128 + ((((nn * 2) >> 4) ^ (k & 7)) << 4) + ((nn * 2) & 15);
        const bool valid = gk < K && gn < N;
        copy_unit<VEC>(sB + off, B + (valid ? static_cast<int64_t>(gk) * N + gn : 0), valid, B);
    }
}

// Cluster split: each CTA's fp32 tile, staged in its ring after its last MMA (row pitch
// padded by 16 bytes).
constexpr int kClPitch = kBN + 4;  // floats
constexpr int kClStageBytes = kBM * kClPitch * 4;

template <bool kTma, int BN, bool kCl>
__global__ void __launch_bounds__(Roles<kTma>::kThreads, 1)
    tiled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const TiledArgs args) {
    static_assert(!kCl || (kTma && BN == kBN && kClStageBytes <= Geom<BN>::kRingBytes),
                  "cluster split: TMA loads, 256-column tiles, the fp32 tile fits in the ring");
    using R = Roles<kTma>;
    using G = Geom<BN>;
    constexpr int kStageA = G::kStageA, kStageBytes = G::kStageBytes, kStagesN = G::kStagesN;
    constexpr int kBN_ = BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto full_bar = [&](int s) { return sbase + G::kBarFull + 8 * s; };
    auto empty_bar = [&](int s) { return sbase + G::kBarEmpty + 8 * s; };
    auto acc_full_bar = [&](int b) { return sbase + G::kBarAccFull + 8 * b; };
    auto acc_empty_bar = [&](int b) { return sbase + G::kBarAccEmpty + 8 * b; };
    const uint32_t drain_bar = sbase + G::kBarDrain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kAbortSlot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesN; ++s) {
            mbar_init(full_bar(s), kTma ? 1 : R::kProducerWarps * 32);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full_bar(b), 1);
            mbar_init(acc_empty_bar(b), kEpiWarps * 32);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (kTma && threadIdx.x == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == R::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), G::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const WaitCtx wc{abort_flag, args.wd.status, args.wd.limit_ns};

    if (warp < R::kProducerWarps) {
        // ------------------------------------------------------------ producer
        if constexpr (kTma) {
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t issued_mask = 0, issued_parity = 0;
                for (int u = blockIdx.x; u < args.num_units; u += gridDim.x) {
                    const Unit w = unit_of<kCl>(args, u);
                    int mb, nb;
                    tile_coords(w.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
                    bool ok = true;
                    for (int kb = w.kb0; kb < w.kb1; ++kb) {
                        if (!wait_phase(empty_bar(stage), phase ^ 1, wc, kSiteProducerEmpty)) { ok = false; break; }
                        const bool skip = args.wd.skip_first_arrive && u == (int)blockIdx.x && kb == w.kb0;
                        if (!skip) {
                            const uint32_t sA = sbase + stage * kStageBytes;
                            const uint32_t sB = sA + kStageA;
                            mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
                            tma_load_2d(sA, &tmA, full_bar(stage), kb * kBK, mb * kBM);
#pragma unroll
                            for (int j = 0; j < kBN_ / 64; ++j)
                                tma_load_2d(sB + j * kBoxB, &tmB, full_bar(stage), nb * kBN_ + j * 64, kb * kBK);
                            issued_mask |= 1u << stage;
                            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        }
                        if (++stage == kStagesN) { stage = 0; phase ^= 1; }
                    }
                    if (!ok) break;
                }
                // let every copy this thread started land before the CTA can exit
                for (int s = 0; s < kStagesN; ++s)
                    if (issued_mask & (1u << s)) wait_phase_drain(full_bar(s), (issued_parity >> s) & 1, wc);
            }
        } else {
            const int ptid = threadIdx.x;  // 0..127
            int stage = 0;
            uint32_t phase = 0;
            for (int u = blockIdx.x; u < args.num_units; u += gridDim.x) {
                const Unit w = unit_of<kCl>(args, u);
                int mb, nb;
                tile_coords(w.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
                bool ok = true;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1, wc, kSiteProducerEmpty)) { ok = false; break; }
                    uint8_t* sA = smem + stage * kStageBytes;
                    uint8_t* sB = sA + kStageA;
                    const int m0 = mb * kBM, n0 = nb * kBN_, k0 = kb * kBK;
                    if (args.a_vec == 8) stage_A<8>(sA, args.A, args.M, args.K, m0, k0, ptid);
                    else if (args.a_vec == 2) stage_A<2>(sA, args.A, args.M, args.K, m0, k0, ptid);
                    else stage_A<1>(sA, args.A, args.M, args.K, m0, k0, ptid);
                    if (args.b_vec == 8) stage_B<BN, 8>(sB, args.B, args.N, args.K, n0, k0, ptid);
                    else if (args.b_vec == 2) stage_B<BN, 2>(sB, args.B, args.N, args.K, n0, k0, ptid);
                    else stage_B<BN, 1>(sB, args.B, args.N, args.K, n0, k0, ptid);
                    fence_proxy_async_smem();      // this thread's ordinary stores, if any
                    cp_async_arrive(full_bar(stage));  // fires once its cp.async copies land
                    if (++stage == kStagesN) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
            }
            cp_async_wait_all();  // nothing of this thread is in flight when the CTA leaves
        }
    } else if (warp == R::kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x, ++it) {
                const Unit w = unit_of<kCl>(args, u);
                const int b = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_phase(acc_empty_bar(b), acc_phase ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kBN_;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, wc, kSiteMmaFull)) { ok = false; break; }
                    tc_fence_after_sync();
                    // stages filled by cp.async / ordinary stores (generic proxy) are read
                    // by the tensor core (async proxy)
                    if constexpr (!kTma) fence_proxy_async_smem();
                    const uint32_t sA = sbase + stage * kStageBytes;
                    const uint32_t sB = sA + kStageA;
                    const uint64_t a_desc = smem_desc_sw128(sA, 16, 1024);
                    const uint64_t b_desc = smem_desc_sw128(sB, kBoxB, 1024);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        mma_f16(d_tmem, a_desc + (uint64_t)((k * 32) >> 4), b_desc + (uint64_t)((k * 2048) >> 4),
                                G::kIdesc, kb != w.kb0 || k != 0);
                    mma_commit(empty_bar(stage));  // frees the stage once these MMAs finish
                    if (++stage == kStagesN) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(acc_full_bar(b));  // accumulator b is complete
            }
            // all MMAs issued by this thread complete before TMEM is released
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
        const int half = (warp - R::kEpiWarp0) >> 2;  // which half of the 32-column chunks
        const int row_in_tile = quarter * 32 + lane;
        uint8_t* stage = smem + G::kEpiStage + (warp - R::kEpiWarp0) * kStageWarpBytes;
        int it = 0;
        for (int u = blockIdx.x; u < args.num_units; u += gridDim.x, ++it) {
            const Unit w = unit_of<kCl>(args, u);
            int mb, nb;
            tile_coords(w.tile, args.m_blocks, args.n_blocks, args.group_m, mb, nb);
            const int b = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            if (!wait_phase(acc_full_bar(b), acc_phase, wc, kSiteEpilogueAccFull)) break;
            tc_fence_after_sync();
            const int row = mb * kBM + row_in_tile;
            const int n0 = nb * kBN_;
            const int chunks = min(kBN_ / 32, (args.N - n0 + 31) / 32);
            constexpr int kChunksPerWarp = (kBN_ / 32) / (kEpiWarps / 4);
            const int c_begin = half * kChunksPerWarp;
            const int c_end = min(c_begin + kChunksPerWarp, chunks);
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * kBN_;
            if (c_begin >= c_end) {  // no columns of this tile for this warp
                tc_fence_before_sync();
                mbar_arrive(acc_empty_bar(b));
            }
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t r[32];
                __syncwarp();  // tcgen05.ld is warp-collective; lanes diverged on the row mask
                tmem_ld_32x32b_x32(taddr + c * 32, r);
                tmem_ld_wait();
                if (c == c_end - 1) {
                    tc_fence_before_sync();
                    mbar_arrive(acc_empty_bar(b));  // this warp is done with TMEM buffer b
                }
                if (args.splits == 1) {
                    epilogue_chunk(r, stage, args.C, args.bias, row - lane, n0 + c * 32, args.M, args.N, args.gelu,
                                   args.c_store, args.bias_vec);
                } else if (kCl) {
                    // the ring is idle once the accumulator is complete: stage this slice's tile
                    const uint32_t dst = sbase + static_cast<uint32_t>((row_in_tile * kClPitch + c * 32) * 4);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        sts_v4(dst + 16 * q, make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]));
                } else if (row < args.m_pad) {
                    // fp32 partials [slice][n][m_pad]: the warp's lanes are 32 consecutive rows,
                    // so each column's values are one 128-byte store
                    const int nc = n0 + c * 32;
                    const int cols = min(32, args.N - nc);
                    const int64_t off = (static_cast<int64_t>(w.slice) * args.N + nc) * args.m_pad + row;
                    if (dbg_check(dbg_in(off, static_cast<int64_t>(cols - 1) * args.m_pad + 1, args.wd.ws_floats),
                                  args.wd)) {
                        float* dst = args.ws + off;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < cols) dst[static_cast<int64_t>(j) * args.m_pad] = __uint_as_float(r[j]);
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kCl) {
        // every CTA of the cluster has staged its slice (each runs exactly one unit, and every
        // thread reaches both cluster barriers, whether or not a wait gave up)
        cluster_sync();
        const int s = args.splits;
        int tmb, tnb;
        const Unit w = unit_of<kCl>(args, blockIdx.x);
        tile_coords(w.tile, args.m_blocks, args.n_blocks, args.group_m, tmb, tnb);
        // this CTA's share of the tile's rows, summed over the slices in order 0, 1, ...
        const int rows_per = (kBM + s - 1) / s;
        const int r_begin = w.slice * rows_per;
        const int r_end = min(kBM, r_begin + rows_per);
        const int m_tile = tmb * kBM, n_tile = tnb * kBN;
        constexpr int kWarps = R::kThreads / 32;
        for (int rr = r_begin + warp; rr < r_end; rr += kWarps) {
            const int m = m_tile + rr;
            if (m >= args.M) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int col = h * (kBN / 2) + lane * 4;
                const int n = n_tile + col;
                if (n >= args.N) continue;  // N % 8 == 0: four columns are all in or all out
                const uint32_t off = sbase + static_cast<uint32_t>((rr * kClPitch + col) * 4);
                float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                for (int q = 0; q < s; ++q) {
                    const float4 p = ld_cluster_f4(mapa_shared(off, q));
                    acc.x += p.x;
                    acc.y += p.y;
                    acc.z += p.z;
                    acc.w += p.w;
                }
                float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (args.bias != nullptr)
#pragma unroll
                    for (int j = 0; j < 4; ++j) b[j] = __half2float(args.bias[n + j]);
                const __half2 lo = __halves2half2(__float2half_rn(epi_value(acc.x, b[0], args.gelu)),
                                                  __float2half_rn(epi_value(acc.y, b[1], args.gelu)));
                const __half2 hi = __halves2half2(__float2half_rn(epi_value(acc.z, b[2], args.gelu)),
                                                  __float2half_rn(epi_value(acc.w, b[3], args.gelu)));
                __half* dst = args.C + static_cast<int64_t>(m) * args.N + n;
                if (args.c_store == 2) {
                    uint2 v;
                    v.x = *reinterpret_cast<const uint32_t*>(&lo);
                    v.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(dst) = v;
                } else {
                    dst[0] = __low2half(lo);
                    dst[1] = __high2half(lo);
                    dst[2] = __low2half(hi);
                    dst[3] = __high2half(hi);
                }
            }
        }
        cluster_sync();  // no CTA leaves while another may still read its shared memory
    }
    if (warp == R::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, G::kTmemCols);
    }
}

template <bool kTma, int BN, bool kCl = false>
cudaError_t launch(const TiledArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB, int grid,
                   cudaStream_t stream) {
    using R = Roles<kTma>;
    constexpr int kSmem = Geom<BN>::kSmemAlloc;
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(tiled_gemm_kernel<kTma, BN, kCl>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        attr_gen[dev] = g_generation;
    }
    CUtensorMap dummy{};
    if constexpr (kCl) {
        // one cluster of `splits` CTAs per tile, one unit per CTA
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.num_units);
        cfg.blockDim = dim3(R::kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = a.splits;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        (void)grid;
        return cudaLaunchKernelEx(&cfg, tiled_gemm_kernel<kTma, BN, kCl>, tmA ? *tmA : dummy, tmB ? *tmB : dummy, a);
    } else {
        tiled_gemm_kernel<kTma, BN, kCl><<<grid, R::kThreads, kSmem, stream>>>(tmA ? *tmA : dummy, tmB ? *tmB : dummy,
                                                                              a);
        return cudaGetLastError();
    }
}

template <bool kTma>
cudaError_t launch_bn(const TiledArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB, int grid,
                      cudaStream_t stream) {
    if (a.bn == 64) return launch<kTma, 64>(a, tmA, tmB, grid, stream);
    if (a.bn == 128) return launch<kTma, 128>(a, tmA, tmB, grid, stream);
    return launch<kTma, 256>(a, tmA, tmB, grid, stream);
}

}  // namespace

int tiled_smem_bytes(bool) { return Geom<kBN>::kSmemAlloc; }
int tiled_threads(bool tma) { return tma ? Roles<true>::kThreads : Roles<false>::kThreads; }

cudaError_t launch_tiled_tma(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                             cudaStream_t stream) {
    return launch_bn<true>(a, &tmA, &tmB, grid, stream);
}

int tiled_cluster_capacity(int splits) {
    if (splits < 2 || splits > kTiledClusterMax) return 0;
    static int gen[64] = {};
    static int cap[64][kTiledClusterMax + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return 0;
    if (gen[dev] != g_generation) {
        using R = Roles<true>;
        constexpr int kSmem = Geom<kBN>::kSmemAlloc;
        auto kern = tiled_gemm_kernel<true, kBN, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) return 0;
        for (int c = 2; c <= kTiledClusterMax; ++c) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(c * 64);
            cfg.blockDim = dim3(R::kThreads);
            cfg.dynamicSmemBytes = kSmem;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = c;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
            cap[dev][c] = n;
        }
        gen[dev] = g_generation;
    }
    return cap[dev][splits];
}

cudaError_t launch_tiled_cluster(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 cudaStream_t stream) {
    if (a.bn != kBN || a.splits < 2 || a.splits > kTiledClusterMax) return cudaErrorInvalidValue;
    return launch<true, kBN, true>(a, &tmA, &tmB, a.num_units, stream);
}

cudaError_t launch_tiled_lsu(const TiledArgs& a, int grid, cudaStream_t stream) {
    return launch_bn<false>(a, nullptr, nullptr, grid, stream);
}

}  // namespace tg
