// Skinny-M GEMM (M <= 128, e.g. decode with a handful of tokens): swap the
// operands and split K.
//
// With M small, C = A @ B is bound by reading B once from HBM. The kernel
// computes the transposed product C^T = B^T @ A^T so that N fills the
// 128-row side of the tensor-core MMA and M (padded to 16) is the MMA's N:
//   MMA operand "A" = a 128 (n) x 64 (k) slice of B, which is N-major in memory;
//   MMA operand "B" = a 64 (k) x M slice of A^T, i.e. A's rows, K-major.
// One work unit is (256-column slice of N, range of K blocks): two such MMAs
// per K step, into two TMEM accumulators, so each stage streams 512 contiguous
// bytes of every B row it touches. Units are spread over a persistent grid,
// slice-major, so CTAs running side by side read neighbouring columns of the
// same rows of B. With more than one K slice, each unit
// writes an fp32 partial tile to a scratch buffer, and a second kernel
// (splitk_reduce_kernel, below) adds the partials in slice order 0, 1, ...
// over the whole GPU, applies bias and GELU and writes C, so results do not
// depend on which CTA finishes first.
//
// The product and epilogue are those of "TileLang: writing LLM GPU kernels by
// thinking in tiles" (sections 2-3) and "Designing high-performance GPU
// kernels with TileLang ..." (section 3, GELU(MatMul + Bias)); the pages give
// no skinny-shape schedule, this one is designed for GB300's HBM.
#include "tg_device.cuh"
#include "tg_internal.h"
#include "tg_skinny.cuh"

#include <map>
#include <mutex>
#include <tuple>

namespace tg {
namespace {

constexpr int kBoxB = kSkBK * 64 * 2;          // 64 (k) x 64 (n) N-major box, 8 KB
constexpr int kHalfBytes = 2 * kBoxB;          // one 128-column MMA half
constexpr int kStageBBytes = kSkHalves * kHalfBytes;
constexpr int kThreads = 6 * 32;            // producer, MMA, 4 epilogue warps

struct Layout {
    int stage_bytes, ring, bar_full, bar_empty, bar_acc_full, bar_acc_empty, bar_drain, tmem_slot,
        abort_slot, used, alloc;
};

__host__ __device__ inline Layout layout_for(int m_pad, int stages) {
    Layout L;
    L.stage_bytes = kStageBBytes + m_pad * 128;  // multiple of 2048: keeps 1024-B alignment
    L.ring = stages * L.stage_bytes;
    L.bar_full = L.ring;
    L.bar_empty = L.bar_full + 8 * stages;
    L.bar_acc_full = L.bar_empty + 8 * stages;
    L.bar_acc_empty = L.bar_acc_full + 16;
    L.bar_drain = L.bar_acc_empty + 16;
    L.tmem_slot = L.bar_drain + 8;
    L.abort_slot = L.tmem_slot + 4;
    L.used = L.abort_slot + 4;
    L.alloc = L.used + 1024;
    return L;
}

// kCl: the K slices of one unit run as one thread-block cluster (one unit per CTA) and are
// summed across the cluster's shared memory after the product; otherwise partials go to
// scratch for splitk_reduce_kernel.
template <bool kCl>
__global__ void __launch_bounds__(kThreads, 1)
    splitk_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmA,
                       const SplitArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const Layout L = layout_for(args.m_pad, args.stages);
    const int S = args.stages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto full_bar = [&](int s) { return sbase + L.bar_full + 8 * s; };
    auto empty_bar = [&](int s) { return sbase + L.bar_empty + 8 * s; };
    auto acc_full_bar = [&](int b) { return sbase + L.bar_acc_full + 8 * b; };
    auto acc_empty_bar = [&](int b) { return sbase + L.bar_acc_empty + 8 * b; };
    const uint32_t drain_bar = sbase + L.bar_drain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.abort_slot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.tmem_slot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full_bar(b), 1);
            mbar_init(acc_empty_bar(b), kSkEpiThreads);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmA);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), args.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wc{abort_flag, args.wd.status, args.wd.limit_ns};
    const int stage_tx = L.stage_bytes;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();  // B: read exactly once
            const uint64_t pol_keep = l2_policy_evict_last();     // A: re-read by every unit
            int stage = 0;
            uint32_t phase = 0;
            uint64_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int sp = kCl ? u % args.splits : u / args.n_tiles;
                const int nt = kCl ? u / args.splits : u - sp * args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1, wc, kSiteProducerEmpty)) { ok = false; break; }
                    const uint32_t sB = sbase + stage * L.stage_bytes;
                    const uint32_t sA = sB + kStageBBytes;
                    mbar_arrive_expect_tx(full_bar(stage), stage_tx);
#pragma unroll
                    for (int j = 0; j < kStageBBytes / kBoxB; ++j)
                        tma_load_2d_hint(sB + j * kBoxB, &tmB, full_bar(stage), nt * kSkBN + j * 64, kb * kSkBK,
                                         pol_stream);
                    tma_load_2d_hint(sA, &tmA, full_bar(stage), kb * kSkBK, 0, pol_keep);
                    issued_mask |= 1ull << stage;
                    issued_parity = (issued_parity & ~(1ull << stage)) | (uint64_t(phase) << stage);
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < S; ++s)
                if (issued_mask & (1ull << s)) wait_phase_drain(full_bar(s), (issued_parity >> s) & 1, wc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, args.m_pad, /*a_mn_major=*/true, /*b_mn_major=*/false);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x, ++it) {
                const int sp = kCl ? u % args.splits : u / args.n_tiles;
                const int kb0 = sp * args.kb_per_split;
                const int kb1 = min(args.kb_total, kb0 + args.kb_per_split);
                const int b = it & 1;
                if (!wait_phase(acc_empty_bar(b), ((it >> 1) & 1) ^ 1, wc, kSiteMmaAccEmpty)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * kSkHalves * args.tmem_stride;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, wc, kSiteMmaFull)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t sB = sbase + stage * L.stage_bytes;
                    const uint32_t sA = sB + kStageBBytes;
                    const uint64_t b_desc = smem_desc_sw128(sA, 16, 1024);  // K-major rows of A
#pragma unroll
                    for (int h = 0; h < kSkHalves; ++h) {
                        const uint64_t a_desc = smem_desc_sw128(sB + h * kHalfBytes, kBoxB, 1024);  // N-major B
#pragma unroll
                        for (int k = 0; k < kSkBK / 16; ++k)
                            mma_f16(d_tmem + h * args.tmem_stride, a_desc + (uint64_t)((k * 2048) >> 4),
                                    b_desc + (uint64_t)((k * 32) >> 4), idesc, (kb != kb0) || (k != 0));
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(acc_full_bar(b));
            }
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        skinny_epilogue<kSkHalves, kCl>(args, tmem_base, acc_full_bar(0), acc_empty_bar(0), wc, sbase);
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (kCl) {
        // every CTA of the cluster has staged its slice (one unit each; every thread reaches both
        // cluster barriers, whether or not a wait gave up). The unit's m_pad x 256 outputs, as
        // 4-column groups, are shared out over the cluster's CTAs; each group's slices are added
        // in order 0, 1, ... (the order of the reduction kernel, so the same bits).
        cluster_sync();
        const int s = args.splits;
        const int sp = blockIdx.x % s;
        const int n_unit = (blockIdx.x / s) * kSkBN;
        const int groups = args.M * (kSkBN / 4);
        const int per = (groups + s - 1) / s;
        const int g1 = min(groups, (sp + 1) * per);
        for (int g = sp * per + static_cast<int>(threadIdx.x); g < g1; g += kThreads) {
            const int m = g / (kSkBN / 4);
            const int col = (g - m * (kSkBN / 4)) * 4;
            const int n = n_unit + col;
            if (n >= args.N) continue;  // N % 8 == 0: four columns are all in or all out
            const uint32_t off = sbase + static_cast<uint32_t>((m * kSkClPitch + col) * 4);
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int q = 0; q < s; ++q) {
                const float4 p = ld_cluster_f4(mapa_shared(off, q));
                acc.x += p.x;
                acc.y += p.y;
                acc.z += p.z;
                acc.w += p.w;
            }
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
            __half* dst = args.C + static_cast<int64_t>(m) * args.N + n;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = __float2half_rn(epi_value(v[j], args.bias != nullptr ? __half2float(args.bias[n + j]) : 0.0f,
                                                   args.gelu));
        }
        cluster_sync();  // no CTA leaves while another may still read its shared memory
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, args.tmem_cols);
    }
}

}  // namespace

int split_stage_bytes(int m_pad) { return layout_for(m_pad, 1).stage_bytes; }

int split_stages_for(int m_pad) {
    int s = kSkSmemBudget / split_stage_bytes(m_pad);
    if (s > 16) s = 16;
    if (s < 2) s = 2;
    return s;
}

int split_smem_bytes(int m_pad, int stages) { return layout_for(m_pad, stages).alloc; }

bool split_on_chip_fits(int m_pad, int stages) {
    return layout_for(m_pad, stages).ring >= m_pad * kSkClPitch * 4;
}

namespace {

// The K slices' fp32 partials [slice][n][m] summed over the whole GPU: thread = one column n
// and 16 rows m0..m0+15, slices added in order 0, 1, ... starting from 0 (a fixed order, so
// the results do not depend on which CTA finished first), then bias, GELU and one rounding. The loads of four slices are issued before they are
// added. A warp's stores of one row are 32 consecutive columns.
constexpr int kRedThreads = 128;

__global__ void __launch_bounds__(kRedThreads) splitk_reduce_kernel(const SplitArgs a) {
    const int n = blockIdx.x * kRedThreads + threadIdx.x;
    const int m0 = blockIdx.y * 16;
    if (n >= a.N) return;
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
    constexpr int kBatch = 4;
    int q = 0;
    for (; q + kBatch <= a.splits; q += kBatch) {
        float4 p[kBatch][4];
        bool in[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const int64_t off = (static_cast<int64_t>(q + j) * a.N + n) * a.m_pad + m0;
            in[j] = dbg_check(dbg_in(off, 16, a.wd.ws_floats), a.wd);
            const float4* wq = reinterpret_cast<const float4*>(a.ws + (in[j] ? off : 0));
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) p[j][v4] = __ldcg(wq + v4);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (in[j]) add_slice(p[j]);
    }
    for (; q < a.splits; ++q) {
        const int64_t off = (static_cast<int64_t>(q) * a.N + n) * a.m_pad + m0;
        if (!dbg_check(dbg_in(off, 16, a.wd.ws_floats), a.wd)) continue;
        const float4* wq = reinterpret_cast<const float4*>(a.ws + off);
        float4 p[4];
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) p[v4] = __ldcg(wq + v4);
        add_slice(p);
    }
    const float bias_n = a.bias != nullptr ? __half2float(a.bias[n]) : 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (m0 + i < a.M) a.C[static_cast<int64_t>(m0 + i) * a.N + n] = __float2half_rn(epi_value(s[i], bias_n, a.gelu));
}

}  // namespace

cudaError_t launch_splitk_reduce(const SplitArgs& a, cudaStream_t stream) {
    const dim3 grid((a.N + kRedThreads - 1) / kRedThreads, (a.M + 15) / 16);
    splitk_reduce_kernel<<<grid, kRedThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_splitk(const SplitArgs& a, const CUtensorMap& tmB, const CUtensorMap& tmA, int grid,
                          cudaStream_t stream) {
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        for (auto kern : {splitk_gemm_kernel<false>, splitk_gemm_kernel<true>})
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024)) != cudaSuccess)
                return e;
        attr_gen[dev] = g_generation;
    }
    const int smem = split_smem_bytes(a.m_pad, a.stages);
    splitk_gemm_kernel<false><<<grid, kThreads, smem, stream>>>(tmB, tmA, a);
    return cudaGetLastError();
}

int split_cluster_capacity(int splits, int m_pad, int stages) {
    if (splits < 2 || splits > kTiledClusterMax) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const int smem = split_smem_bytes(m_pad, stages);
    // cached by (device, generation, cluster size, shared memory)
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int>, int> cache;
    const auto key = std::make_tuple(dev, g_generation, splits, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaFuncSetAttribute(splitk_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(splits * 64);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = splits;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, splitk_gemm_kernel<true>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    } else {
        cudaGetLastError();
    }
    cache[key] = n;
    return n;
}

cudaError_t launch_splitk_cluster(const SplitArgs& a, const CUtensorMap& tmB, const CUtensorMap& tmA,
                                  cudaStream_t stream) {
    if (a.splits < 2 || a.splits > kTiledClusterMax || !split_on_chip_fits(a.m_pad, a.stages))
        return cudaErrorInvalidValue;
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        if ((e = cudaFuncSetAttribute(splitk_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      227 * 1024)) != cudaSuccess)
            return e;
        attr_gen[dev] = g_generation;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.num_units);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = split_smem_bytes(a.m_pad, a.stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = a.splits;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_gemm_kernel<true>, tmB, tmA, a);
}

}  // namespace tg
