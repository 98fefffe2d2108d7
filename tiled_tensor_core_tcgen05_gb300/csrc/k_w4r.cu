// Weight-only 4-bit GEMM for decode-sized M (at most 16 rows of A):
// C = epi(A @ W + bias), W[k][n] = fp16(v(q[k][n]) * scale[k/128][n]), the
// same product as the tensor-memory kernel (k_w4.cu), for the shape where that
// kernel is furthest from the HBM bound.
//
// "TileLang: writing LLM GPU kernels by thinking in tiles" (section
// "Quantized LLM inference") has the packed weights brought on chip, converted
// there and fed to the tensor-core product without an fp16 copy in memory.
// Here the converted tile does not touch shared memory either: each thread
// decodes its own packed words into the fp16 pairs of a warp-level MMA's
// operand registers.
//
// Why warp-level MMAs. A tcgen05 MMA has at least 64 rows and costs at least
// ~93 cycles per instruction; with 16 tokens the tensor-memory kernel pads M
// to 64 and still spends ~29 us on MMA issue for 16 x 28672 x 8192. The
// m16n8k16 MMA takes both operands from registers and issues one per 8 cycles
// per warp; the 7.5 GFLOP of that shape need ~12 us of it, and no converted
// tile is written to or read back from shared memory (the tensor-memory
// kernel's bound: 4 bytes of shared-memory traffic per converted weight).
// Operand roles: the product is computed transposed, C^T = W^T A^T. The MMA's
// 16 rows are 16 weight columns (its A operand, decoded in registers) and its 8
// columns are 8 tokens (its B operand), two MMAs for the 16 tokens. A B
// fragment holds consecutive k pairs of one token, which is what one 16-byte
// shared-memory load of that token's activations delivers, so the loaded
// registers feed the MMA as they are; the opposite roles would interleave two
// tokens' registers in every fragment and cost a register move per pair.
//
// Work. A CTA owns 64 consecutive output columns (two warp-columns of 32) for
// the whole K, so no partial sums leave the CTA. K is streamed in chunks of
// 256 through a ring of shared-memory stages filled by TMA: the chunk's
// activations (16 rows x 256 k, one 3-D box whose lines are (row, 64-k block)
// pairs, so the 128-byte swizzle phase differs between the k blocks the four
// lanes of a quad read: conflict-free), the packed weights of the 64 columns
// (64 rows x 128 bytes, 128-byte swizzle) and their two scale rows.
// Per CTA:
//   warps 0-3  consumers: warp (nw, ks) = (warp % 2, warp / 2) computes
//              warp-column nw over the chunks c with c % 2 == ks; lane
//              (g, t) = (lane / 4, lane % 4) holds weight column 8 i + g of
//              the warp-column's four 8-column tiles i and the k range
//              [64 t, 64 t + 64) of each chunk (two 16-byte words per tile),
//              decodes each 8-weight word into the A registers of two MMAs
//              (tiles 2b and 2b + 1 are the MMA rows g and g + 8 of 16-column
//              block b), and reads tokens g and g + 8 of the same k range
//              from shared memory as the B registers (for INT4 reordered
//              into the decoder's (k, k+4) pairs with byte permutes; FP4
//              pairs are already in order);
//   warp 4     producer: one lane issues the three TMA copies of each chunk.
// The two partial sums of a warp-column (even and odd chunks) are added in
// that order through shared memory; bias, GELU and one rounding to fp16 follow.
// Barriers: full[s] (TMA bytes), empty[s] (the two warps that read stage s,
// after a proxy fence: the next TMA write into the stage is an async-proxy
// write after their generic-proxy reads).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kRTiles = 4;                         // 8-column MMA tiles per warp
constexpr int kRWarpCols = kW4rCols / (8 * kRTiles);  // warp-columns per CTA (2)
constexpr int kRKSplit = 2;                        // warps per warp-column, taking chunks in turn
constexpr int kRConsumers = kRWarpCols * kRKSplit;
constexpr int kRThreads = (kRConsumers + 1) * 32;
constexpr int kRChunk = 256;                       // k per stage
constexpr int kRWRow = kRChunk / 2;                // bytes of one weight row per stage (128)
constexpr int kRXB = kRChunk / 64;                 // 64-k activation blocks per stage
constexpr int kRWords = kRChunk / 32;              // 8-weight words per lane and tile per stage
constexpr int kRGroups = kRChunk / kW4Group;       // scale rows per stage
constexpr int kRXBytes = 16 * kRChunk * 2;         // activations: 16 rows
constexpr int kRWBytes = kW4rCols * kRWRow;        // packed weights
constexpr int kRSBytes = kW4rCols * 2 * kRGroups;  // scale rows
constexpr int kRTx = kRXBytes + kRWBytes + kRSBytes;
constexpr int kRStage = (kRTx + 1023) / 1024 * 1024;
constexpr int kRStages = 4;
constexpr int kRRedBytes = kRWarpCols * (kRKSplit - 1) * 32 * kRTiles * 4 * 4;  // 4 floats per lane and tile
static_assert(kRStages % kRKSplit == 0, "a stage is always read by the same warps");
static_assert(kRWRow == 128, "weight rows of one 128-byte swizzle span");

struct RLayout {
    static constexpr int red = kRStages * kRStage;
    static constexpr int bar_full = red + kRRedBytes;
    static constexpr int bar_empty = bar_full + 8 * kRStages;
    static constexpr int abort_slot = bar_empty + 8 * kRStages;
    static constexpr int used = abort_slot + 16;
    static constexpr int alloc = used + 1024;  // 1 KB alignment slack
};

__device__ __forceinline__ void mma_m16n8k16(float (&c)[4], const uint4& a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

template <int kFmt>
__global__ void __launch_bounds__(kRThreads, 3)
    w4r_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmX, const W4rArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto full = [&](int s) { return sb + RLayout::bar_full + 8 * s; };
    auto empty = [&](int s) { return sb + RLayout::bar_empty + 8 * s; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + RLayout::abort_slot);
    const int n0 = blockIdx.x * kW4rCols;
    const int nch = a.n_chunks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kRWarpCols);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmS);
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();
    const WaitCtx wc{abort_flag, a.wd.status, a.wd.limit_ns};

    if (warp == kRConsumers) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_stream = l2_policy_evict_first();  // weights and scales: read once
            const uint64_t pol_keep = l2_policy_evict_last();     // activations: read by every CTA
            const bool skip_first = a.wd.skip_first_arrive != 0;
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int slot = c % kRStages;
                if (!wait_phase(empty(slot), ((c / kRStages) & 1) ^ 1, wc, kSiteProducerEmpty)) break;
                const uint32_t st = sb + slot * kRStage;
                // test hook (watchdog tests): the first stage is never filled, so its
                // consumers' bounded wait must expire
                if (!(skip_first && c == 0)) {
                    mbar_arrive_expect_tx(full(slot), kRTx);
                    tma_load_3d_hint(st, &tmX, full(slot), 0, c * kRXB, 0, pol_keep);
                    tma_load_2d_hint(st + kRXBytes, &tmW, full(slot), c * kRWRow, n0, pol_stream);
                    tma_load_2d_hint(st + kRXBytes + kRWBytes, &tmS, full(slot), n0, c * kRGroups, pol_stream);
                }
                issued = c + 1;
            }
            // let the copies in flight land before the CTA can exit (consumers that
            // gave up no longer wait for them)
            for (int c = issued - kRStages < 0 ? 0 : issued - kRStages; c < issued; ++c)
                if (!(skip_first && c == 0)) wait_phase_drain(full(c % kRStages), (c / kRStages) & 1, wc);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int nw = warp % kRWarpCols, ks = warp / kRWarpCols;
    float acc[kRTiles][4];
#pragma unroll
    for (int i = 0; i < kRTiles; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    constexpr int kTk = kRChunk / 4;  // k per lane per stage: [kTk t, kTk t + kTk)
    for (int c = ks; c < nch; c += kRKSplit) {
        const int slot = c % kRStages;
        if (!__all_sync(0xFFFFFFFFu, wait_phase(full(slot), (c / kRStages) & 1, wc, kSiteConvFull))) break;
        const uint32_t st = sb + slot * kRStage;
        // this lane's packed words: rows 8 i + g of the warp-column, bytes [kTk t / 2, kTk t / 2 + kTk / 2)
        // of the 128-byte row: 16-byte units 2 t + j, swizzled by row % 8 = g
        uint4 wq[kRTiles][kRWords / 4];
        __half2 sc[kRTiles];
#pragma unroll
        for (int i = 0; i < kRTiles; ++i) {
            const int r = nw * 8 * kRTiles + 8 * i + g;
#pragma unroll
            for (int j = 0; j < kRWords / 4; ++j) {
                wq[i][j] = lds_v4(st + kRXBytes + r * kRWRow + 16 * ((2 * t + j) ^ g));
            }
            // the lane's k range lies in scale group (kTk t) / 128 of the stage
            sc[i] = __half2half2(__ushort_as_half(
                lds_u16(st + kRXBytes + kRWBytes + (kTk * t / kW4Group) * kW4rCols * 2 + 2 * r)));
        }
#pragma unroll
        for (int w = 0; w < kRWords; ++w) {
            // word w: k = kTk t + 8 w .. + 7; activation line (row, 64-k block), unit within the line
            const int k = kTk * t + 8 * w;
            const int l0 = g * kRXB + k / 64, l1 = (g + 8) * kRXB + k / 64, unit = (k % 64) / 8;
            const uint4 u0 = lds_v4(st + l0 * 128 + 16 * (unit ^ (l0 & 7)));
            const uint4 u1 = lds_v4(st + l1 * 128 + 16 * (unit ^ (l1 & 7)));
            // B fragments (token g of each 8-token half h, u0 for rows 0-7 and u1 for rows 8-15):
            // the k pairs of the word's two k16 steps, in the order the decoder delivers the weights
            uint32_t xb[2][4];
            if (kFmt == 0) {  // pairs (k, k+4), (k+1, k+5), ...
                xb[0][0] = __byte_perm(u0.x, u0.z, 0x5410);
                xb[0][1] = __byte_perm(u0.x, u0.z, 0x7632);
                xb[0][2] = __byte_perm(u0.y, u0.w, 0x5410);
                xb[0][3] = __byte_perm(u0.y, u0.w, 0x7632);
                xb[1][0] = __byte_perm(u1.x, u1.z, 0x5410);
                xb[1][1] = __byte_perm(u1.x, u1.z, 0x7632);
                xb[1][2] = __byte_perm(u1.y, u1.w, 0x5410);
                xb[1][3] = __byte_perm(u1.y, u1.w, 0x7632);
            } else {  // natural pairs (k, k+1): the loaded registers as they are
                xb[0][0] = u0.x, xb[0][1] = u0.y, xb[0][2] = u0.z, xb[0][3] = u0.w;
                xb[1][0] = u1.x, xb[1][1] = u1.y, xb[1][2] = u1.z, xb[1][3] = u1.w;
            }
            uint32_t bw[kRTiles][4];
#pragma unroll
            for (int i = 0; i < kRTiles; ++i) {
                const uint4& q = wq[i][w >> 2];
                const uint32_t word = (w & 3) == 0 ? q.x : (w & 3) == 1 ? q.y : (w & 3) == 2 ? q.z : q.w;
                if (kFmt == 0)
                    dequant_word(word, sc[i], bw[i]);
                else
                    dequant_word_fp4(word, sc[i], bw[i]);
            }
            // A fragments: MMA rows g and g + 8 are the weight columns of tiles 2b and 2b + 1
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int b = 0; b < kRTiles / 2; ++b) {
                    const uint4 af = make_uint4(bw[2 * b][2 * s], bw[2 * b + 1][2 * s], bw[2 * b][2 * s + 1],
                                                bw[2 * b + 1][2 * s + 1]);
#pragma unroll
                    for (int h = 0; h < 2; ++h) mma_m16n8k16(acc[2 * b + h], af, xb[h][2 * s], xb[h][2 * s + 1]);
                }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(slot));
    }

    // ---------------------------------------------------------------- epilogue
    // accumulator 2 b + h (16-column block b, token half h): columns 16 b + g and 16 b + 8 + g
    // of the warp-column (MMA rows g, g + 8) x tokens 8 h + 2 t and 8 h + 2 t + 1 (MMA columns)
    float* red = reinterpret_cast<float*>(smem + RLayout::red);
    constexpr int kRedWarp = 32 * kRTiles * 4;  // floats per warp
    if (ks > 0) {
        float* dst = red + ((ks - 1) * kRWarpCols + nw) * kRedWarp;
#pragma unroll
        for (int i = 0; i < kRTiles; ++i)
            *reinterpret_cast<float4*>(dst + (i * 32 + lane) * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    named_barrier_sync(1, kRConsumers * 32);
    if (ks != 0) return;
    for (int q = 1; q < kRKSplit; ++q) {
        const float* src = red + ((q - 1) * kRWarpCols + nw) * kRedWarp;
#pragma unroll
        for (int i = 0; i < kRTiles; ++i) {
            const float4 v = *reinterpret_cast<const float4*>(src + (i * 32 + lane) * 4);
            acc[i][0] += v.x;
            acc[i][1] += v.y;
            acc[i][2] += v.z;
            acc[i][3] += v.w;
        }
    }
#pragma unroll
    for (int b = 0; b < kRTiles / 2; ++b) {
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {  // column g or g + 8 of the 16-column block
            const int col = n0 + nw * 8 * kRTiles + 16 * b + 8 * hi + g;
            if (col >= a.N) continue;
            const float bv = a.bias ? __half2float(a.bias[col]) : 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int row = 8 * h + 2 * t + e;
                    if (row >= a.M) continue;
                    const int64_t off = static_cast<int64_t>(row) * a.N + col;
                    if (!dbg_check(dbg_in(off, 1, static_cast<int64_t>(a.M) * a.N), a.wd)) continue;
                    a.C[off] = __float2half_rn(epi_value(acc[2 * b + h][2 * hi + e], bv, a.gelu));
                }
        }
    }
}

}  // namespace

int w4r_smem_bytes() { return RLayout::alloc; }
int w4r_chunk() { return kRChunk; }

template <int kFmt>
static cudaError_t launch_w4r_t(const W4rArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmS,
                                const CUtensorMap& tmX, int grid, cudaStream_t stream) {
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(w4r_gemm_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, RLayout::alloc);
        if (e != cudaSuccess) return e;
        attr_gen[dev] = g_generation;
    }
    w4r_gemm_kernel<kFmt><<<grid, kRThreads, RLayout::alloc, stream>>>(tmW, tmS, tmX, a);
    return cudaGetLastError();
}

cudaError_t launch_w4r(const W4rArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmS, const CUtensorMap& tmX,
                       int grid, cudaStream_t stream) {
    return a.fmt == 1 ? launch_w4r_t<1>(a, tmW, tmS, tmX, grid, stream)
                      : launch_w4r_t<0>(a, tmW, tmS, tmX, grid, stream);
}

}  // namespace tg
