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
// GB300 mapping. One CTA per (batch, head, 128-query block), two CTAs per SM,
// so that one CTA's tensor-core work overlaps the other's softmax.
//   warp 0      TMA producer: Q once (two 64-column boxes), then each block of
//               128 keys: K into its slot as soon as the previous K has been
//               read, V likewise;
//   warp 1      allocates 256 TMEM columns; one thread issues, per key block,
//               S_j = Q K_j^T (M = N = 128, K = d) and, once P_j is written,
//               O += P_j V_j with P_j read from TMEM as the A operand;
//   warps 2-9   softmax, two threads per query row (its TMEM lane), each with
//               half of the keys: read its 64 scores of S_j, the row maximum
//               (halves exchanged through shared memory), the exponentials,
//               P_j (fp16 pairs) written over the scores just read and handed
//               over 32 keys at a time, so the MMA thread starts O += P_j V_j
//               on keys 0-31 and 64-95 while the rest are still exponentiated;
//               each half rescales and finally writes 64 of O's columns.
// The softmax warps sit on the critical path of each key block (scores ->
// P -> second product), and their time is instruction issue rather than the
// exponential unit, so their arithmetic is kept lean: masking only in blocks
// that reach past a row's last visible key, the maximum by three-input max,
// scaling and sums in paired fp32 instructions, and one named barrier per
// block (the maximum exchange, which also carries the abort vote).
// The accumulator is only rescaled when a row's maximum grows by more than
// 2^8 (in the base-2 domain); otherwise the old maximum stays the reference,
// so the exponentials are at most 2^8 and the final O / sum is unchanged.
//
// TMEM columns: S [0, 128) with each half's P over the first 32 of its 64
// score columns (keys 64g.. -> columns 64g..64g+31), O [128, 256).
// S_{j+1} is issued only after O += P_j V_j has completed, since it
// overwrites P_j.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kD = kAttnD;
constexpr int kBM = 128;                       // queries per CTA
constexpr int kBN = 128;                       // keys per block
constexpr int kBoxBytes = 128 * 64 * 2;        // 128 rows x 64 columns fp16
constexpr int kTileBytes = 2 * kBoxBytes;      // 128 rows x 128 columns
constexpr int kSoftmaxWarps = 8;                // two per TMEM lane quarter, each half the keys
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kThreads = (2 + kSoftmaxWarps) * 32;
constexpr int kCtasPerSm = 2;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 0, kColO = 128;
constexpr float kRescaleLog2 = 8.0f;           // lazy rescale threshold (base-2 exponent)
constexpr long long kL2Budget = 64LL << 20;     // K and V bytes of the heads in flight: half of L2
static_assert(kD == 128, "head dimension 128");

// shared memory: Q, K, V, then barriers (about 97 KB: two CTAs fit on an SM)
constexpr int kOffQ = 0;
constexpr int kOffK = kTileBytes;
constexpr int kOffV = 2 * kTileBytes;
constexpr int kOffBar = 3 * kTileBytes;
constexpr int kBarQ = kOffBar;
constexpr int kBarKFull = kBarQ + 8;
constexpr int kBarKEmpty = kBarKFull + 8;
constexpr int kBarVFull = kBarKEmpty + 8;
constexpr int kBarVEmpty = kBarVFull + 8;
constexpr int kBarSFull = kBarVEmpty + 8;
constexpr int kBarPFull = kBarSFull + 8;       // two: P of keys 0-31 and 64-95, then of the rest
constexpr int kBarODone = kBarPFull + 16;
constexpr int kBarDrain = kBarODone + 8;
constexpr int kOffRedMax = kBarDrain + 8;                 // [2 (key-block parity)][2 halves][128 rows] floats
constexpr int kOffRedSum = kOffRedMax + 2 * 2 * 128 * 4;  // [2 halves][128 rows] floats
constexpr int kTmemSlot = kOffRedSum + 2 * 128 * 4;
constexpr int kAbortSlot = kTmemSlot + 4;
constexpr int kMergeSlot = kAbortSlot + 4;     // split blocks: this CTA merges the two parts
constexpr int kSmemUsed = kMergeSlot + 4;
// a split block's part in the scratch: O (128 x 128 fp32, unnormalised), then per row the
// running maximum (base-2 units) and the sum
constexpr int kPartFloats = kBM * kD + 2 * kBM;
constexpr int kSmemAlloc = kSmemUsed + 1024;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnArgs args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // block -> (query block, head, batch). The (batch, head) pairs are taken in groups whose K
    // and V (4 S d bytes each) fit in kL2Budget, so the blocks in flight re-read keys and values
    // from L2; within a group, every head's last query block first, then the one before, ...
    // so with the causal mask the longest CTAs start first (and the shortest fill the tail),
    // and the CTAs in flight spread over many heads rather than queueing on one head's blocks
    // The last n_split query blocks of that order (the last, partial round of the grid) are
    // each split into two CTAs, one per half of the key blocks, whose partial results the
    // second to finish merges: CTA n_plain + 2 p + part is part `part` of block n_plain + p.
    const int n_blocks = args.n_plain + args.n_split;
    const int split_idx = static_cast<int>(blockIdx.x) - args.n_plain;
    const int part = split_idx >= 0 ? (split_idx & 1) : -1;
    const int pair = split_idx >= 0 ? (split_idx >> 1) : 0;
    const int blk = split_idx >= 0 ? args.n_plain + pair : static_cast<int>(blockIdx.x);
    const int n_bh = n_blocks / args.n_qt;
    const long long kv_bytes = 4LL * args.S * kD;
    const int gsz = static_cast<int>(max(1LL, min(static_cast<long long>(n_bh), kL2Budget / kv_bytes)));
    const int per_group = gsz * args.n_qt;
    const int grp = blk / per_group;
    const int first = grp * gsz;
    const int this_gsz = min(gsz, n_bh - first);
    const int local = blk - grp * per_group;
    const int qt = args.n_qt - 1 - local / this_gsz;
    const int bh = first + local % this_gsz;
    const int h = bh % args.H;
    const int b = bh / args.H;
    const int n_kt = (args.S + kBN - 1) / kBN;
    // key blocks j_first..j_last (a split block's halves: [0, n_kt / 2) and [n_kt / 2, n_kt))
    const int j_first = part == 1 ? n_kt / 2 : 0;
    const int j_last = part == 0 ? n_kt / 2 - 1 : (args.causal ? min(qt, n_kt - 1) : n_kt - 1);

    const uint32_t bar_q = sbase + kBarQ, k_full = sbase + kBarKFull, k_empty = sbase + kBarKEmpty;
    const uint32_t v_full = sbase + kBarVFull, v_empty = sbase + kBarVEmpty, s_full = sbase + kBarSFull;
    const uint32_t p_full0 = sbase + kBarPFull, p_full1 = sbase + kBarPFull + 8;
    const uint32_t o_done = sbase + kBarODone, drain_bar = sbase + kBarDrain;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortSlot);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTmemSlot);
    volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + kMergeSlot);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        mbar_init(k_full, 1);
        mbar_init(k_empty, 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full0, kSoftmaxWarps);  // one arrival per softmax warp
        mbar_init(p_full1, kSoftmaxWarps);
        mbar_init(o_done, 1);
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
            int k_issued = 0, v_issued = 0;
            for (int j = j_first; j <= j_last; ++j) {
                const uint32_t ph = static_cast<uint32_t>(j - j_first) & 1u;
                if (!wait_phase_sleep(k_empty, ph ^ 1, wc, kSiteProducerEmpty, 64)) break;
                mbar_arrive_expect_tx(k_full, kTileBytes);
                for (int i = 0; i < 2; ++i)
                    tma_load_4d(sbase + kOffK + i * kBoxBytes, &tmK, k_full, 64 * i, h, j * kBN, b);
                ++k_issued;
                if (!wait_phase_sleep(v_empty, ph ^ 1, wc, kSiteProducerEmpty, 64)) break;
                mbar_arrive_expect_tx(v_full, kTileBytes);
                for (int i = 0; i < 2; ++i)
                    tma_load_4d(sbase + kOffV + i * kBoxBytes, &tmV, v_full, 64 * i, h, j * kBN, b);
                ++v_issued;
            }
            // let every copy in flight land before the CTA exits
            wait_phase_drain(bar_q, 0, wc);
            if (k_issued > 0) wait_phase_drain(k_full, static_cast<uint32_t>(k_issued - 1) & 1u, wc);
            if (v_issued > 0) wait_phase_drain(v_full, static_cast<uint32_t>(v_issued - 1) & 1u, wc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc_s = idesc_f16_f32(kBM, kBN, /*a_mn_major=*/false, /*b_mn_major=*/false);
            const uint32_t idesc_o = idesc_f16_f32(kBM, kD, /*a_mn_major=*/false, /*b_mn_major=*/true);
            bool ok = wait_phase(bar_q, 0, wc, kSiteMmaFull);
            for (int j = j_first; ok && j <= j_last; ++j) {
                const uint32_t ph = static_cast<uint32_t>(j - j_first) & 1u;
                // S_j = Q K_j^T (both operands K-major, d contiguous, two 64-column boxes); it
                // overwrites P_{j-1}, so O += P_{j-1} V_{j-1} must have completed
                if (!wait_phase(k_full, ph, wc, kSiteMmaFull) ||
                    (j > j_first && !wait_phase(o_done, ph ^ 1, wc, kSiteMmaAccEmpty))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(sbase + kOffQ + (kk >> 2) * kBoxBytes, 16, 1024) +
                                       static_cast<uint64_t>(((kk & 3) * 32) >> 4);
                    const uint64_t bd = smem_desc_sw128(sbase + kOffK + (kk >> 2) * kBoxBytes, 16, 1024) +
                                        static_cast<uint64_t>(((kk & 3) * 32) >> 4);
                    mma_f16(tmem_base + kColS, a, bd, idesc_s, kk != 0);
                }
                mma_commit(s_full);
                mma_commit(k_empty);
                // O += P_j V_j: P from TMEM (8 columns per 16 keys), V N-major (d contiguous); the
                // key steps whose P the softmax wrote first (keys 0-31 and 64-95) go first
                if (!wait_phase(p_full0, ph, wc, kSiteMmaFull) || !wait_phase(v_full, ph, wc, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                auto pv_step = [&](int kk) {
                    const uint64_t bd = smem_desc_sw128(sbase + kOffV, kBoxBytes, 1024) +
                                        static_cast<uint64_t>((kk * 2048) >> 4);
                    // keys 64 g .. 64 g + 63 (softmax half g) are P columns 64 g .. 64 g + 31
                    const uint32_t a_col = kColP + (kk >> 2) * 64 + (kk & 3) * 8;
                    mma_f16_tmem_a(tmem_base + kColO, tmem_base + a_col, bd, idesc_o, (j != j_first) || (kk != 0));
                };
                pv_step(0);
                pv_step(1);
                pv_step(4);
                pv_step(5);
                if (!wait_phase(p_full1, ph, wc, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                pv_step(2);
                pv_step(3);
                pv_step(6);
                pv_step(7);
                mma_commit(o_done);
                mma_commit(v_empty);
            }
            mma_commit(drain_bar);
            wait_phase_drain(drain_bar, 0, wc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + output
        // warp w handles the rows of TMEM lane quarter w % 4 and, with half g = (w - 2) / 4,
        // keys 64 g .. 64 g + 63 of each block and O columns 64 g .. 64 g + 63; the two halves
        // of a row exchange their maxima through shared memory every key block (named barrier
        // 1, all softmax warps) and their sums at the end.
        const int quarter = warp & 3;
        const int g = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;  // query row within the block = TMEM lane
        const int q_pos = qt * kBM + row;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t s_cols = kColS + g * 64;  // this half's 64 score columns; its P goes to the first 32
        float* red_max = reinterpret_cast<float*>(smem + kOffRedMax);
        float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
        const float scale = args.scale_log2;
        const int limit = args.causal ? min(args.S, q_pos + 1) : args.S;  // visible keys: < limit
        float m_run = 0.0f, l_run = 0.0f;
        bool ok = true;
        for (int j = j_first; j <= j_last; ++j) {
            const uint32_t ph = static_cast<uint32_t>(j - j_first) & 1u;
            // a wait that gave up still reads the scores (allocated columns: harmless values) and
            // reaches the barrier of the maximum exchange, where every softmax warp learns of it and
            // all stop together, so no named barrier ever waits for a thread that has left
            ok = wait_phase(s_full, ph, wc, kSiteEpilogueAccFull);
            tc_fence_after_sync();
            const int key0 = j * kBN + g * 64;
            const bool masked = key0 + 64 > limit;
            uint32_t r[2][32];
            tmem_ld_32x32b_x32(lane_base + s_cols, r[0]);
            tmem_ld_32x32b_x32(lane_base + s_cols + 32, r[1]);
            tmem_ld_wait();
            if (masked) {  // only blocks that reach past a row's last visible key
#pragma unroll
                for (int hc = 0; hc < 2; ++hc)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + hc * 32 + e >= limit) r[hc][e] = __float_as_uint(-INFINITY);
            }
            auto score = [&](int i) { return __uint_as_float(r[i >> 5][i & 31]); };
            // this half's maximum: four independent chains of three-input maxima
            float acc[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] = score(c);
#pragma unroll
            for (int i = 4; i < 60; i += 8)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c] = fmax3(acc[c], score(i + 2 * c), score(i + 2 * c + 1));
            acc[0] = fmax3(acc[0], score(60), score(61));
            acc[1] = fmax3(acc[1], score(62), score(63));
            float mx = fmaxf(fmax3(acc[0], acc[1], acc[2]), acc[3]);
            // the row maximum over both halves
            red_max[ph * 256 + g * 128 + row] = mx;
            if (named_barrier_or(1, kSoftmaxThreads, !ok)) {
                ok = false;
                break;
            }
            mx = fmaxf(mx, red_max[ph * 256 + (g ^ 1) * 128 + row]);
            const float m_tile = mx * scale;
            float alpha = 1.0f;
            bool rescale = false;
            if (j == j_first) {
                m_run = m_tile;
            } else if (m_tile > m_run + kRescaleLog2) {
                alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
                rescale = true;
            }
            // exponentials in pairs, this half's sum, P (fp16 pairs) over the scores just read,
            // handed to the MMA thread 32 keys at a time
            const float2 scale2 = make_float2(scale, scale);
            const float2 neg_m2 = make_float2(-m_run, -m_run);
            float2 sum2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 x2 = __ffma2_rn(make_float2(score(hc * 32 + 2 * e), score(hc * 32 + 2 * e + 1)),
                                                 scale2, neg_m2);
                    const float2 p2 = make_float2(ex2_approx(x2.x), ex2_approx(x2.y));
                    sum2[e & 1] = __fadd2_rn(sum2[e & 1], p2);
                    pk[e] = pack_half2(p2.x, p2.y);
                }
                tmem_st_32x32b_x16(lane_base + s_cols + hc * 16, pk);
                // this half's O columns *= alpha before the first hand-off: O holds
                // P_{j-1} V_{j-1} (S_j was issued after it completed) and O += P_j V_j starts
                // at the first hand-off; both halves of a row take the same decision
                if (hc == 0 && j > j_first && __any_sync(0xFFFFFFFFu, rescale)) {
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(lane_base + kColO + g * 64 + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st_32x32b_x32(lane_base + kColO + g * 64 + c * 32, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(hc == 0 ? p_full0 : p_full1);
            }
            const float2 s2 = __fadd2_rn(sum2[0], sum2[1]);
            const float sum = s2.x + s2.y;
            l_run = l_run * alpha + sum;
        }
        // O / (sum of both halves), written as fp16 once the last O += P V has landed; a split
        // block's part first publishes its unnormalised O, running maximum and sum
        if (!named_barrier_or(1, kSoftmaxThreads, !ok)) {
            red_sum[g * 128 + row] = l_run;
            const bool done = wait_phase_sleep(o_done, static_cast<uint32_t>(j_last - j_first) & 1u, wc,
                                               kSiteEpilogueAccFull, 64);
            if (!named_barrier_or(1, kSoftmaxThreads, !done)) {
                tc_fence_after_sync();
                const float l_tot = __fadd_rn(l_run, red_sum[(g ^ 1) * 128 + row]);
                __half* dst = args.O + ((static_cast<int64_t>(b) * args.S + q_pos) * args.H + h) * kD + g * 64;
                float inv = 1.0f / l_tot, a_own = 1.0f, a_oth = 0.0f;
                const float* other = nullptr;
                bool store = true;
                if (part >= 0) {
                    // in debug builds a part whose scratch lies outside the buffer writes nothing and
                    // merges nothing (the failed check is reported)
                    const bool ws_ok = dbg_check(dbg_in(static_cast<int64_t>(2 * pair) * kPartFloats, 2 * kPartFloats,
                                                        args.wd.ws_floats) &&
                                                     dbg_in(pair, 1, args.wd.n_counters),
                                                 args.wd);
                    float* mine = args.ws + (ws_ok ? static_cast<int64_t>(2 * pair + part) * kPartFloats : 0);
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(lane_base + kColO + g * 64 + c * 32, o);
                        tmem_ld_wait();
                        if (!ws_ok) continue;
                        float4* w4 = reinterpret_cast<float4*>(mine + row * kD + g * 64 + c * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            __stcg(w4 + q, make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                                       __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3])));
                    }
                    if (g == 0 && ws_ok) {
                        __stcg(mine + kBM * kD + row, m_run);
                        __stcg(mine + kBM * kD + kBM + row, l_tot);
                    }
                    // the second part of the pair to get here merges both
                    __threadfence();
                    named_barrier_sync(1, kSoftmaxThreads);
                    if (threadIdx.x == 64) *merge_flag = ws_ok && atomicAdd(args.counters + pair, 1u) == 1u ? 1 : 0;
                    named_barrier_sync(1, kSoftmaxThreads);
                    store = *merge_flag != 0;
                    if (store) {
                        __threadfence();
                        other = args.ws + static_cast<int64_t>(2 * pair + (part ^ 1)) * kPartFloats;
                        const float m_oth = __ldcg(other + kBM * kD + row);
                        const float l_oth = __ldcg(other + kBM * kD + kBM + row);
                        // symmetric in the two parts (no fused operations), so the result does not
                        // depend on which part finished first
                        const float m_max = fmaxf(m_run, m_oth);
                        a_own = ex2_approx(m_run - m_max);
                        a_oth = ex2_approx(m_oth - m_max);
                        inv = 1.0f / __fadd_rn(__fmul_rn(l_tot, a_own), __fmul_rn(l_oth, a_oth));
                        if (threadIdx.x == 64) atomicExch(args.counters + pair, 0u);
                    }
                }
                if (store) {
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld_32x32b_x32(lane_base + kColO + g * 64 + c * 32, o);
                        tmem_ld_wait();
                        float v[32];
                        if (other != nullptr) {
                            const float4* r4 = reinterpret_cast<const float4*>(other + row * kD + g * 64 + c * 32);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 x = __ldcg(r4 + q);
                                const float xo[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    v[4 * q + e] = __fmul_rn(__fadd_rn(__fmul_rn(__uint_as_float(o[4 * q + e]), a_own),
                                                                       __fmul_rn(xo[e], a_oth)),
                                                             inv);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(o[e]) * inv;
                        }
                        if (q_pos < args.S) {
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                reinterpret_cast<uint4*>(dst + c * 32)[q] =
                                    make_uint4(pack_half2(v[8 * q], v[8 * q + 1]), pack_half2(v[8 * q + 2], v[8 * q + 3]),
                                               pack_half2(v[8 * q + 4], v[8 * q + 5]),
                                               pack_half2(v[8 * q + 6], v[8 * q + 7]));
                        }
                    }
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

int attn_part_floats() { return kPartFloats; }

cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        int grid, cudaStream_t stream) {
    static int attr_gen[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && attr_gen[dev] != g_generation) {
        e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_gen[dev] = g_generation;
    }
    attn_fwd_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(tmQ, tmK, tmV, a);
    return cudaGetLastError();
}

}  // namespace tg
