// Internal interface between the C-ABI front end (tg_api.cu) and the kernel
// translation units. Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace tg {

// ---- tiled kernel geometry: one CTA computes a 128 x 256 tile of C, walking K
// in 64-wide blocks through a 4-deep ring of shared-memory stages.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
// Rasterisation: tiles are visited in groups of G tile rows (all columns of a
// group before the next), so the A strips of one group are re-read from L2
// while B streams past. G is sized so that those strips (G x tile rows x K x 2
// bytes) take about kGroupBytes: measured on GB300 for 8192^3, groups of
// 8 x 256 rows (32 MB) read 1.06 GB from HBM per launch, 16 rows 1.25 GB and
// 32 rows 2.09 GB.
#ifndef TG_GROUP_MB
#define TG_GROUP_MB 32
#endif
constexpr int64_t kGroupBytes = static_cast<int64_t>(TG_GROUP_MB) << 20;
// Epilogue warps of the tiled kernels: one per TMEM lane quarter (4), or two
// per quarter each taking half of a tile's 32-column chunks (8). Measured on
// GB300, 4 is as fast as 8 with erf-GELU and slightly faster without it.
#ifndef TG_EPI_WARPS
#define TG_EPI_WARPS 4
#endif
constexpr int kEpiWarps = TG_EPI_WARPS;
static_assert(kEpiWarps == 4 || kEpiWarps == 8, "epilogue warps: one or two per TMEM lane quarter");

// ---- split-K (swap-AB) kernel geometry: one work unit is a 256-column slice of
// N (two 128-row MMA halves) times a range of 64-wide K blocks; M (<= 128) is
// the MMA's N, padded to 16.
constexpr int kSkHalves = 2;
constexpr int kSkBN = 128 * kSkHalves;
constexpr int kSkBK = 64;
constexpr int kSkMaxM = 128;
constexpr int kSkMaxSplits = 64;
constexpr int kSkSmemBudget = 200 * 1024;  // operand ring budget per CTA

// ---- weight-only 4-bit kernel geometry: one work unit is a 256-column slice
// of N (the MMA's N) times a range of 256-wide K blocks; tokens are the MMA's
// M (64 rows, at most 64 real ones per launch). A stage holds the slice's
// packed weights (256 rows of 128 bytes), the matching 256 columns of A and
// the two scale rows of the block.
constexpr int kW4BN = 256;
constexpr int kW4BK = 256;
constexpr int kW4Group = 128;          // rows of K sharing one scale per column
constexpr int kW4MaxM = 64;            // rows of A per launch
constexpr int kW4SmemBudget = 224 * 1024;
constexpr int kW4rCols = 64;           // register-dequant 4-bit kernel: output columns per CTA
constexpr int kW4rMaxM = 16;           // and rows of A (its MMA's M)

// Debug builds (compiled with TG_DEBUG=1) check, on the device, that every
// scratch, counter and output index a kernel computes lies inside its buffer,
// record a failure in the status word (kSiteBounds) and skip the access; in
// normal builds the checks compile away.
#ifndef TG_DEBUG
#define TG_DEBUG 0
#endif

// Watchdog plumbing handed to every kernel: where to record the first wait that
// expired, the limit, and the test hook that withholds one producer arrival;
// plus the buffer sizes the debug builds' bounds checks compare against.
struct Watchdog {
    int* status;          // device word; 0 = ok, else the code of the expired wait or failed check
    uint64_t limit_ns;
    int skip_first_arrive;
    int64_t ws_floats;    // floats of scratch the kernel may touch (debug checks)
    int64_t n_counters;   // arrival counters it may touch (debug checks)
};

// Codes recorded in the status word (which wait expired first).
enum WaitSite : int {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaAccEmpty = 3,
    kSiteEpilogueAccFull = 4,
    kSiteDrain = 5,
    kSiteConvFull = 6,   // 4-bit kernel: a converter waiting for packed weights
    kSiteConvEmpty = 7,  // 4-bit kernel: a converter waiting for a free TMEM slot
    kSiteBounds = 8,     // debug builds: a device-side bounds check failed
};

struct TiledArgs {
    const __half* A;
    const __half* B;
    const __half* bias;  // may be null
    __half* C;
    int M, N, K;
    int gelu;
    int m_blocks, n_blocks, num_tiles, num_kb, group_m;
    int c_store;   // how C may be written: 2 = 16-byte units (C 16-byte aligned, N % 8 == 0),
                   // 1 = 4-byte units (C 4-byte aligned, N even), 0 = single elements
    int bias_vec;  // bias 16-byte aligned: 16-byte loads
    int a_vec;     // ordinary-load staging width for A in elements: 8, 2 or 1
    int b_vec;     // same for B
    // CTA-pair kernel: tiles [split_from, num_tiles) of the last, partial wave
    // run as two half-width units each; num_units = split_from +
    // 2 * (num_tiles - split_from), set by its launcher. Single-CTA kernel:
    // num_units = num_tiles * splits.
    int split_from, num_units;
    int bn;        // single-CTA kernel: tile width (256, or 128 / 64 when 256-wide tiles would
                   // leave most SMs idle)
    // Single-CTA kernel, K split over `splits` slices of kb_per_split K blocks (1 = no split,
    // num_units = num_tiles then): unit u is slice u / num_tiles of tile u % num_tiles, and
    // with splits > 1 each unit writes fp32 partials [slice][n][m_pad] to ws, summed by
    // launch_splitk_reduce.
    int splits, kb_per_split, m_pad;
    int tile0;     // cluster split: the launch's first tile (a split tail after whole-tile waves)
    float* ws;
    Watchdog wd;
};

struct SplitArgs {
    const __half* A;
    const __half* B;
    const __half* bias;
    __half* C;
    int M, N, K;
    int gelu;
    int m_pad;         // MMA N: M rounded up to a multiple of 16 (16..128)
    int tmem_stride;   // TMEM columns per accumulator (pow2 >= m_pad); a buffer holds
                       // kSkHalves accumulators, two buffers alternate between units
    int tmem_cols;     // TMEM columns allocated (2 * kSkHalves * tmem_stride, >= 32)
    int stages;        // ring depth
    int n_tiles, kb_total, kb_per_split, splits, num_units;
    float* ws;               // splits * N * m_pad fp32 partial sums, [slice][n][m] (splits > 1),
                             // summed by launch_splitk_reduce
    unsigned int* counters;  // 4-bit kernel: n_tiles arrival counters, zero between launches
    Watchdog wd;
};

// The 4-bit kernel: the skinny fields above (A, bias, C, sizes, m_pad,
// split bookkeeping, stages = raw ring depth) plus the packed weights, their
// scales, their format and the depth of the converted-weight ring.
struct W4Args {
    SplitArgs s;               // s.B and s.tmem_* unused
    const uint8_t* Bq;         // N rows of K/2 bytes, low nibble = even k
    const __half* scales;      // K/128 rows of N
    int fmt;                   // 0: two's-complement INT4, 1: FP4 (E2M1)
    int a_slots;               // activation slots (one 256-k stage of A each)
    int b_slots;               // converted 64-k sub-tiles in flight
    int c_vec;                 // C 16-byte aligned and N % 8 == 0: 16-byte stores
};

// The register-dequant 4-bit kernel (M <= kW4rMaxM): a CTA per kW4rCols
// output columns over the whole K.
struct W4rArgs {
    const __half* bias;
    __half* C;
    int M, N;
    int n_chunks;              // K / 256, rounded up
    int gelu;
    int fmt;                   // 0: two's-complement INT4, 1: FP4 (E2M1)
    Watchdog wd;
};

// Attention forward: (batch, sequence, head, dim) fp16, dim = kAttnD.
constexpr int kAttnD = 128;
struct AttnArgs {
    __half* O;
    int S, H;
    int causal;
    int n_qt;            // 128-query blocks per (batch, head)
    float scale_log2;    // log2(e) / sqrt(dim): scores in base-2 exponent units
    int n_plain;         // query blocks computed by one CTA each (the first in launch order)
    int n_split;         // query blocks after those, each computed by two CTAs (key halves)
    float* ws;           // n_split pairs of parts (attn_part_floats() floats each), or null
    unsigned int* counters;  // n_split arrival counters, zero between launches
    Watchdog wd;
};

// Incremented by tg_shutdown. Launchers cache per-device, per-context state
// (kernel attributes such as the dynamic shared-memory limit) together with
// the generation they were made in, and make them again when it has changed,
// so the library keeps working after tg_shutdown and a cudaDeviceReset.
// Read and written with the front end's lock held.
extern int g_generation;

cudaError_t launch_splitk_reduce(const SplitArgs& a, cudaStream_t stream);
int split_stage_bytes(int m_pad);
int split_smem_bytes(int m_pad, int stages);
int split_stages_for(int m_pad);
int tiled_smem_bytes(bool tma);
int tiled_threads(bool tma);

cudaError_t launch_tiled_tma(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             int grid, cudaStream_t stream);
// The single-CTA kernel with K split over 2..kTiledClusterMax slices as thread-block clusters
// (one CTA per slice of each 256-column tile, num_units = num_tiles * splits CTAs): the slices
// are summed in distributed shared memory, no scratch, no second kernel.
constexpr int kTiledClusterMax = 8;
// Clusters of `splits` CTAs of that kernel that fit on the current device at once (0 when
// splits is out of range or the query fails).
int tiled_cluster_capacity(int splits);
cudaError_t launch_tiled_cluster(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                 cudaStream_t stream);
cudaError_t launch_tiled_lsu(const TiledArgs& a, int grid, cudaStream_t stream);
int tiled_pair_smem_bytes();
// tmC: map of C (32 x 32 box, 64-byte swizzle) to write C by TMA stores, or
// NULL for ordinary stores.
cudaError_t launch_tiled_pair(const TiledArgs& a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const CUtensorMap* tmC, int max_clusters, cudaStream_t stream);
cudaError_t launch_splitk(const SplitArgs& a, const CUtensorMap& tmB, const CUtensorMap& tmA,
                          int grid, cudaStream_t stream);
// The skinny kernel with its 2..kTiledClusterMax K slices of each unit as one thread-block
// cluster (num_units = n_tiles * splits CTAs, one unit each), summed across the cluster's
// shared memory: no scratch, no second kernel. split_on_chip_fits: the ring holds the staged
// fp32 tile. split_cluster_capacity: such clusters resident at once (0 if unknown).
cudaError_t launch_splitk_cluster(const SplitArgs& a, const CUtensorMap& tmB, const CUtensorMap& tmA,
                                  cudaStream_t stream);
bool split_on_chip_fits(int m_pad, int stages);
int split_cluster_capacity(int splits, int m_pad, int stages);
void w4_pipeline(int m_pad, int* stages, int* act_slots, int* slots);
int w4_smem_bytes(int m_pad, int stages, int act_slots, int slots);
cudaError_t launch_w4(const W4Args& a, const CUtensorMap& tmBq, const CUtensorMap& tmA, const CUtensorMap& tmS,
                      int grid, cudaStream_t stream);
int w4r_smem_bytes();
int w4r_chunk();   // k per ring stage of the register-dequant kernel (128 or 256)
cudaError_t launch_w4r(const W4rArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmS, const CUtensorMap& tmX,
                       int grid, cudaStream_t stream);
cudaError_t launch_softmax(const __half* X, __half* Y, int M, int N, bool vec, int sm_count, cudaStream_t stream);
int attn_smem_bytes();
int attn_part_floats();
cudaError_t launch_attn(const AttnArgs& a, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                        int grid, cudaStream_t stream);
cudaError_t launch_bias_gelu(__half* C, const __half* bias, int64_t M, int64_t N, int gelu, bool vec8, int sm_count,
                             cudaStream_t stream);
cudaError_t launch_pad_rows(const __half* src, __half* dst, int64_t rows, int64_t cols, int64_t dst_ld,
                            int sm_count, cudaStream_t stream);
cudaError_t launch_fill(const __half* bias, __half* C, int64_t M, int64_t N, int gelu,
                        int sm_count, cudaStream_t stream);

}  // namespace tg
