// C-ABI front end: argument checks, kernel choice, TMA descriptors, per-stream
// scratch, the device watchdog word, and launches. The operation and its
// conventions are documented in include/tg_gemm.h.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "tg_gemm.h"
#include "tg_internal.h"

namespace tg {
int g_generation = 1;
}

namespace {

using namespace tg;

thread_local std::string t_last_error;
std::atomic<uint64_t> g_watchdog_ns{2000000000ull};
std::atomic<int> g_skip_first_arrive{0};
std::atomic<int64_t> g_bounds_limit{0};  // debug builds: cap on the scratch floats the checks allow

// First expired wait of any kernel since the last tg_device_status (0 = none).
__device__ int g_status_word;

tg_status fail(tg_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

tg_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct Scratch {
    float* ws = nullptr;
    size_t ws_bytes = 0;
    unsigned int* counters = nullptr;
    size_t n_counters = 0;
    __half* pad = nullptr;  // aligned-stride copies of operands TMA cannot describe
    size_t pad_bytes = 0;
};

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int* status_ptr = nullptr;
    std::unordered_map<cudaStream_t, Scratch> scratch;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Encoded tensor maps by (device, element type, rank, base address, extents,
// strides, box, swizzle). A map only describes an address range and its
// layout, so a hit is valid even if the memory behind the address was freed
// and allocated again; the cache saves the host cost of re-encoding on every
// call (decode-sized calls are host-latency-bound). Bounded: cleared when it
// reaches kMapCacheMax entries, and by tg_shutdown. Guarded by g_mu.
struct MapKey {
    uint64_t v[16];
    bool operator==(const MapKey& o) const { return std::memcmp(v, o.v, sizeof v) == 0; }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = 1469598103934665603ull;
        for (uint64_t x : k.v) h = (h ^ x) * 1099511628211ull;
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMapCacheMax = 4096;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
int g_map_dev = 0;  // device the current call runs on (set by current_device)

CUresult encode_cached(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       CUtensorMapSwizzle swizzle) {
    MapKey k{};
    k.v[0] = static_cast<uint64_t>(g_map_dev) | (static_cast<uint64_t>(dtype) << 16) |
             (static_cast<uint64_t>(rank) << 32) | (static_cast<uint64_t>(swizzle) << 40);
    k.v[1] = reinterpret_cast<uint64_t>(base);
    for (uint32_t i = 0; i < rank; ++i) {
        k.v[2 + i] = dims[i];
        k.v[6 + i] = box[i];
        if (i + 1 < rank) k.v[10 + i] = strides[i];
    }
    auto it = g_maps.find(k);
    if (it != g_maps.end()) {
        *m = it->second;
        return CUDA_SUCCESS;
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        if (g_maps.size() >= kMapCacheMax) g_maps.clear();
        g_maps.emplace(k, *m);
    }
    return r;
}

// Current device, checked to be compute capability 10.3; fills the per-device
// state on first use. Caller holds g_mu.
tg_status current_device(int* dev_out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(TG_ERR_UNSUPPORTED_DEVICE, "device ordinal %d out of range", dev);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return fail(TG_ERR_UNSUPPORTED_DEVICE, "device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                        dev, major, minor);
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status_ptr), g_status_word)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
                return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        d.ready = true;
    }
    g_map_dev = dev;
    *dev_out = dev;
    return TG_OK;
}

// C (M x N fp16, row-major) for the epilogue's TMA stores: 32 x 32 boxes,
// 64-byte swizzle.
tg_status make_map_c(CUtensorMap* m, const void* base, uint64_t N, uint64_t M) {
    cuuint64_t dims[2] = {N, M};
    cuuint64_t strides[1] = {N * 2};
    cuuint32_t box[2] = {32, 32};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_64B);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the %llu x %llu output", (int)r,
                    (unsigned long long)M, (unsigned long long)N);
    return TG_OK;
}

// Row-major [outer][inner] byte matrix, box of box_inner x box_outer bytes,
// 128-byte swizzle (or none); out-of-bounds bytes read as zero.
tg_status make_map_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                      uint32_t box_outer, bool swizzle = true) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {box_inner, box_outer};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box,
                               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu byte matrix", (int)r,
                    (unsigned long long)outer, (unsigned long long)inner);
    return TG_OK;
}

// Row-major [outer][inner] fp16 matrix, unswizzled box (the 4-bit GEMM's scale rows).
tg_status make_map_scales(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                          uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu scale matrix", (int)r,
                    (unsigned long long)outer, (unsigned long long)inner);
    return TG_OK;
}

// M x K fp16 activations (row-major, M <= 16) as a 3-D map {64, K/64, M}: box
// {64, chunk/64, 16} = 16 rows x chunk k whose 128-byte lines are (row, 64-k
// block) pairs, 128-byte swizzle; rows past M read as zero.
tg_status make_map_x3(CUtensorMap* m, const void* base, uint64_t M, uint64_t K, uint32_t chunk) {
    cuuint64_t dims[3] = {64, K / 64, M};
    cuuint64_t strides[2] = {128, K * 2};
    cuuint32_t box[3] = {64, chunk / 64, 16};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the %llu x %llu activations", (int)r,
                    (unsigned long long)M, (unsigned long long)K);
    return TG_OK;
}

// (batch, sequence, head, dim) fp16 tensor as a 4-D map, innermost first:
// {dim, head, sequence, batch}; box {64, 1, 128, 1} with the 128-byte swizzle
// (one 64-column slice of 128 consecutive positions of one head).
tg_status make_map_bshd(CUtensorMap* m, const void* base, uint64_t B, uint64_t S, uint64_t H, uint64_t D) {
    cuuint64_t dims[4] = {D, H, S, B};
    cuuint64_t strides[3] = {D * 2, H * D * 2, S * H * D * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu x %llu x %llu tensor", (int)r,
                    (unsigned long long)B, (unsigned long long)S, (unsigned long long)H, (unsigned long long)D);
    return TG_OK;
}

// Row-major [outer][inner] fp16 matrix with a row stride of `ld` elements
// (a multiple of 8), 128-byte-swizzled box.
tg_status make_map_ld(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                      uint32_t box_inner, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    CUresult r = encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (r != CUDA_SUCCESS)
        return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llu x %llu matrix (row stride %llu)",
                    (int)r, (unsigned long long)outer, (unsigned long long)inner, (unsigned long long)ld);
    return TG_OK;
}

// Row-major [outer][inner] fp16 matrix, 128-byte-swizzled box.
tg_status make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                   uint32_t box_outer) {
    return make_map_ld(m, base, inner, outer, inner, box_inner, box_outer);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    if (!a || !b || a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

int vec_width(const void* p, int64_t ld) {
    if (ld % 8 == 0 && aligned(p, 16)) return 8;
    if (ld % 2 == 0 && aligned(p, 4)) return 2;
    return 1;
}

// The kernels' watchdog settings; no scratch until the caller grants some (debug_limits).
Watchdog watchdog(const DeviceState& d) {
    return Watchdog{d.status_ptr, g_watchdog_ns.load(), g_skip_first_arrive.load(), 0, 0};
}

// The scratch a kernel may touch, for the bounds checks of debug builds (capped by the
// tg_debug_bounds_limit test hook).
void debug_limits(Watchdog& wd, size_t ws_bytes, size_t n_counters) {
    int64_t floats = static_cast<int64_t>(ws_bytes / sizeof(float));
    const int64_t cap = g_bounds_limit.load();
    if (cap > 0 && cap < floats) floats = cap;
    wd.ws_floats = floats;
    wd.n_counters = static_cast<int64_t>(n_counters);
}

// Tile rows per rasterisation group: A strips of about kGroupBytes, at least 1,
// at most all tile rows.
int group_rows(int tile_rows, int K, int m_blocks) {
    const int64_t strip = static_cast<int64_t>(tile_rows) * K * 2;
    int64_t g = strip > 0 ? kGroupBytes / strip : m_blocks;
    if (g < 1) g = 1;
    if (g > m_blocks) g = m_blocks;
    return static_cast<int>(g);
}

// Split count for the skinny kernels. Time is modelled in units of one K
// block's transfer at one SM's streaming rate: a CTA's share is its waves of
// work units, each costing its K blocks plus a fixed charge for refilling the
// pipeline and running the epilogue (unit_overhead, in K blocks). HBM
// saturates before every SM streams, so the job can never beat
// total / (kHbmFraction * SMs). Every split beyond the first adds the
// partial-sum traffic of the final reduction (reduce_per_split, in K blocks).
// Ties keep fewer splits. The fp16 kernel streams HBM at full rate from 70%
// of the SMs; the 4-bit kernel is limited per SM (decoding and staging the
// weights), so every SM counts and its K block (256 x 256 packed, 32 KB) is
// charged less fixed overhead.
// extra(s): a further cost of s slices (the skinny path charges a split summed through scratch
// for the reduction kernel's launch, ~6 us or 11 K blocks, which a split summed on chip avoids).
template <typename Extra>
int choose_splits(int n_tiles, int kb_total, int sm_count, double unit_overhead, double reduce_per_split,
                  double hbm_fraction, Extra extra) {
    const double kUnitOverhead = unit_overhead;
    const double kReducePerSplit = reduce_per_split;
    const double kHbmFraction = hbm_fraction;  // share of SMs whose streams saturate HBM
    const double hbm_floor = static_cast<double>(n_tiles) * kb_total / (kHbmFraction * sm_count);
    int best_s = 1;
    double best = 1e300;
    const int smax = kb_total < kSkMaxSplits ? kb_total : kSkMaxSplits;
    for (int s = 1; s <= smax; ++s) {
        const int kbps = (kb_total + s - 1) / s;
        const int s_eff = (kb_total + kbps - 1) / kbps;
        if (s_eff != s) continue;
        const long units = static_cast<long>(n_tiles) * s;
        const long waves = (units + sm_count - 1) / sm_count;
        double t = static_cast<double>(waves) * (kbps + kUnitOverhead);
        if (t < hbm_floor) t = hbm_floor;
        const double cost = t + kReducePerSplit * (s - 1) + extra(s);
        if (cost < best) {
            best = cost;
            best_s = s;
        }
    }
    return best_s;
}

int choose_splits(int n_tiles, int kb_total, int sm_count, double unit_overhead = 6.0,
                  double reduce_per_split = 2.0, double hbm_fraction = 0.7) {
    return choose_splits(n_tiles, kb_total, sm_count, unit_overhead, reduce_per_split, hbm_fraction,
                         [](int) { return 0.0; });
}

tg_status ensure_scratch(DeviceState& d, cudaStream_t stream, size_t ws_bytes, size_t n_counters, Scratch** out) {
    Scratch& s = d.scratch[stream];
    cudaError_t e;
    if (s.ws_bytes < ws_bytes) {
        if (s.ws) cudaFree(s.ws);
        s.ws = nullptr;
        s.ws_bytes = 0;
        if ((e = cudaMalloc(reinterpret_cast<void**>(&s.ws), ws_bytes)) != cudaSuccess) {
            cudaGetLastError();
            return fail(TG_ERR_NO_MEMORY, "split-K scratch of %zu bytes: %s", ws_bytes, cudaGetErrorString(e));
        }
        s.ws_bytes = ws_bytes;
    }
    if (s.n_counters < n_counters) {
        if (s.counters) cudaFree(s.counters);
        s.counters = nullptr;
        s.n_counters = 0;
        if ((e = cudaMalloc(reinterpret_cast<void**>(&s.counters), n_counters * sizeof(unsigned int))) != cudaSuccess) {
            cudaGetLastError();
            return fail(TG_ERR_NO_MEMORY, "split-K counters: %s", cudaGetErrorString(e));
        }
        if ((e = cudaMemsetAsync(s.counters, 0, n_counters * sizeof(unsigned int), stream)) != cudaSuccess)
            return cuda_fail(e, "cudaMemsetAsync(counters)");
        s.n_counters = n_counters;
    }
    *out = &s;
    return TG_OK;
}

// The skinny kernel's arguments for one call, all but its scratch pointers.
#ifndef TG_SPLIT_CLUSTER
#define TG_SPLIT_CLUSTER 1
#endif

// split_k > 0 fixes the number of K slices; 0 takes the cost model's choice,
// capped at max_splits (at least 1).
void splitk_args(const DeviceState& d, const __half* A, const __half* B, const __half* bias, __half* C, int M, int N,
                 int K, int gelu, int split_k, int max_splits, SplitArgs& a) {
    a = SplitArgs{};
    a.A = A; a.B = B; a.bias = bias; a.C = C;
    a.M = M; a.N = N; a.K = K; a.gelu = gelu;
    a.m_pad = (M + 15) / 16 * 16;
    a.tmem_stride = 16;
    while (a.tmem_stride < a.m_pad) a.tmem_stride *= 2;
    a.tmem_cols = 2 * kSkHalves * a.tmem_stride < 32 ? 32 : 2 * kSkHalves * a.tmem_stride;
    a.stages = split_stages_for(a.m_pad);
    a.n_tiles = (N + kSkBN - 1) / kSkBN;
    a.kb_total = (K + kSkBK - 1) / kSkBK;
    int s = split_k;
    if (s <= 0) {
        const int m_pad = a.m_pad, stages = a.stages, n_tiles = a.n_tiles;
        s = choose_splits(a.n_tiles, a.kb_total, d.sm_count, 6.0, 2.0, 0.7, [&](int c) {
            const bool on_chip = TG_SPLIT_CLUSTER && c <= kTiledClusterMax && split_on_chip_fits(m_pad, stages) &&
                                 n_tiles <= split_cluster_capacity(c, m_pad, stages);
            return c > 1 && !on_chip ? 11.0 : 0.0;
        });
        if (s > max_splits) s = max_splits;
    }
    if (s > a.kb_total) s = a.kb_total;
    if (s < 1) s = 1;
    a.kb_per_split = (a.kb_total + s - 1) / s;
    a.splits = (a.kb_total + a.kb_per_split - 1) / a.kb_per_split;
    a.num_units = a.n_tiles * a.splits;
    a.wd = watchdog(d);
}

// True when the skinny kernel's K slices run as clusters summed on chip: 2..kTiledClusterMax
// slices, the staged fp32 tile fits the ring, and every unit's cluster is resident at once.
bool split_on_chip(const SplitArgs& a) {
    return TG_SPLIT_CLUSTER && a.splits > 1 && a.splits <= kTiledClusterMax && split_on_chip_fits(a.m_pad, a.stages) &&
           a.n_tiles <= split_cluster_capacity(a.splits, a.m_pad, a.stages);
}

// Tensor maps and launch of the skinny kernel, its scratch (when the slices are not summed
// on chip) already in `a`.
tg_status splitk_launch(const DeviceState& d, const SplitArgs& a, cudaStream_t stream) {
    CUtensorMap tmB, tmA;
    tg_status st = make_map(&tmB, a.B, a.N, a.K, 64, kSkBK);
    if (st != TG_OK) return st;
    if ((st = make_map(&tmA, a.A, a.K, a.M, kSkBK, a.m_pad)) != TG_OK) return st;
    if (split_on_chip(a)) {
        const cudaError_t e = launch_splitk_cluster(a, tmB, tmA, stream);
        return e == cudaSuccess ? TG_OK : cuda_fail(e, "split-K cluster kernel launch");
    }
    const int grid = a.num_units < d.sm_count ? a.num_units : d.sm_count;
    cudaError_t e = launch_splitk(a, tmB, tmA, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "split-K kernel launch");
    if (a.splits > 1 && (e = launch_splitk_reduce(a, stream)) != cudaSuccess)
        return cuda_fail(e, "split-K reduction launch");
    return TG_OK;
}

tg_status run_splitk(DeviceState& d, const __half* A, const __half* B, const __half* bias, __half* C, int M, int N,
                     int K, int gelu, int split_k, cudaStream_t stream) {
    SplitArgs a;
    splitk_args(d, A, B, bias, C, M, N, K, gelu, split_k, kSkMaxSplits, a);
    if (a.splits > 1 && !split_on_chip(a)) {
        Scratch* sc = nullptr;
        // the partials only: the reduction kernel needs no arrival counters
        tg_status st = ensure_scratch(d, stream, static_cast<size_t>(a.splits) * N * a.m_pad * sizeof(float), 0, &sc);
        if (st != TG_OK) return st;
        a.ws = sc->ws;
        debug_limits(a.wd, sc->ws_bytes, 0);
    }
    return splitk_launch(d, a, stream);
}

// Tile width of the single-CTA kernel without a K split: narrower tiles (128, then 64
// columns) while 256-wide ones would leave more than half of the SMs idle: small and
// ragged problems are latency-bound, more CTAs finish sooner.
int tiled_bn(const DeviceState& d, int64_t m_blocks, int64_t N) {
    int bn = kBN;
    while (bn > 64 && m_blocks * ((N + bn - 1) / bn) < d.sm_count / 2) bn /= 2;
    return bn;
}

#ifndef TG_TILED_CLUSTER_SPLIT
#define TG_TILED_CLUSTER_SPLIT 1
#endif

// True when a K split of `splits` slices runs as clusters that sum the slices on chip: TMA
// loads, at most kTiledClusterMax slices, and every tile's cluster resident at once.
bool tiled_on_chip(bool tma, int64_t tiles256, int splits) {
    return TG_TILED_CLUSTER_SPLIT && tma && splits > 1 && splits <= kTiledClusterMax &&
           tiles256 <= tiled_cluster_capacity(splits);
}

// K slices for the single-CTA kernel (1 = no split), from a time model fitted to GB300
// measurements (N, K in 2048..28672, M in 64..1024; wherever the tiled kernel runs, its pick
// is within 1% of the fastest measured choice). Times in us: a K block costs 0.36 (a 128 x
// 256 tile) or 0.26 (128 or 64 columns: loads, not MMAs, bound those tiles) per wave; reading
// A and B once from HBM at ~7.4 TB/s is the other term, and the two combine as a 2.5-norm (the
// larger dominates, the smaller still counts). A split adds 5.5 when the slices of each tile
// run as one cluster and are summed on chip, or 7.4 plus 0.44 per MB of fp32 partials when
// they go through scratch and the reduction kernel. Only problems whose 256-wide tiles number
// fewer than the SMs are split.
int tiled_splits(const DeviceState& d, int64_t M, int64_t N, int64_t K, bool tma) {
    const int64_t m_blocks = (M + kBM - 1) / kBM;
    const int64_t kb = (K + kBK - 1) / kBK;
    const int64_t tiles256 = m_blocks * ((N + kBN - 1) / kBN);
    if (tiles256 >= d.sm_count) return 1;
    const double hbm = (static_cast<double>(M) * K + static_cast<double>(K) * N) * 2.0 / 1e6 / 7.4;
    auto time = [&](double compute) { return std::pow(std::pow(compute, 2.5) + std::pow(hbm, 2.5), 0.4); };
    const int bn = tiled_bn(d, m_blocks, N);
    const int64_t tiles = m_blocks * ((N + bn - 1) / bn);
    double best = time(static_cast<double>((tiles + d.sm_count - 1) / d.sm_count) * kb * (bn == 256 ? 0.36 : 0.26));
    int best_s = 1;
    const double m_pad = static_cast<double>((M + 15) / 16 * 16);
    for (int s = 2; s <= kSkMaxSplits && s <= kb; ++s) {
        const int64_t kbps = (kb + s - 1) / s;
        if ((kb + kbps - 1) / kbps != s) continue;
        double t;
        if (tiled_on_chip(tma, tiles256, s)) {
            t = time(static_cast<double>(kbps) * 0.36) + 5.5;
        } else {
            const int64_t waves = (tiles256 * s + d.sm_count - 1) / d.sm_count;
            t = time(static_cast<double>(waves) * kbps * 0.36) + 7.4 + 0.44 * s * m_pad * static_cast<double>(N) * 4.0 / 1e6;
        }
        if (t < best) {
            best = t;
            best_s = s;
        }
    }
    return best_s;
}

// A tail split for the single-CTA kernel with TMA loads: when its 128 x 256 tiles fill whole
// waves plus a short last one, the whole waves run as usual and the last wave's tiles run K
// split over `s` slices as clusters summed on chip (one more launch), instead of a wave of a
// few tiles with most SMs idle. Returns s (0: no tail split). The tail costs a launch of K / s
// blocks (0.36 us each) plus 11.5 us against a whole wave of K blocks at 0.41 us each (GB300).
int tiled_tail_split(const DeviceState& d, int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int64_t rest = tiles % d.sm_count;
    if (tiles < d.sm_count || rest == 0) return 0;
    const int64_t kb = (K + kBK - 1) / kBK;
    const double whole = static_cast<double>(kb) * 0.41;
    double best = whole;
    int best_s = 0;
    for (int s = 2; s <= kTiledClusterMax && s <= kb; ++s) {
        if (rest > tiled_cluster_capacity(s)) continue;
        const double t = static_cast<double>((kb + s - 1) / s) * 0.36 + 11.5;
        if (t < best) {
            best = t;
            best_s = s;
        }
    }
    return best_s;
}

tg_status run_tiled(DeviceState& d, bool tma, const __half* A, const __half* B, const __half* bias, __half* C, int M,
                    int N, int K, int gelu, cudaStream_t stream, int64_t lda = 0, int64_t ldb = 0, int split_k = 0) {
    TiledArgs a{};
    a.A = A; a.B = B; a.bias = bias; a.C = C;
    a.M = M; a.N = N; a.K = K; a.gelu = gelu;
    a.m_blocks = (M + kBM - 1) / kBM;
    a.num_kb = (K + kBK - 1) / kBK;
    int s = split_k > 0 ? split_k : tiled_splits(d, M, N, K, tma);
    if (s > a.num_kb) s = a.num_kb;
    a.kb_per_split = (a.num_kb + s - 1) / s;
    a.splits = (a.num_kb + a.kb_per_split - 1) / a.kb_per_split;
    // a split problem keeps the full-width tiles (their MMAs are the most efficient); the
    // slices fill the SMs
    a.bn = a.splits > 1 ? kBN : tiled_bn(d, a.m_blocks, N);
    a.n_blocks = (N + a.bn - 1) / a.bn;
    a.num_tiles = a.m_blocks * a.n_blocks;
    a.num_units = a.num_tiles * a.splits;
    a.m_pad = (M + 15) / 16 * 16;
    a.group_m = group_rows(kBM, K, a.m_blocks);
    a.c_store = (N % 8 == 0 && aligned(C, 16)) ? 2 : ((N % 2 == 0 && aligned(C, 4)) ? 1 : 0);
    a.bias_vec = (bias != nullptr && aligned(bias, 16)) ? 1 : 0;
    a.a_vec = vec_width(A, K);
    a.b_vec = vec_width(B, N);
    a.wd = watchdog(d);
    // slices summed on chip by clusters when they fit (tiled_on_chip); otherwise through scratch
    // and the reduction kernel
    const bool on_chip = tiled_on_chip(tma, static_cast<int64_t>(a.m_blocks) * ((N + kBN - 1) / kBN), a.splits);
    if (a.splits > 1 && !on_chip) {
        if ((static_cast<int64_t>(M) + 15) / 16 > 65535)
            return fail(TG_ERR_INVALID_ARG, "a K split of the tiled kernels supports M <= 1048560, got %d", M);
        Scratch* sc = nullptr;
        tg_status st = ensure_scratch(d, stream, static_cast<size_t>(a.splits) * N * a.m_pad * sizeof(float), 0, &sc);
        if (st != TG_OK) return st;
        a.ws = sc->ws;
        debug_limits(a.wd, sc->ws_bytes, 0);
    }
    const int grid = a.num_units < d.sm_count ? a.num_units : d.sm_count;
    cudaError_t e;
    // whole waves, then the short last wave's tiles split over K (automatic choice only)
    const int tail_s = (tma && split_k == 0 && a.splits == 1 && a.bn == kBN) ? tiled_tail_split(d, M, N, K) : 0;
    if (tma) {
        CUtensorMap tmA, tmB;
        tg_status st = make_map_ld(&tmA, A, K, M, lda ? lda : K, kBK, kBM);
        if (st != TG_OK) return st;
        if ((st = make_map_ld(&tmB, B, N, K, ldb ? ldb : N, 64, kBK)) != TG_OK) return st;
        if (tail_s > 1) {
            const int whole = a.num_tiles - a.num_tiles % d.sm_count;
            TiledArgs w = a;
            w.num_units = whole;  // tiles [0, whole), one slice each
            if ((e = launch_tiled_tma(w, tmA, tmB, d.sm_count, stream)) != cudaSuccess)
                return cuda_fail(e, "tiled kernel launch");
            TiledArgs t = a;
            t.tile0 = whole;
            t.kb_per_split = (a.num_kb + tail_s - 1) / tail_s;
            t.splits = (a.num_kb + t.kb_per_split - 1) / t.kb_per_split;
            t.num_units = (a.num_tiles - whole) * t.splits;
            e = launch_tiled_cluster(t, tmA, tmB, stream);
        } else {
            e = on_chip ? launch_tiled_cluster(a, tmA, tmB, stream) : launch_tiled_tma(a, tmA, tmB, grid, stream);
        }
    } else {
        e = launch_tiled_lsu(a, grid, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "tiled kernel launch");
    if (a.splits > 1 && !on_chip) {
        // the skinny path's reduction: slices summed in order, then bias, GELU, one rounding
        SplitArgs r{};
        r.bias = bias; r.C = C;
        r.M = M; r.N = N; r.K = K; r.gelu = gelu;
        r.m_pad = a.m_pad;
        r.splits = a.splits;
        r.ws = a.ws;
        r.wd = a.wd;
        if ((e = launch_splitk_reduce(r, stream)) != cudaSuccess) return cuda_fail(e, "split-K reduction launch");
    }
    return TG_OK;
}

// The pair kernel writes an aligned C by TMA stores (else by ordinary stores).
#ifndef TG_PAIR_TMA_STORE
#define TG_PAIR_TMA_STORE 1
#endif
constexpr bool kPairTmaStore = TG_PAIR_TMA_STORE != 0;

tg_status run_tiled_pair(DeviceState& d, const __half* A, const __half* B, const __half* bias, __half* C, int M,
                         int N, int K, int gelu, cudaStream_t stream, int64_t lda = 0, int64_t ldb = 0) {
    TiledArgs a{};
    a.A = A; a.B = B; a.bias = bias; a.C = C;
    a.M = M; a.N = N; a.K = K; a.gelu = gelu;
    a.m_blocks = (M + 2 * kBM - 1) / (2 * kBM);
    a.bn = kBN;
    a.n_blocks = (N + kBN - 1) / kBN;
    a.num_tiles = a.m_blocks * a.n_blocks;
    a.num_kb = (K + kBK - 1) / kBK;
    a.group_m = group_rows(2 * kBM, K, a.m_blocks);
    a.c_store = (N % 8 == 0 && aligned(C, 16)) ? 2 : ((N % 2 == 0 && aligned(C, 4)) ? 1 : 0);
    a.bias_vec = (bias != nullptr && aligned(bias, 16)) ? 1 : 0;
    a.a_vec = a.b_vec = 8;
    a.wd = watchdog(d);
    CUtensorMap tmA, tmB, tmC;
    tg_status st = make_map_ld(&tmA, A, K, M, lda ? lda : K, kBK, kBM);
    if (st != TG_OK) return st;
    if ((st = make_map_ld(&tmB, B, N, K, ldb ? ldb : N, 64, kBK)) != TG_OK) return st;
    // C aligned for TMA (16-byte base, rows of a multiple of 16 bytes): the epilogue writes it by
    // TMA stores of 32 x 32 boxes
    const bool tma_store = kPairTmaStore && a.c_store == 2;
    if (tma_store && (st = make_map_c(&tmC, C, N, M)) != TG_OK) return st;
    cudaError_t e = launch_tiled_pair(a, tmA, tmB, tma_store ? &tmC : nullptr, d.sm_count / 2, stream);
    if (e != cudaSuccess) return cuda_fail(e, "pair tiled kernel launch");
    return TG_OK;
}

// Unaligned operands: products of at least this many flops take the aligned-copy path.
constexpr double kCopyPathFlops = 4294967296.0;  // 2^32

// True when the CTA-pair kernel beats the single-CTA kernel (with its K split). When the
// single-CTA kernel's tiles fill a wave and the pairs' fewer than eight, by a time model of
// their waves (below); with more, always; otherwise with at least one wave of 256x256
// tiles, or, for K >= 8192, at least 0.3 of a wave (measured on GB300:
// 8192 x 8192 at M = 512, 64 pair tiles, 49 vs 55 us; 4096 x 14336 at M = 768, 48 tiles,
// 76 vs 85 us; with K = 4096 the single-CTA kernel stays ahead at 48-64 tiles).
bool pair_pays(const DeviceState& d, int64_t M, int64_t N, int64_t K) {
    const int64_t pair_tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + kBN - 1) / kBN);
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int64_t clusters = d.sm_count / 2;
    if (tiles >= d.sm_count && pair_tiles < 8 * clusters) {
        // both kernels fill at least a wave, and the last wave still weighs: compare their
        // times (us). A wave of K blocks costs 0.41 per block for single-CTA tiles, 0.97 of
        // that for pairs. The pairs' last wave costs 0.63 of one when it fits as half-width
        // units. The single-CTA kernel's last wave may instead run K-split on chip: a second
        // launch of K / s blocks at 0.36 plus 11.5. 14336 x 4096 at M = 640: single CTAs
        // 57.5 us against pairs 68.9; 8192 x 8192 at M = 640 (split tail): 73.9 vs 87.8;
        // 14336 x 4096 at M = 384: pairs 48.9 vs 52.7; 28672 x 8192 at M = 640: single CTAs 233
        // vs 258. From eight waves of pairs on (square 8192, the FFN shapes) the pairs stay.
        const double kb = static_cast<double>((K + kBK - 1) / kBK);
        const int64_t prest = pair_tiles % clusters;
        const double pair = 0.97 * 0.41 * kb *
                            (static_cast<double>(pair_tiles / clusters) +
                             (prest == 0 ? 0.0 : 2 * prest <= clusters ? 0.63 : 1.0));
        const int64_t trest = tiles % d.sm_count;
        double tail = trest == 0 ? 0.0 : 0.41 * kb;
        if (trest > 0)
            for (int s = 2; s <= kTiledClusterMax && s <= kb; ++s)
                if (trest <= tiled_cluster_capacity(s)) {
                    const double t = std::ceil(kb / s) * 0.36 + 11.5;
                    if (t < tail) tail = t;
                }
        return pair < static_cast<double>(tiles / d.sm_count) * 0.41 * kb + tail;
    }
    if (tiles >= d.sm_count) return true;
    if (pair_tiles >= d.sm_count / 2) return true;
    return K >= 8192 && 10 * pair_tiles >= 3 * static_cast<int64_t>(d.sm_count);
}

// True when the skinny split-K kernel beats the single-CTA tiled kernel for M <= 128
// (measured on GB300 over N = 2048..28672, K = 2048..28672, M = 16..128, both kernels summing
// their K slices on chip where they can). With K >= 2048, skinny up to 64 rows and tiled above
// (the tiled kernel wins by up to 9% at 48-64 rows on 14336 x 4096 and 4096 x 8192, skinny by
// up to 16% elsewhere at those sizes; at 96 rows and up the tiled kernel is within 5%). For
// shorter K, outside that sweep, the earlier rule against the unsplit tiled kernel: with
// fewer 64-column tiles than SMs, skinny when K/64 times the SMs per tile is at least 1.5 M;
// otherwise only when, with M <= 64, the product streams 256 MiB or more of B.
bool skinny_pays(const DeviceState& d, int64_t M, int64_t N, int64_t K) {
    if (M <= 16) return true;
    if (K >= 2048) return M <= 64;
    const int64_t tiles64 = (N + 63) / 64;  // one 128-row block: M <= 128
    const int64_t kb = (K + 63) / 64;
    if (tiles64 < d.sm_count) return 2 * kb * d.sm_count >= 3 * M * tiles64;
    return M <= 64 && 2.0 * static_cast<double>(K) * static_cast<double>(N) >= 256.0 * 1048576.0;
}

// A GEMM whose A or B TMA cannot describe (row stride not a multiple of 16
// bytes, or base not 16-byte aligned): each such operand is first copied into
// the stream's aligned-stride buffer (row stride rounded up to 8 elements),
// then the TMA kernels run on the copies with the original logical extents.
tg_status run_padded(DeviceState& d, const __half* A, const __half* B, const __half* bias, __half* C, int M, int N,
                     int K, int gelu, cudaStream_t stream) {
    const bool pad_a = K % 8 != 0 || !aligned(A, 16);
    const bool pad_b = N % 8 != 0 || !aligned(B, 16);
    const int64_t lda = pad_a ? (static_cast<int64_t>(K) + 7) / 8 * 8 : K;
    const int64_t ldb = pad_b ? (static_cast<int64_t>(N) + 7) / 8 * 8 : N;
    const size_t a_bytes = pad_a ? static_cast<size_t>(M) * lda * 2 : 0;  // multiple of 16
    const size_t b_bytes = pad_b ? static_cast<size_t>(K) * ldb * 2 : 0;
    Scratch& s = d.scratch[stream];
    if (s.pad_bytes < a_bytes + b_bytes) {
        if (s.pad) cudaFree(s.pad);
        s.pad = nullptr;
        s.pad_bytes = 0;
        cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&s.pad), a_bytes + b_bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(TG_ERR_NO_MEMORY, "aligned operand copies of %zu bytes: %s", a_bytes + b_bytes,
                        cudaGetErrorString(e));
        }
        s.pad_bytes = a_bytes + b_bytes;
    }
    const __half* a = A;
    const __half* b = B;
    cudaError_t e;
    if (pad_a) {
        if ((e = launch_pad_rows(A, s.pad, M, K, lda, d.sm_count, stream)) != cudaSuccess)
            return cuda_fail(e, "copy of A to an aligned stride");
        a = s.pad;
    }
    if (pad_b) {
        __half* pb = s.pad + a_bytes / 2;
        if ((e = launch_pad_rows(B, pb, K, N, ldb, d.sm_count, stream)) != cudaSuccess)
            return cuda_fail(e, "copy of B to an aligned stride");
        b = pb;
    }
    if (pair_pays(d, M, N, K)) return run_tiled_pair(d, a, b, bias, C, M, N, K, gelu, stream, lda, ldb);
    return run_tiled(d, true, a, b, bias, C, M, N, K, gelu, stream, lda, ldb);
}

// The automatic choice of tg_gemm: the kernel, whether operands are first copied to aligned
// strides, and the K slices (1 = none) the chosen kernel's own model takes.
struct Plan {
    int kernel;
    bool copy;
    int splits;
};

Plan plan_auto(const DeviceState& d, int64_t M, int64_t N, int64_t K, bool tma_ok) {
    Plan p{TG_KERNEL_TILED_TMA, false, 1};
    if (!tma_ok) {
        // large problems: an aligned copy of the operand plus the TMA kernels beats staging it
        // by 4- or 2-byte loads (4096 x 4094 x 4096: 3.6x); small ones are latency-bound and the
        // copy's launch costs more than it saves (1000 x 1030 x 520: 19.3 vs 17.3 us); skinny M
        // keeps the loads (a copy would double the weight traffic that bounds it)
        if (M > kSkMaxM && 2.0 * M * N * K >= kCopyPathFlops) {
            p.copy = true;
            p.kernel = pair_pays(d, M, N, K) ? TG_KERNEL_TILED_PAIR : TG_KERNEL_TILED_TMA;
        } else {
            p.kernel = TG_KERNEL_TILED_LSU;
        }
    } else if (M <= kSkMaxM) {
        // 256-row pair tiles would be mostly padding here
        p.kernel = skinny_pays(d, M, N, K) ? TG_KERNEL_SPLITK : TG_KERNEL_TILED_TMA;
    } else {
        // CTA pairs once there are enough 256x256 tiles for them (pair_pays); smaller problems
        // keep more, smaller tiles on single CTAs, with K split when they leave SMs idle
        p.kernel = pair_pays(d, M, N, K) ? TG_KERNEL_TILED_PAIR : TG_KERNEL_TILED_TMA;
    }
    if (K > 0 && p.kernel == TG_KERNEL_SPLITK) {
        SplitArgs a;
        splitk_args(d, nullptr, nullptr, nullptr, nullptr, static_cast<int>(M), static_cast<int>(N),
                    static_cast<int>(K), 0, 0, kSkMaxSplits, a);
        p.splits = a.splits;
    } else if (K > 0 && p.kernel != TG_KERNEL_TILED_PAIR) {
        const int kb = static_cast<int>((K + kBK - 1) / kBK);
        int s = tiled_splits(d, M, N, K, p.kernel == TG_KERNEL_TILED_TMA);
        if (s > kb) s = kb;
        const int kbps = (kb + s - 1) / s;
        p.splits = (kb + kbps - 1) / kbps;
        if (p.splits == 1 && p.kernel == TG_KERNEL_TILED_TMA) {
            const int t = tiled_tail_split(d, M, N, K);  // whole waves, then a split last wave
            if (t > 1) p.splits = (kb + (kb + t - 1) / t - 1) / ((kb + t - 1) / t);
        }
    }
    return p;
}

// ---------------------------------------------------------------------------
// tg_gemm_splitk_noalloc: the skinny split-K path with its scratch in a fixed
// array of the library's own device image instead of library-allocated memory.

// Layout: a reserved area of 4 bytes per 256-column slice of N (padded to 256 bytes; the
// reduction kernel needs no arrival counters, the area keeps the documented size rule),
// then the fp32 partial sums [split][N][M rounded up to 16]. Loaded with the library's device
// code, so every device that loads the library holds these bytes until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TG_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch for each device, looked up on the first
// call on that device (with that device current).
unsigned char* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

extern "C" {

tg_status tg_gemm_ex(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                     int epilogue, int kernel, int split_k, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    // ---- arguments (host only, nothing enqueued on failure)
    if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_GELU)
        return fail(TG_ERR_INVALID_ARG, "epilogue must be TG_EPI_NONE (0) or TG_EPI_GELU (1), got %d", epilogue);
    if (kernel < TG_KERNEL_AUTO || kernel > TG_KERNEL_TILED_PAIR)
        return fail(TG_ERR_INVALID_ARG, "unknown kernel %d", kernel);
    const int64_t kMax = 0x7FFFFFFFll;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                    (long long)N, (long long)K);
    if (split_k < 0 || split_k > kSkMaxSplits)
        return fail(TG_ERR_INVALID_ARG, "split_k must be 0 (automatic) or 1..%d, got %d", kSkMaxSplits, split_k);
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr) return fail(TG_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(TG_ERR_INVALID_ARG, "A or B is NULL");
    const int64_t c_bytes = M * N * 2;
    if (overlaps(C, c_bytes, A, K > 0 ? M * K * 2 : 0) || overlaps(C, c_bytes, B, K > 0 ? K * N * 2 : 0) ||
        overlaps(C, c_bytes, bias, bias ? N * 2 : 0))
        return fail(TG_ERR_INVALID_ARG, "C overlaps an input");
    const bool tma_ok = K % 8 == 0 && N % 8 == 0 && aligned(A, 16) && aligned(B, 16);
    if ((kernel == TG_KERNEL_TILED_TMA || kernel == TG_KERNEL_TILED_PAIR) && !tma_ok)
        return fail(TG_ERR_INVALID_ARG, "%s needs K %% 8 == 0, N %% 8 == 0 and 16-byte aligned A, B",
                    kernel == TG_KERNEL_TILED_TMA ? "TG_KERNEL_TILED_TMA" : "TG_KERNEL_TILED_PAIR");
    if (kernel == TG_KERNEL_SPLITK && (!tma_ok || M > kSkMaxM))
        return fail(TG_ERR_INVALID_ARG, "TG_KERNEL_SPLITK needs M <= %d, K %% 8 == 0, N %% 8 == 0 and 16-byte aligned A, B",
                    kSkMaxM);
    if (split_k > 0 && kernel == TG_KERNEL_TILED_PAIR)
        return fail(TG_ERR_INVALID_ARG, "split_k does not apply to TG_KERNEL_TILED_PAIR");

    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    DeviceState& d = g_dev[dev];
    const __half* a = static_cast<const __half*>(A);
    const __half* b = static_cast<const __half*>(B);
    const __half* bi = static_cast<const __half*>(bias);
    __half* c = static_cast<__half*>(C);
    const int gelu = epilogue == TG_EPI_GELU ? 1 : 0;

    if (K == 0) {
        cudaError_t e = launch_fill(bi, c, M, N, gelu, d.sm_count, stream);
        return e == cudaSuccess ? TG_OK : cuda_fail(e, "fill kernel launch");
    }
    int k = kernel;
    if (k == TG_KERNEL_AUTO) {
        const Plan p = plan_auto(d, M, N, K, tma_ok);
        if (p.copy) return run_padded(d, a, b, bi, c, (int)M, (int)N, (int)K, gelu, stream);
        k = p.kernel;
    }
    if (k == TG_KERNEL_SPLITK)
        return run_splitk(d, a, b, bi, c, (int)M, (int)N, (int)K, gelu, split_k, stream);
    if (k == TG_KERNEL_TILED_PAIR) return run_tiled_pair(d, a, b, bi, c, (int)M, (int)N, (int)K, gelu, stream);
    return run_tiled(d, k == TG_KERNEL_TILED_TMA, a, b, bi, c, (int)M, (int)N, (int)K, gelu, stream, 0, 0,
                     kernel == TG_KERNEL_AUTO ? 0 : split_k);
}

tg_status tg_gemm(const void* A, const void* B, const void* bias, void* C, int64_t M, int64_t N, int64_t K,
                  int epilogue, tg_stream_t stream) {
    return tg_gemm_ex(A, B, bias, C, M, N, K, epilogue, TG_KERNEL_AUTO, 0, stream);
}

tg_status tg_gemm_plan(const void* A, const void* B, int64_t M, int64_t N, int64_t K, int* kernel, int* split_k,
                       int* aligned_copy) {
    t_last_error.clear();
    const int64_t kMax = 0x7FFFFFFFll;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                    (long long)N, (long long)K);
    if (kernel == nullptr || split_k == nullptr) return fail(TG_ERR_INVALID_ARG, "kernel or split_k is NULL");
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    const bool tma_ok = K % 8 == 0 && N % 8 == 0 && aligned(A, 16) && aligned(B, 16);
    const Plan p = plan_auto(g_dev[dev], M, N, K, tma_ok);
    *kernel = p.kernel;
    *split_k = p.splits;
    if (aligned_copy) *aligned_copy = p.copy ? 1 : 0;
    return TG_OK;
}

tg_status tg_gemm_staged(const void* hA, const void* hB, const void* hbias, void* hC, void* dA, void* dB, void* dbias,
                         void* dC, int64_t M, int64_t N, int64_t K, int epilogue, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if ((hbias == nullptr) != (dbias == nullptr))
        return fail(TG_ERR_INVALID_ARG, "hbias and dbias must both be NULL or both be set");
    if (M < 0 || N < 0 || K < 0) return fail(TG_ERR_INVALID_ARG, "negative size");
    if (M > 0 && N > 0 && (hC == nullptr || dC == nullptr)) return fail(TG_ERR_INVALID_ARG, "C buffer is NULL");
    if (M > 0 && N > 0 && K > 0 && (!hA || !hB || !dA || !dB)) return fail(TG_ERR_INVALID_ARG, "A or B buffer is NULL");
    cudaError_t e;
    if (M > 0 && N > 0 && K > 0) {
        if ((e = cudaMemcpyAsync(dA, hA, M * K * 2, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
            return cuda_fail(e, "copy A to device");
        if ((e = cudaMemcpyAsync(dB, hB, K * N * 2, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
            return cuda_fail(e, "copy B to device");
    }
    if (hbias && N > 0 && (e = cudaMemcpyAsync(dbias, hbias, N * 2, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        return cuda_fail(e, "copy bias to device");
    tg_status st = tg_gemm(dA, dB, dbias, dC, M, N, K, epilogue, stream_);
    if (st != TG_OK) return st;
    if (M > 0 && N > 0 && (e = cudaMemcpyAsync(hC, dC, M * N * 2, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
        return cuda_fail(e, "copy C to host");
    return TG_OK;
}

tg_status tg_device_status(tg_stream_t stream_, int* where) {
    t_last_error.clear();
    if (where) *where = 0;
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    if ((e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof v)) != cudaSuccess)
        return cuda_fail(e, "read status word");
    if (v == 0) return TG_OK;
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero)) != cudaSuccess)
        return cuda_fail(e, "clear status word");
    // a CTA of the 4-bit kernel that gave up may have left arrival counters non-zero
    for (auto& kv : g_dev[dev].scratch)
        if (kv.second.counters) cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(unsigned int));
    cudaDeviceSynchronize();
    if (where) *where = v;
    if (v == kSiteBounds) return fail(TG_ERR_BOUNDS, "a device-side bounds check failed (debug build)");
    return fail(TG_ERR_TIMEOUT, "a kernel wait expired (site %d)", v);
}

tg_status tg_debug_bounds_limit(int64_t floats) {
    if (floats < 0) return fail(TG_ERR_INVALID_ARG, "the limit must be >= 0, got %lld", (long long)floats);
    g_bounds_limit.store(floats);
    return TG_OK;
}

int tg_debug_build(void) { return TG_DEBUG ? 1 : 0; }

tg_status tg_debug_status(tg_stream_t stream) { return tg_device_status(stream, nullptr); }

tg_status tg_bias_gelu(void* C, const void* bias, int64_t M, int64_t N, int epilogue, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_GELU)
        return fail(TG_ERR_INVALID_ARG, "epilogue must be TG_EPI_NONE (0) or TG_EPI_GELU (1), got %d", epilogue);
    if (M < 0 || N < 0 || M > 0x7FFFFFFFll || N > 0x7FFFFFFFll)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld", (long long)M, (long long)N);
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr) return fail(TG_ERR_INVALID_ARG, "C is NULL");
    if (overlaps(C, M * N * 2, bias, bias ? N * 2 : 0)) return fail(TG_ERR_INVALID_ARG, "C overlaps bias");
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    const bool vec8 = N % 8 == 0 && aligned(C, 16) && (bias == nullptr || aligned(bias, 16));
    cudaError_t e = launch_bias_gelu(static_cast<__half*>(C), static_cast<const __half*>(bias), M, N,
                                     epilogue == TG_EPI_GELU ? 1 : 0, vec8, g_dev[dev].sm_count, stream);
    return e == cudaSuccess ? TG_OK : cuda_fail(e, "epilogue kernel launch");
}

tg_status tg_set_watchdog_ns(uint64_t ns) {
    g_watchdog_ns.store(ns == 0 ? 2000000000ull : ns);
    return TG_OK;
}

tg_status tg_debug_skip_first_arrive(int on) {
    g_skip_first_arrive.store(on ? 1 : 0);
    return TG_OK;
}

const char* tg_status_string(int s) {
    switch (s) {
        case TG_OK: return "TG_OK";
        case TG_ERR_INVALID_ARG: return "TG_ERR_INVALID_ARG: invalid argument";
        case TG_ERR_UNSUPPORTED_DEVICE: return "TG_ERR_UNSUPPORTED_DEVICE: not a compute capability 10.3 device";
        case TG_ERR_CUDA: return "TG_ERR_CUDA: a CUDA call failed";
        case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT: a kernel wait expired";
        case TG_ERR_NO_MEMORY: return "TG_ERR_NO_MEMORY: scratch allocation failed";
        case TG_ERR_BOUNDS: return "TG_ERR_BOUNDS: a device-side bounds check failed";
        default: return "unknown tg_status";
    }
}

const char* tg_last_error(void) { return t_last_error.c_str(); }

int tg_version(void) { return 10000; }

int64_t tg_ring_bytes(int kernel) {
    switch (kernel) {
        case TG_KERNEL_TILED_TMA:
        case TG_KERNEL_TILED_LSU:
            return static_cast<int64_t>(kStages) * (kBM * kBK + kBK * kBN) * 2;
        case TG_KERNEL_TILED_PAIR:  // per CTA: its 128 rows of A and 128 columns of B, 6 stages
            return static_cast<int64_t>(6) * (kBM * kBK + kBK * (kBN / 2)) * 2;
        case TG_KERNEL_SPLITK:
            return static_cast<int64_t>(split_stages_for(16)) * (16 * kSkBK + kSkBK * kSkBN) * 2;
        default:
            return -1;
    }
}

void tg_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& d : g_dev) {
        for (auto& kv : d.scratch) {
            if (kv.second.ws) cudaFree(kv.second.ws);
            if (kv.second.counters) cudaFree(kv.second.counters);
            if (kv.second.pad) cudaFree(kv.second.pad);
        }
        d.scratch.clear();
        d.ready = false;  // the status word's address is looked up again
    }
    // device addresses and per-context kernel attributes are looked up again on the
    // next call, so the library keeps working after a cudaDeviceReset that follows this
    for (auto& p : g_noalloc_ptr) p = nullptr;
    g_maps.clear();
    ++g_generation;
}

}  // extern "C"

extern "C" tg_status tg_gemm_splitk_noalloc(const void* A, const void* B, const void* bias, void* C, int64_t M,
                                            int64_t N, int64_t K, int epilogue, int split_k, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_GELU)
        return fail(TG_ERR_INVALID_ARG, "epilogue must be TG_EPI_NONE (0) or TG_EPI_GELU (1), got %d", epilogue);
    const int64_t kMax = 0x7FFFFFFFll;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                    (long long)N, (long long)K);
    if (split_k < 0 || split_k > kSkMaxSplits)
        return fail(TG_ERR_INVALID_ARG, "split_k must be 0 (automatic) or 1..%d, got %d", kSkMaxSplits, split_k);
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr) return fail(TG_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || B == nullptr)) return fail(TG_ERR_INVALID_ARG, "A or B is NULL");
    const int64_t c_bytes = M * N * 2;
    if (overlaps(C, c_bytes, A, K > 0 ? M * K * 2 : 0) || overlaps(C, c_bytes, B, K > 0 ? K * N * 2 : 0) ||
        overlaps(C, c_bytes, bias, bias ? N * 2 : 0))
        return fail(TG_ERR_INVALID_ARG, "C overlaps an input");
    if (M > kSkMaxM || (K > 0 && !(K % 8 == 0 && N % 8 == 0 && aligned(A, 16) && aligned(B, 16))))
        return fail(TG_ERR_INVALID_ARG,
                    "tg_gemm_splitk_noalloc needs M <= %d, K %% 8 == 0, N %% 8 == 0 and 16-byte aligned A, B", kSkMaxM);

    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    DeviceState& d = g_dev[dev];
    const int gelu = epilogue == TG_EPI_GELU ? 1 : 0;
    if (K == 0) {
        cudaError_t e = launch_fill(static_cast<const __half*>(bias), static_cast<__half*>(C), M, N, gelu,
                                    d.sm_count, stream);
        return e == cudaSuccess ? TG_OK : cuda_fail(e, "fill kernel launch");
    }
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static split-K scratch)");
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
    }

    // the most K slices whose partials fit in the array beside the reserved area (one slice needs
    // no scratch, so the automatic choice always fits)
    const int m_pad = (static_cast<int>(M) + 15) / 16 * 16;
    const int n_tiles = static_cast<int>((N + kSkBN - 1) / kSkBN);
    const size_t counter_bytes = (static_cast<size_t>(n_tiles) * sizeof(unsigned int) + 255) / 256 * 256;
    const size_t per_split = static_cast<size_t>(N) * m_pad * sizeof(float);
    const size_t room = TG_NOALLOC_SCRATCH_BYTES > counter_bytes ? TG_NOALLOC_SCRATCH_BYTES - counter_bytes : 0;
    const int fit = static_cast<int>(room / per_split < static_cast<size_t>(kSkMaxSplits) ? room / per_split
                                                                                          : kSkMaxSplits);
    SplitArgs a;
    splitk_args(d, static_cast<const __half*>(A), static_cast<const __half*>(B), static_cast<const __half*>(bias),
                static_cast<__half*>(C), static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), gelu, split_k,
                fit < 1 ? 1 : fit, a);
    if (a.splits > 1 && !split_on_chip(a)) {
        const size_t partial_bytes = static_cast<size_t>(a.splits) * per_split;
        if (counter_bytes + partial_bytes > static_cast<size_t>(TG_NOALLOC_SCRATCH_BYTES))
            return fail(TG_ERR_INVALID_ARG,
                        "tg_gemm_splitk_noalloc: %d K slices of a %lld x %lld product need %zu bytes of scratch, "
                        "more than the %zu-byte static scratch (use fewer slices, 0 for automatic, or tg_gemm)",
                        a.splits, (long long)M, (long long)N, counter_bytes + partial_bytes,
                        static_cast<size_t>(TG_NOALLOC_SCRATCH_BYTES));
        // the partials follow the counter area, which the size limit keeps reserved (the
        // reduction kernel that sums them uses no counters); they are written before read
        a.ws = reinterpret_cast<float*>(g_noalloc_ptr[dev] + counter_bytes);
        debug_limits(a.wd, TG_NOALLOC_SCRATCH_BYTES - counter_bytes, 0);
    }
    return splitk_launch(d, a, stream);
}

// ---------------------------------------------------------------------------
// tg_gemm_w4: the skinny GEMM with 4-bit weights.

extern "C" tg_status tg_gemm_w4_kernel(const void* A, const void* Bq, const void* scales, const void* bias,
                                       void* C, int64_t M, int64_t N, int64_t K, int epilogue, int weight_format,
                                       int kernel, int split_k, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_GELU)
        return fail(TG_ERR_INVALID_ARG, "epilogue must be TG_EPI_NONE (0) or TG_EPI_GELU (1), got %d", epilogue);
    if (weight_format != TG_W4_INT4 && weight_format != TG_W4_FP4_E2M1)
        return fail(TG_ERR_INVALID_ARG, "weight_format must be TG_W4_INT4 (0) or TG_W4_FP4_E2M1 (1), got %d",
                    weight_format);
    const int64_t kMax = 0x7FFFFFFFll;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                    (long long)N, (long long)K);
    if (split_k < 0 || split_k > kSkMaxSplits)
        return fail(TG_ERR_INVALID_ARG, "split_k must be 0 (automatic) or 1..%d, got %d", kSkMaxSplits, split_k);
    if (M > kSkMaxM) return fail(TG_ERR_INVALID_ARG, "tg_gemm_w4 needs M <= %d, got %lld", kSkMaxM, (long long)M);
    if (kernel != TG_W4_KERNEL_AUTO && kernel != TG_W4_KERNEL_TMEM && kernel != TG_W4_KERNEL_REG)
        return fail(TG_ERR_INVALID_ARG, "kernel must be TG_W4_KERNEL_AUTO, _TMEM or _REG (0..2), got %d", kernel);
    if (kernel == TG_W4_KERNEL_REG && M > kW4rMaxM)
        return fail(TG_ERR_INVALID_ARG, "TG_W4_KERNEL_REG needs M <= %d, got %lld", kW4rMaxM, (long long)M);
    if (kernel == TG_W4_KERNEL_REG && split_k > 1)
        return fail(TG_ERR_INVALID_ARG, "TG_W4_KERNEL_REG runs one K slice, got split_k=%d", split_k);
    if (K % kW4Group != 0)
        return fail(TG_ERR_INVALID_ARG, "tg_gemm_w4 needs K %% %d == 0, got K=%lld", kW4Group, (long long)K);
    if (N % 8 != 0) return fail(TG_ERR_INVALID_ARG, "tg_gemm_w4 needs N %% 8 == 0, got N=%lld", (long long)N);
    if (M == 0 || N == 0) return TG_OK;
    if (C == nullptr) return fail(TG_ERR_INVALID_ARG, "C is NULL");
    if (K > 0 && (A == nullptr || Bq == nullptr || scales == nullptr))
        return fail(TG_ERR_INVALID_ARG, "A, Bq or scales is NULL");
    if (K > 0 && !(aligned(A, 16) && aligned(Bq, 16) && aligned(scales, 16)))
        return fail(TG_ERR_INVALID_ARG, "tg_gemm_w4 needs 16-byte aligned A, Bq and scales");
    const int64_t c_bytes = M * N * 2;
    if (overlaps(C, c_bytes, A, K > 0 ? M * K * 2 : 0) || overlaps(C, c_bytes, Bq, K > 0 ? N * K / 2 : 0) ||
        overlaps(C, c_bytes, scales, K > 0 ? (K / kW4Group) * N * 2 : 0) ||
        overlaps(C, c_bytes, bias, bias ? N * 2 : 0))
        return fail(TG_ERR_INVALID_ARG, "C overlaps an input");

    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    DeviceState& d = g_dev[dev];
    const int gelu = epilogue == TG_EPI_GELU ? 1 : 0;
    if (K == 0) {
        cudaError_t e = launch_fill(static_cast<const __half*>(bias), static_cast<__half*>(C), M, N, gelu,
                                    d.sm_count, stream);
        return e == cudaSuccess ? TG_OK : cuda_fail(e, "fill kernel launch");
    }

    const bool use_reg = kernel == TG_W4_KERNEL_REG ||
                         (kernel == TG_W4_KERNEL_AUTO && M <= kW4rMaxM && split_k <= 1 &&
                          (N + kW4rCols - 1) / kW4rCols >= d.sm_count);
    if (use_reg) {
        W4rArgs r{};
        r.bias = static_cast<const __half*>(bias);
        r.C = static_cast<__half*>(C);
        r.M = (int)M; r.N = (int)N; r.gelu = gelu; r.fmt = weight_format;
        const int chunk = w4r_chunk();
        r.n_chunks = (int)((K + chunk - 1) / chunk);
        r.wd = watchdog(d);
        CUtensorMap tmW, tmS, tmX;
        if ((st = make_map_u8(&tmW, Bq, K / 2, N, chunk / 2, kW4rCols, chunk / 2 == 128)) != TG_OK) return st;
        if ((st = make_map_scales(&tmS, scales, N, K / kW4Group, kW4rCols, chunk / kW4Group)) != TG_OK) return st;
        if ((st = make_map_x3(&tmX, A, M, K, chunk)) != TG_OK) return st;
        const int grid = (int)((N + kW4rCols - 1) / kW4rCols);
        cudaError_t e = launch_w4r(r, tmW, tmS, tmX, grid, stream);
        return e == cudaSuccess ? TG_OK : cuda_fail(e, "4-bit register kernel launch");
    }

    // at most kW4MaxM rows of A per launch: larger M runs as row blocks (each
    // reading the weights again)
    for (int64_t r0 = 0; r0 < M; r0 += kW4MaxM) {
        const int64_t rows = M - r0 < kW4MaxM ? M - r0 : kW4MaxM;
        W4Args w{};
        SplitArgs& a = w.s;
        a.A = static_cast<const __half*>(A) + r0 * K;
        a.bias = static_cast<const __half*>(bias);
        a.C = static_cast<__half*>(C) + r0 * N;
        a.M = (int)rows; a.N = (int)N; a.K = (int)K; a.gelu = gelu;
        a.m_pad = (a.M + 15) / 16 * 16;
        w4_pipeline(a.m_pad, &a.stages, &w.a_slots, &w.b_slots);
        a.n_tiles = (a.N + kW4BN - 1) / kW4BN;
        a.kb_total = (a.K + kW4BK - 1) / kW4BK;
        int s = split_k > 0 ? split_k : choose_splits(a.n_tiles, a.kb_total, d.sm_count, 2.0, 1.0, 1.0);
        if (s > a.kb_total) s = a.kb_total;
        a.kb_per_split = (a.kb_total + s - 1) / s;
        a.splits = (a.kb_total + a.kb_per_split - 1) / a.kb_per_split;
        a.num_units = a.n_tiles * a.splits;
        a.wd = watchdog(d);
        if (a.splits > 1) {
            Scratch* sc = nullptr;
            st = ensure_scratch(d, stream, static_cast<size_t>(a.splits) * a.N * a.m_pad * sizeof(float),
                                static_cast<size_t>(a.n_tiles), &sc);
            if (st != TG_OK) return st;
            a.ws = sc->ws;
            a.counters = sc->counters;
            debug_limits(a.wd, sc->ws_bytes, sc->n_counters);
        }
        w.Bq = static_cast<const uint8_t*>(Bq);
        w.scales = static_cast<const __half*>(scales);
        w.fmt = weight_format;
        w.c_vec = aligned(a.C, 16) ? 1 : 0;  // N % 8 == 0 is required above
        CUtensorMap tmBq, tmA, tmS;
        if ((st = make_map_u8(&tmBq, Bq, K / 2, N, kW4BK / 2, kW4BN)) != TG_OK) return st;
        if ((st = make_map(&tmA, a.A, K, a.M, 64, a.m_pad)) != TG_OK) return st;
        if ((st = make_map_scales(&tmS, scales, N, K / kW4Group, kW4BN, kW4BK / kW4Group)) != TG_OK) return st;
        const int grid = a.num_units < d.sm_count ? a.num_units : d.sm_count;
        cudaError_t e = launch_w4(w, tmBq, tmA, tmS, grid, stream);
        if (e != cudaSuccess) return cuda_fail(e, "4-bit kernel launch");
    }
    return TG_OK;
}

extern "C" tg_status tg_gemm_w4_ex(const void* A, const void* Bq, const void* scales, const void* bias, void* C,
                                   int64_t M, int64_t N, int64_t K, int epilogue, int weight_format, int split_k,
                                   tg_stream_t stream) {
    return tg_gemm_w4_kernel(A, Bq, scales, bias, C, M, N, K, epilogue, weight_format, TG_W4_KERNEL_AUTO, split_k,
                             stream);
}

extern "C" tg_status tg_gemm_w4(const void* A, const void* Bq, const void* scales, const void* bias, void* C,
                                int64_t M, int64_t N, int64_t K, int epilogue, int split_k, tg_stream_t stream) {
    return tg_gemm_w4_ex(A, Bq, scales, bias, C, M, N, K, epilogue, TG_W4_INT4, split_k, stream);
}

// ---------------------------------------------------------------------------
// tg_attention_fwd: FlashAttention forward on (batch, sequence, head, dim).

// Split the last, partial round of query blocks into key halves (non-causal).
#ifndef TG_ATTN_SPLIT_TAIL
#define TG_ATTN_SPLIT_TAIL 1
#endif
constexpr bool kAttnSplitTail = TG_ATTN_SPLIT_TAIL != 0;

extern "C" tg_status tg_attention_fwd(const void* Q, const void* K, const void* V, void* O, int64_t B, int64_t S,
                                      int64_t H, int64_t D, int causal, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (causal != 0 && causal != 1) return fail(TG_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
    if (B < 0 || S < 0 || H < 0 || D < 0 || B > 0xFFFF || S > 0x7FFFFFFFll || H > 0xFFFF)
        return fail(TG_ERR_INVALID_ARG, "sizes out of range: B=%lld S=%lld H=%lld D=%lld", (long long)B, (long long)S,
                    (long long)H, (long long)D);
    if (D != kAttnD) return fail(TG_ERR_INVALID_ARG, "tg_attention_fwd supports head dimension %d, got %lld", kAttnD,
                                 (long long)D);
    if (B == 0 || S == 0 || H == 0) return TG_OK;
    if (!Q || !K || !V || !O) return fail(TG_ERR_INVALID_ARG, "Q, K, V or O is NULL");
    if (!(aligned(Q, 16) && aligned(K, 16) && aligned(V, 16) && aligned(O, 16)))
        return fail(TG_ERR_INVALID_ARG, "tg_attention_fwd needs 16-byte aligned Q, K, V and O");
    const int64_t bytes = B * S * H * D * 2;
    if (overlaps(O, bytes, Q, bytes) || overlaps(O, bytes, K, bytes) || overlaps(O, bytes, V, bytes))
        return fail(TG_ERR_INVALID_ARG, "O overlaps an input");
    const int64_t n_qt = (S + 127) / 128;
    if (B * H * n_qt > 0x3FFFFFFFll) return fail(TG_ERR_INVALID_ARG, "too many query blocks");

    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    DeviceState& ds = g_dev[dev];
    AttnArgs a{};
    a.O = static_cast<__half*>(O);
    a.S = (int)S; a.H = (int)H; a.causal = causal;
    a.n_qt = (int)n_qt;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(D)));
    a.wd = watchdog(ds);
    // Query blocks run two per SM. Without the mask every block costs the same, so when the
    // last round is at most half full its blocks are split into key halves (two CTAs each),
    // which fills that round and halves its length.
    const int64_t n_blocks = B * H * n_qt;
    const int64_t slots = 2LL * ds.sm_count;
    const int64_t rest = n_blocks % slots;
    a.n_plain = static_cast<int>(n_blocks);
    if (kAttnSplitTail && !causal && n_blocks >= slots && rest > 0 && 2 * rest <= slots && (S + 127) / 128 >= 2) {
        Scratch* sc = nullptr;
        st = ensure_scratch(ds, stream, static_cast<size_t>(rest) * 2 * attn_part_floats() * sizeof(float),
                            static_cast<size_t>(rest), &sc);
        if (st != TG_OK) return st;
        a.n_plain = static_cast<int>(n_blocks - rest);
        a.n_split = static_cast<int>(rest);
        a.ws = sc->ws;
        a.counters = sc->counters;
        debug_limits(a.wd, sc->ws_bytes, sc->n_counters);
    }
    CUtensorMap tmQ, tmK, tmV;
    if ((st = make_map_bshd(&tmQ, Q, B, S, H, D)) != TG_OK) return st;
    if ((st = make_map_bshd(&tmK, K, B, S, H, D)) != TG_OK) return st;
    if ((st = make_map_bshd(&tmV, V, B, S, H, D)) != TG_OK) return st;
    cudaError_t e = launch_attn(a, tmQ, tmK, tmV, a.n_plain + 2 * a.n_split, stream);
    if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
    return TG_OK;
}

// ---------------------------------------------------------------------------
// tg_softmax_rows: row softmax of an M x N fp16 matrix.

extern "C" tg_status tg_softmax_rows(const void* X, void* Y, int64_t M, int64_t N, tg_stream_t stream_) {
    t_last_error.clear();
    const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (M < 0 || N < 0 || M > 0x7FFFFFFFll || N > 0x7FFFFFFFll)
        return fail(TG_ERR_INVALID_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld", (long long)M, (long long)N);
    if (M == 0 || N == 0) return TG_OK;
    if (!X || !Y) return fail(TG_ERR_INVALID_ARG, "X or Y is NULL");
    if (X != Y && overlaps(Y, M * N * 2, X, M * N * 2))
        return fail(TG_ERR_INVALID_ARG, "Y overlaps X without being the same buffer");
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    tg_status st = current_device(&dev);
    if (st != TG_OK) return st;
    const bool vec = N % 8 == 0 && aligned(X, 16) && aligned(Y, 16);
    cudaError_t e = launch_softmax(static_cast<const __half*>(X), static_cast<__half*>(Y), (int)M, (int)N, vec,
                                   g_dev[dev].sm_count, stream);
    return e == cudaSuccess ? TG_OK : cuda_fail(e, "softmax kernel launch");
}
