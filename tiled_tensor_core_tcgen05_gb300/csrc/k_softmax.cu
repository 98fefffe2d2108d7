// Row softmax: Y[i, :] = exp(X[i, :] - max X[i, :]) / sum exp(X[i, :] - max X[i, :])
// on M x N fp16, computed in fp32, rounded once to fp16.
//
// "Designing high-performance GPU kernels with TileLang ..." (section 4,
// "Advanced Reductions and Softmax") describes the operation as two
// reductions over each row, the maximum (for numerical stability) and the sum
// of exponentials, kept in registers and shared memory; the same page's
// benchmark section puts such kernels at HBM bandwidth. Each row is read from
// HBM once and written once:
//   - softmax_rows_reg: a group of TPR threads holds the whole row in
//     registers as packed fp16 (16-byte loads, lane-interleaved so a warp's
//     loads are contiguous), reduces the maximum and the sum with warp
//     shuffles (and shared memory across the group's warps), computes each
//     exponential once in fp32 and keeps it as fp16 in place of its input,
//     then writes the row with 16-byte stores. Rows must start 16-byte
//     aligned (N % 8 == 0, aligned X and Y) and N <= TPR * VEC * 8.
//   - softmax_rows_2pass: any N and alignment; one block per row; the
//     maximum and the sum in one pass (a running pair per thread), then the
//     write pass over the row again, from L2.
// Exponentials are base 2: exp(x - m) = 2^((x - m) log2e), with x - m exact in
// fp32 for fp16 inputs.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBlock = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Reduce v over the TPR threads of one row group. Warps of a group combine
// through red[] (one slot per warp of the block); every thread of the block
// calls this the same number of times (the barriers are block-wide).
template <int TPR, bool kMax>
__device__ __forceinline__ float group_reduce(float v, float* red) {
    v = kMax ? warp_max(v) : warp_sum(v);
    if constexpr (TPR > 32) {
        constexpr int kWarps = TPR / 32;
        const int warp = threadIdx.x >> 5;
        const int first = warp - (warp % kWarps);
        if ((threadIdx.x & 31) == 0) red[warp] = v;
        __syncthreads();
        v = red[first];
#pragma unroll
        for (int i = 1; i < kWarps; ++i) v = kMax ? fmaxf(v, red[first + i]) : v + red[first + i];
        __syncthreads();  // red[] is reused by the next reduction
    }
    return v;
}

template <int TPR, int VEC>
__global__ void __launch_bounds__(TPR > kBlock ? TPR : kBlock)
    softmax_rows_reg(const __half* X, __half* Y, int M, int N) {
    constexpr int kBlockThreads = TPR > kBlock ? TPR : kBlock;
    constexpr int kRowsPerBlock = kBlockThreads / TPR;
    __shared__ float red[kBlockThreads / 32];
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const __half2 kNegInf2 = __halves2half2(__ushort_as_half(0xFC00), __ushort_as_half(0xFC00));
    for (int base = blockIdx.x * kRowsPerBlock; base < M; base += gridDim.x * kRowsPerBlock) {
        const int row = base + g;
        const bool row_ok = row < M;
        const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(row_ok ? row : 0) * N);
        // chunk v of thread t: elements (v * TPR + t) * 8 .. + 7, kept as packed fp16 (2 bytes an
        // element, so more of the row is in flight per SM); padding reads as -inf
        uint4 x[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            if (row_ok && (v * TPR + t) * 8 < N) {
                x[v] = __ldcs(src + v * TPR + t);
            } else {
                const uint32_t ni = *reinterpret_cast<const uint32_t*>(&kNegInf2);
                x[v] = make_uint4(ni, ni, ni, ni);
            }
        }
        __half2 m2 = kNegInf2;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const __half2* h = reinterpret_cast<const __half2*>(&x[v]);
#pragma unroll
            for (int q = 0; q < 4; ++q) m2 = __hmax2(m2, h[q]);
        }
        float mx = fmaxf(__low2float(m2), __high2float(m2));
        mx = group_reduce<TPR, true>(mx, red);
        // exponentials in fp32, summed in fp32, kept as fp16 in place of the inputs
        float sum = 0.0f;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            __half2* h = reinterpret_cast<__half2*>(&x[v]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(h[q]);
                const float p0 = ex2_approx((f.x - mx) * kLog2e);  // x - mx is exact for fp16 inputs
                const float p1 = ex2_approx((f.y - mx) * kLog2e);
                sum += p0 + p1;
                h[q] = __floats2half2_rn(p0, p1);
            }
        }
        sum = group_reduce<TPR, false>(sum, red);
        const float inv = 1.0f / sum;
        uint4* dst = reinterpret_cast<uint4*>(Y + static_cast<int64_t>(row_ok ? row : 0) * N);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            if (row_ok && (v * TPR + t) * 8 < N) {
                __half2* h = reinterpret_cast<__half2*>(&x[v]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h[q]);
                    h[q] = __floats2half2_rn(f.x * inv, f.y * inv);
                }
                __stcs(dst + v * TPR + t, x[v]);
            }
        }
    }
}

// Fold (m, l) = (maximum, sum of exp(x - m)) of one part of a row into another.
__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both parts empty or all -inf so far
    l = l * ex2_approx((m - mn) * kLog2e) + l2 * ex2_approx((m2 - mn) * kLog2e);
    m = mn;
}

__device__ __forceinline__ void online_add(float& m, float& l, float x) {
    if (x == -INFINITY) return;  // contributes exp(-inf) = 0 (and would turn a fresh pair into NaN)
    if (x > m) {
        l = l * ex2_approx((m - x) * kLog2e) + 1.0f;
        m = x;
    } else {
        l += ex2_approx((x - m) * kLog2e);
    }
}

// Any N and alignment: one block per row (grid-stride over rows), two passes
// over the row: the maximum and the sum together (each thread keeps a running
// pair, rescaling its sum when its maximum grows; the block merges the pairs),
// then the write pass, served from L2. 16-byte accesses when vec.
template <bool kVec>
__global__ void __launch_bounds__(kBlock) softmax_rows_2pass(const __half* X, __half* Y, int M, int N) {
    __shared__ float red_m[kBlock / 32], red_l[kBlock / 32];
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        const __half* x = X + static_cast<int64_t>(row) * N;
        __half* y = Y + static_cast<int64_t>(row) * N;
        float m = -INFINITY, l = 0.0f;
        if constexpr (kVec) {
            const uint4* xv = reinterpret_cast<const uint4*>(x);
            for (int j = threadIdx.x; j < N / 8; j += kBlock) {
                const uint4 u = __ldcg(xv + j);
                const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    online_add(m, l, __low2float(h[q]));
                    online_add(m, l, __high2float(h[q]));
                }
            }
        } else {
            for (int j = threadIdx.x; j < N; j += kBlock) online_add(m, l, __half2float(x[j]));
        }
        // merge the pairs: within the warp, then across warps
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
            const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, o);
            online_merge(m, l, m2, l2);
        }
        const int warp = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) {
            red_m[warp] = m;
            red_l[warp] = l;
        }
        __syncthreads();
        m = red_m[0];
        l = red_l[0];
#pragma unroll
        for (int i = 1; i < kBlock / 32; ++i) online_merge(m, l, red_m[i], red_l[i]);
        __syncthreads();
        const float mx = m;
        const float inv = 1.0f / l;
        if constexpr (kVec) {
            const uint4* xv = reinterpret_cast<const uint4*>(x);
            uint4* yv = reinterpret_cast<uint4*>(y);
            for (int j = threadIdx.x; j < N / 8; j += kBlock) {
                uint4 u = __ldcg(xv + j);
                __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 f = __half22float2(h[q]);
                    h[q] = __floats2half2_rn(ex2_approx((f.x - mx) * kLog2e) * inv, ex2_approx((f.y - mx) * kLog2e) * inv);
                }
                __stcs(yv + j, u);
            }
        } else {
            for (int j = threadIdx.x; j < N; j += kBlock)
                y[j] = __float2half_rn(ex2_approx((__half2float(x[j]) - mx) * kLog2e) * inv);
        }
    }
}

template <int TPR, int VEC>
cudaError_t launch_reg(const __half* X, __half* Y, int M, int N, int sm_count, cudaStream_t stream) {
    constexpr int kBlockThreads = TPR > kBlock ? TPR : kBlock;
    constexpr int kRowsPerBlock = kBlockThreads / TPR;
    int64_t blocks = (static_cast<int64_t>(M) + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = static_cast<int64_t>(sm_count) * (2048 / kBlockThreads);
    if (blocks > cap) blocks = cap;
    softmax_rows_reg<TPR, VEC><<<static_cast<int>(blocks), kBlockThreads, 0, stream>>>(X, Y, M, N);
    return cudaGetLastError();
}

}  // namespace

// Register-resident path when the rows are 16-byte aligned and fit, else the
// two-pass path. Row groups of TPR threads hold 8 * VEC elements each: a warp
// per row up to 4096 elements, then 64..512 threads (128 elements each).
cudaError_t launch_softmax(const __half* X, __half* Y, int M, int N, bool vec, int sm_count, cudaStream_t stream) {
    if (vec && N <= 512 * 128) {
        if (N <= 32 * 8) return launch_reg<32, 1>(X, Y, M, N, sm_count, stream);
        if (N <= 32 * 16) return launch_reg<32, 2>(X, Y, M, N, sm_count, stream);
        if (N <= 32 * 32) return launch_reg<32, 4>(X, Y, M, N, sm_count, stream);
        if (N <= 32 * 64) return launch_reg<32, 8>(X, Y, M, N, sm_count, stream);
        if (N <= 32 * 128) return launch_reg<32, 16>(X, Y, M, N, sm_count, stream);
        if (N <= 64 * 128) return launch_reg<64, 16>(X, Y, M, N, sm_count, stream);
        if (N <= 128 * 128) return launch_reg<128, 16>(X, Y, M, N, sm_count, stream);
        if (N <= 256 * 128) return launch_reg<256, 16>(X, Y, M, N, sm_count, stream);
        return launch_reg<512, 16>(X, Y, M, N, sm_count, stream);
    }
    int64_t blocks = M;
    if (blocks > static_cast<int64_t>(sm_count) * 8) blocks = static_cast<int64_t>(sm_count) * 8;
    if (vec)
        softmax_rows_2pass<true><<<static_cast<int>(blocks), kBlock, 0, stream>>>(X, Y, M, N);
    else
        softmax_rows_2pass<false><<<static_cast<int>(blocks), kBlock, 0, stream>>>(X, Y, M, N);
    return cudaGetLastError();
}

}  // namespace tg
