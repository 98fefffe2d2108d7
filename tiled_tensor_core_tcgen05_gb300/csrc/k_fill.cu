// K == 0: every sum over k is empty, so C[i,j] = epi(bias[j]) (epi(0) without
// bias) -- the definition C[i,j] = sum_k A[i,k] B[k,j] of "TileLang: writing
// LLM GPU kernels by thinking in tiles", section 2, with an empty k range.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

__global__ void fill_kernel(const __half* __restrict__ bias, __half* __restrict__ C, int64_t M, int64_t N,
                            int gelu) {
    const int64_t total = M * N;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx % N;
        const float b = bias ? __half2float(bias[j]) : 0.0f;
        C[idx] = __float2half_rn(epi_value(0.0f, b, gelu));
    }
}

}  // namespace

cudaError_t launch_fill(const __half* bias, __half* C, int64_t M, int64_t N, int gelu, int sm_count,
                        cudaStream_t stream) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    fill_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(bias, C, M, N, gelu);
    return cudaGetLastError();
}

}  // namespace tg
