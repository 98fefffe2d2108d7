// The epilogue on its own: C = epi(C + bias) in place on a binary16 matrix.
//
// This is the unfused comparator for the fused epilogue of "Designing
// high-performance GPU kernels with TileLang ...", section 3 (GELU(MatMul +
// Bias) applied while the product is on chip): a GEMM that writes its
// product to HBM followed by this pass, which reads it back, adds the bias,
// applies GELU and writes it again. Unlike the fused path the product is
// rounded to binary16 before the bias and GELU are applied. HBM-bound: 2 bytes
// read and 2 written per element (plus the bias, read from L2).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

// 8 elements (16 bytes) per step; rows are 16-byte aligned (N % 8 == 0, C aligned).
__global__ void bias_gelu_vec8_kernel(__half* __restrict__ C, const __half* __restrict__ bias, int64_t M, int64_t N,
                                      int gelu) {
    const int64_t per_row = N / 8;
    const int64_t total = M * per_row;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total; u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = u / per_row;
        const int64_t c0 = (u - row * per_row) * 8;
        uint4* p = reinterpret_cast<uint4*>(C + row * N + c0);
        uint4 x = *p;
        __half2* h = reinterpret_cast<__half2*>(&x);
        uint4 bv = make_uint4(0, 0, 0, 0);
        if (bias) bv = __ldg(reinterpret_cast<const uint4*>(bias + c0));
        const __half2* hb = reinterpret_cast<const __half2*>(&bv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(h[e]);
            const float2 g = bias ? __half22float2(hb[e]) : make_float2(0.0f, 0.0f);
            h[e] = __floats2half2_rn(epi_value(f.x, g.x, gelu), epi_value(f.y, g.y, gelu));
        }
        *p = x;
    }
}

// Any shape and alignment: one element per step.
__global__ void bias_gelu_scalar_kernel(__half* __restrict__ C, const __half* __restrict__ bias, int64_t M, int64_t N,
                                        int gelu) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = i % N;
        const float b = bias ? __half2float(bias[j]) : 0.0f;
        C[i] = __float2half_rn(epi_value(__half2float(C[i]), b, gelu));
    }
}

}  // namespace

cudaError_t launch_bias_gelu(__half* C, const __half* bias, int64_t M, int64_t N, int gelu, bool vec8, int sm_count,
                             cudaStream_t stream) {
    const int64_t units = vec8 ? M * (N / 8) : M * N;
    int64_t blocks = (units + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 16;  // enough loads in flight for HBM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (vec8)
        bias_gelu_vec8_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(C, bias, M, N, gelu);
    else
        bias_gelu_scalar_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(C, bias, M, N, gelu);
    return cudaGetLastError();
}

}  // namespace tg
