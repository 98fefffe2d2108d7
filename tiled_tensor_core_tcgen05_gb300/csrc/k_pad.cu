// Copy of a row-major fp16 matrix into a buffer whose row stride is a multiple
// of 8 elements (16 bytes) at a 16-byte-aligned base, so that a tensor map can
// describe it. Only the `cols` columns of each row are written; the tensor map
// keeps the logical extent `cols`, so the loads read the padding as
// out-of-range (zero) and never its contents.
#include "tg_internal.h"

namespace tg {
namespace {

// 4-byte words: source rows start 4-byte aligned (even `cols`, 4-byte aligned base)
__global__ void pad_rows_u32(const uint32_t* __restrict__ src, uint32_t* __restrict__ dst, int64_t rows,
                             int64_t words, int64_t dst_words) {
    const int64_t total = rows * words;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / words, w = i - r * words;
        dst[r * dst_words + w] = src[i];
    }
}

__global__ void pad_rows_u16(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t rows,
                             int64_t cols, int64_t dst_ld) {
    const int64_t total = rows * cols;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols, c = i - r * cols;
        dst[r * dst_ld + c] = src[i];
    }
}

}  // namespace

cudaError_t launch_pad_rows(const __half* src, __half* dst, int64_t rows, int64_t cols, int64_t dst_ld,
                            int sm_count, cudaStream_t stream) {
    const bool words = cols % 2 == 0 && (reinterpret_cast<uintptr_t>(src) & 3) == 0;
    const int64_t units = words ? rows * (cols / 2) : rows * cols;
    int64_t blocks = (units + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (words)
        pad_rows_u32<<<static_cast<int>(blocks), 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(src),
                                                                   reinterpret_cast<uint32_t*>(dst), rows, cols / 2,
                                                                   dst_ld / 2);
    else
        pad_rows_u16<<<static_cast<int>(blocks), 256, 0, stream>>>(reinterpret_cast<const uint16_t*>(src),
                                                                   reinterpret_cast<uint16_t*>(dst), rows, cols, dst_ld);
    return cudaGetLastError();
}

}  // namespace tg
