// pi_order.cu -- offline hot-first neuron order (sm_103a).
//
// "PowerInfer" paper walk-through page, section "offline profiling" (code
// block): count how often each FFN neuron is non-zero over calibration text,
// then sort neuron ids by that count, largest first. The sort there is Python's
// sorted(), which is stable, so equal counts keep their original order. The
// order is used here only to make frequently active rows contiguous in HBM.
#include "pi_common.cuh"
#include "pi_internal.h"

namespace pi {

// position of neuron i = #{j : c_j > c_i} + #{j < i : c_j == c_i}; perm[position] = i.
// O(f^2) comparisons, tiled through shared memory; an offline step.
__global__ void __launch_bounds__(NT) k_hot_first(const uint32_t *__restrict__ counts, int f, int32_t *__restrict__ perm)
{
    constexpr int TILE = 2048;
    __shared__ uint32_t tile[TILE];
    const int i = blockIdx.x * NT + threadIdx.x;
    const uint32_t ci = i < f ? counts[i] : 0u;
    int pos = 0;
    for (int t0 = 0; t0 < f; t0 += TILE) {
        const int tn = min(TILE, f - t0);
        __syncthreads();
        for (int k = threadIdx.x; k < tn; k += NT) tile[k] = counts[t0 + k];
        __syncthreads();
        for (int k = 0; k < tn; ++k) {
            const uint32_t cj = tile[k];
            pos += (cj > ci) | ((cj == ci) & (t0 + k < i));
        }
    }
    if (i < f) perm[pos] = i;
}

// dst row k = src row perm[k]; one CTA per row (grid-strided).
__global__ void __launch_bounds__(NT) k_permute_rows(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                                     const int32_t *__restrict__ perm, int64_t rows,
                                                     int64_t row_bytes, int32_t *__restrict__ err, int vec16)
{
    for (int64_t k = blockIdx.x; k < rows; k += gridDim.x) {
        const int64_t s = perm[k];
        if (s < 0 || s >= rows) {
            if (threadIdx.x == 0 && err) atomicAdd(err, 1);
            continue;
        }
        const uint8_t *a = src + s * row_bytes;
        uint8_t *b = dst + k * row_bytes;
        if (vec16) {
            const int64_t n16 = row_bytes / 16;
            for (int64_t t = threadIdx.x; t < n16; t += NT)
                reinterpret_cast<uint4 *>(b)[t] = reinterpret_cast<const uint4 *>(a)[t];
        } else {
            for (int64_t t = threadIdx.x; t < row_bytes; t += NT) b[t] = a[t];
        }
    }
}

cudaError_t launch_hot_first(const uint32_t *counts, int f, int32_t *perm, cudaStream_t s)
{
    if (f <= 0) return cudaSuccess;
    k_hot_first<<<(f + NT - 1) / NT, NT, 0, s>>>(counts, f, perm);
    return cudaGetLastError();
}

cudaError_t launch_permute_rows(const void *src, void *dst, const int32_t *perm, int64_t rows, int64_t row_bytes,
                                int32_t *err, cudaStream_t s)
{
    if (rows <= 0 || row_bytes <= 0) return cudaSuccess;
    const int vec16 = (row_bytes % 16 == 0) && ((uintptr_t)src % 16 == 0) && ((uintptr_t)dst % 16 == 0);
    const int64_t grid = rows < 65535 * 8 ? rows : 65535 * 8;
    k_permute_rows<<<(unsigned)grid, NT, 0, s>>>((const uint8_t *)src, (uint8_t *)dst, perm, rows, row_bytes, err, vec16);
    return cudaGetLastError();
}

}  // namespace pi
