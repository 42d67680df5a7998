// pi_selftest.cu -- failure detection of the bounded grid barrier, without a GPU fault.
//
// A tiny cooperative grid meets at the same barrier the decode-step kernel uses,
// told to expect `extra` more CTAs than it has. With extra > 0 nobody can complete
// it: every CTA gives up after the barrier's time limit, records PI_ERR_TIMEOUT and
// returns, and the context stays usable.
#include "pi_async.cuh"
#include "pi_ffn.h"

using namespace pi;

static __global__ void k_barrier_selftest(unsigned *work, unsigned expected, uint32_t *status)
{
    __shared__ int s_flag;
    unsigned long long *cnt = reinterpret_cast<unsigned long long *>(work);
    __shared__ unsigned long long base;
    if (threadIdx.x == 0) base = barrier_base(cnt, expected);
    __syncthreads();
    if (grid_sync_to(cnt, base + expected, status, &s_flag) && threadIdx.x == 0) atomicAdd(work + 2, 1u);
}

extern "C" pi_status_t pi_selftest_grid_barrier(uint32_t *work, int32_t extra, void *stream)
{
    if (!work || ((uintptr_t)work % 8) || extra < 0 || extra > 1024) return PI_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, work) != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return PI_ERR_INVALID_ARG;
    constexpr unsigned GRID = 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(GRID);
    cfg.blockDim = dim3(32);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_barrier_selftest, (unsigned *)work, GRID + (unsigned)extra, work + 3);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_CUDA;
    }
    return PI_OK;
}

// ---------------------------------------------------------------- tensor-core tile check ----
//
// One CTA stages A and B in the 128-byte-swizzled shared-memory layouts the sparse-FFN
// tensor-core kernels use, runs the tcgen05 products, and writes D = A * B^T out of
// tensor memory. mode 0: A [128 x K] staged K-major. mode 1: A given as its transpose
// [K x 128] and staged MN-major. B [N x K] staged K-major.
#include "pi_umma.cuh"

namespace {

constexpr int UT_SLACK = 16384;   // bytes past the operands, so every descriptor reading stays in the buffer

__global__ void __launch_bounds__(128) k_umma_selftest(const uint4 *__restrict__ A, const uint4 *__restrict__ Bm,
                                                       float *__restrict__ D, int mode, int N, int K, int bf16,
                                                       uint32_t *status)
{
    extern __shared__ uint8_t dsm[];
    __shared__ uint64_t bar;
    __shared__ uint32_t taddr_s;
    const uint32_t base = (smem_u32(dsm) + 1023u) & ~1023u;
    uint8_t *gbase = dsm + (base - smem_u32(dsm));
    const int kbs = K / 64;
    const uint32_t a_bytes = (uint32_t)kbs * 16384u, b_blk = (uint32_t)(N / 8) * 1024u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ncols = N <= 32 ? 32u : (uint32_t)N;

    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&taddr_s, ncols);
    // operands -> shared memory (generic stores, then a proxy fence for the tensor core)
    for (int t = threadIdx.x; t < 128 * K / 8; t += blockDim.x) {
        uint32_t off;
        if (mode == 0) {   // A row m, chunk q of K
            const int m = t / (K / 8), q = t % (K / 8);
            off = (uint32_t)(q / 8) * 16384u + sw128_off(m, q % 8);
        } else {           // A^T row k, chunk q of M
            const int k = t / 16, q = t % 16;
            off = (uint32_t)(k / 64) * 16384u + (uint32_t)(q / 8) * 8192u + sw128_off(k % 64, q % 8);
        }
        *reinterpret_cast<uint4 *>(gbase + off) = A[t];
    }
    for (int t = threadIdx.x; t < N * K / 8; t += blockDim.x) {
        const int n = t / (K / 8), q = t % (K / 8);
        *reinterpret_cast<uint4 *>(gbase + a_bytes + (uint32_t)(q / 8) * b_blk + sw128_off(n, q % 8)) = Bm[t];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = taddr_s;
    if (threadIdx.x == 0) {
        const uint32_t idesc = f16_idesc(bf16, mode, 0, 128, N);
        for (int kb = 0; kb < kbs; ++kb)
            for (int j = 0; j < 4; ++j) {
                const uint64_t ad = mode == 0 ? sw128_desc(base + kb * 16384u + j * 32u, 16u, 1024u)
                                              : sw128_desc(base + kb * 16384u + j * 2048u, 8192u, 1024u);
                const uint64_t bd = sw128_desc(base + a_bytes + kb * b_blk + j * 32u, 16u, 1024u);
                umma_f16(tmem, ad, bd, idesc, (kb | j) != 0);
            }
        umma_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar, 0);
    if (!ok && lane == 0) set_status(status, ST_TIMEOUT);
    tc_fence_after();
    if (ok) {
        for (int c = 0; c < N; c += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, v);
            const int m = 32 * warp + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[(size_t)m * N + c + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

}  // namespace

extern "C" pi_status_t pi_selftest_umma(const void *a, const void *b, float *d, int32_t mode, int32_t n, int32_t k,
                                        int32_t dtype, uint32_t *status, void *stream)
{
    if (!a || !b || !d || !status || (mode != 0 && mode != 1) || (dtype != PI_BF16 && dtype != PI_F16))
        return PI_ERR_INVALID_ARG;
    if ((n != 16 && n != 32 && n != 64 && n != 128) || (k != 64 && k != 128)) return PI_ERR_INVALID_ARG;
    if (((uintptr_t)a | (uintptr_t)b | (uintptr_t)d) % 16 || (uintptr_t)status % 4) return PI_ERR_INVALID_ARG;
    const void *ptrs[4] = {a, b, d, status};
    for (const void *p : ptrs) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();
            return PI_ERR_INVALID_ARG;
        }
        if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return PI_ERR_INVALID_ARG;
    }
    const size_t smem = 1024 + (size_t)k / 64 * 16384 + (size_t)k / 64 * (n / 8) * 1024 + UT_SLACK;
    if (cudaFuncSetAttribute(k_umma_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_CUDA;
    }
    k_umma_selftest<<<1, 128, smem, (cudaStream_t)stream>>>((const uint4 *)a, (const uint4 *)b, d, mode, n, k,
                                                             dtype == PI_BF16 ? 1 : 0, status);
    if (cudaGetLastError() != cudaSuccess) return PI_ERR_CUDA;
    return PI_OK;
}
