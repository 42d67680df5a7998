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
