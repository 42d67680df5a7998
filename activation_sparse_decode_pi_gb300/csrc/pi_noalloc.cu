// pi_noalloc.cu -- neuron-sparse FFN of one layer for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: for example, code running inside a
// host-side allocator callback, a plugin whose host process owns every device
// allocation, or a runtime that forbids allocation after start-up. They cannot
// create a pi_ffn_t handle, because pi_ffn_create allocates its workspace.
// pi_sparse_ffn_noalloc runs the same three kernels as pi_sparse_ffn (gate/up
// gather, W_down axpy, fixed-order reduction) with their scratch memory (the
// h values and the fp32 partial sums) in the file-scope device array below, so
// the call itself allocates nothing.
//
// The array is part of this library's device code: every GPU that loads the
// library holds its PI_NOALLOC_SCRATCH_BYTES until the process exits. All calls
// share it, and it keeps the previous call's contents. This path never needs it
// to start at zero (every entry it reads is written earlier in the same call),
// but two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pi_ffn.h"
#include "pi_internal.h"

using namespace pi;

static __device__ __align__(256) unsigned char g_noalloc_scratch[PI_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
void *g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device. Host code cannot
// use the array's name as a device address; it asks the runtime once per device.
pi_status_t scratch_for(int dev, void **out)
{
    if (dev < 0 || dev >= MAX_DEVICES) return PI_ERR_UNSUPPORTED;
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return PI_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PI_OK;
}

pi_status_t check_dev_ptr(const void *p, size_t align, int dev)
{
    if (!p || ((uintptr_t)p % align) != 0) return PI_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return PI_ERR_INVALID_ARG;
    if (a.type == cudaMemoryTypeDevice && a.device != dev) return PI_ERR_INVALID_ARG;
    return PI_OK;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

extern "C" pi_status_t pi_sparse_ffn_noalloc(const pi_ffn_desc_t *desc, const pi_layer_weights_t *layer,
                                              const float *u, int32_t B, const int32_t *idx, const int32_t *count,
                                              float *y, int32_t *status, void *stream)
{
    if (!desc || !layer || B < 1) return PI_ERR_INVALID_ARG;
    const pi_ffn_desc_t &D = *desc;
    if (D.d < 8 || D.d % 8 || D.f < 1 || D.r < 8 || D.r % 8) return PI_ERR_INVALID_ARG;
    if (D.kind != PI_FFN_GATED_RELU && D.kind != PI_FFN_RELU) return PI_ERR_INVALID_ARG;
    if (D.wdtype < PI_F32 || D.wdtype > PI_INT4_G128) return PI_ERR_INVALID_ARG;
    if (D.wdtype == PI_INT4_G128 && D.d % 128) return PI_ERR_UNSUPPORTED;
    if ((size_t)D.d * 4 > SMEM_VEC_CAP) return PI_ERR_UNSUPPORTED;

    // scratch: h [B x f] fp32, then the partial sums [MAX_GROUPS x B x d] fp32
    const size_t h_bytes = align256((size_t)B * D.f * 4);
    const size_t part_bytes = (size_t)MAX_GROUPS * B * D.d * 4;
    if (h_bytes + part_bytes > PI_NOALLOC_SCRATCH_BYTES) return PI_ERR_UNSUPPORTED;

    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_CUDA;
    }
    pi_status_t s;
    const bool gated = D.kind == PI_FFN_GATED_RELU, int4 = D.wdtype == PI_INT4_G128;
    if ((s = check_dev_ptr(layer->w_gate, 16, dev))) return s;
    if ((s = check_dev_ptr(layer->w_down_t, 16, dev))) return s;
    if (gated && (s = check_dev_ptr(layer->w_up, 16, dev))) return s;
    if (int4 && ((s = check_dev_ptr(layer->s_gate, 2, dev)) || (s = check_dev_ptr(layer->s_down, 2, dev)) ||
                 (gated && (s = check_dev_ptr(layer->s_up, 2, dev)))))
        return s;
    if (layer->b_gate && (s = check_dev_ptr(layer->b_gate, 4, dev))) return s;
    if ((s = check_dev_ptr(u, 16, dev)) || (s = check_dev_ptr(idx, 4, dev)) || (s = check_dev_ptr(count, 4, dev)) ||
        (s = check_dev_ptr(y, 16, dev)))
        return s;
    if (status && (s = check_dev_ptr(status, 4, dev))) return s;

    void *scratch = nullptr;
    if ((s = scratch_for(dev, &scratch))) return s;
    float *hbuf = (float *)scratch;
    float *part = (float *)((char *)scratch + h_bytes);

    cudaStream_t st = (cudaStream_t)stream;
    auto mk = [&](dim3 grid, size_t smem, bool pdl) {
        Launch L;
        L.grid = grid;
        L.block = dim3(NT);
        L.smem = smem;
        L.stream = st;
        L.pdl = pdl;
        L.nsm = nsm;
        return L;
    };
    int bt = 1;
    while (bt * 2 <= 8 && (size_t)bt * 2 * D.d * 4 <= SMEM_VEC_CAP && bt < B) bt *= 2;
    int btd = 1;
    while (btd * 2 <= (int4 ? 2 : 8) && btd < B) btd *= 2;
    uint32_t *st_word = (uint32_t *)status;
    cudaError_t e = launch_ffn_h(mk(dim3(0), (size_t)bt * D.d * 4, false), D.wdtype, D.kind, bt, layer->w_gate,
                                 layer->w_up, layer->s_gate, layer->s_up, layer->b_gate, D.d, D.f, u, nullptr, B, idx,
                                 count, hbuf, D.f, st_word);
    if (e == cudaSuccess)
        e = launch_ffn_down(mk(dim3(0), 0, true), D.wdtype, btd, layer->w_down_t, layer->s_down, D.d, D.f, idx, count,
                            hbuf, D.f, B, part, st_word);
    if (e == cudaSuccess)
        e = launch_reduce(mk(dim3((D.d + RED_COLS - 1) / RED_COLS, B), 0, true), part, D.d, B, D.f, count, nullptr,
                          y, nullptr, nullptr, nullptr, 0.f);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_CUDA;
    }
    return PI_OK;
}
