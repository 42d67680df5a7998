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
#include <mutex>

#include "pi_ffn.h"
#include "pi_internal.h"

using namespace pi;

static __device__ __align__(256) unsigned char g_noalloc_scratch[PI_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;

// The array's device address, looked up once per device and context. Host code cannot use the
// array's name as a device address (it names a host-side stand-in), so the runtime is asked,
// with the device current. The entry is refreshed when the device's context changes (after a
// cudaDeviceReset the module is loaded again, possibly elsewhere). A mutex makes concurrent
// first calls from several host threads safe.
struct ScratchSlot {
    unsigned long long ctx = 0;   // context id the address belongs to (0: unknown)
    void *ptr = nullptr;
};
ScratchSlot g_slots[MAX_DEVICES];
std::mutex g_slots_mu;

typedef CUresult (*CtxCurrentFn)(CUcontext *);
typedef CUresult (*CtxIdFn)(CUcontext, unsigned long long *);

void *driver_entry(const char *name)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

// Unique id of the calling thread's current context, 0 if the driver cannot say.
unsigned long long current_ctx_id()
{
    static CtxCurrentFn get_cur = (CtxCurrentFn)driver_entry("cuCtxGetCurrent");
    static CtxIdFn get_id = (CtxIdFn)driver_entry("cuCtxGetId");
    if (!get_cur || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

pi_status_t scratch_for(int dev, void **out)
{
    if (dev < 0 || dev >= MAX_DEVICES) return PI_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_slots_mu);
    ScratchSlot &slot = g_slots[dev];
    const unsigned long long id = current_ctx_id();
    if (slot.ptr && id != 0 && slot.ctx == id) {
        *out = slot.ptr;
        return PI_OK;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return PI_ERR_CUDA;
    }
    slot.ptr = p;
    slot.ctx = current_ctx_id();   // the lookup above created the context if there was none
    *out = p;
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
    const bool int4 = D.wdtype == PI_INT4_G128;
    // the same checks as a handle's: every byte the kernels touch lies inside its allocation
    if ((s = check_layer(D, *layer, dev, false))) return s;
    const size_t vec = (size_t)B * D.d * 4;
    if ((s = check_ptr(u, vec, 16, dev)) || (s = check_ptr(y, vec, 16, dev))) return s;
    if ((s = check_ptr(idx, 4, 4, dev)) || (s = check_ptr(count, 4, 4, dev))) return s;   // idx: *count entries, checked on the device
    if (status && (s = check_ptr(status, 4, 4, dev))) return s;

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
    const int bt = pick_bt(B, D.d), btd = pick_bt(B, 1, int4 ? 2 : 8);   // the tiles pi_sparse_ffn picks
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
