// pi_internal.h -- launchers shared between the host side (pi_api.cu) and the kernel TUs.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <unordered_map>

#include "pi_ffn.h"

namespace pi {

// ---------------------------------------------------------------- host-side validation (pi_api.cu)

// A pointer the kernels may read or write `bytes` bytes at: non-NULL, aligned, device (or
// managed) memory of device `dev`, and, where the driver can say, inside one allocation.
pi_status_t check_ptr(const void *p, size_t bytes, size_t align, int dev);

// Every weight pointer of one layer for its shape: sizes inside their allocations, 16-byte
// aligned rows, NULL exactly where the kind and type say. predictor: also p1_t / p2_t / b_pred.
pi_status_t check_layer(const pi_ffn_desc_t &D, const pi_layer_weights_t &w, int dev, bool predictor);

// Largest batch tile (1, 2, 4 or 8, at most cap) whose fp32 vectors of length K fit the
// shared-memory budget of one staged tile, capped near B.
int pick_bt(int B, int K, int cap = 8);

// Host-side fault injection, read from PI_FAULT at each pi_ffn_create: "alloc" fails the
// workspace allocation (nothing is allocated), "upload" fails after the workspace exists
// (the clean-up path frees it), "badarg" fails descriptor validation.
enum { FAULT_NONE = 0, FAULT_ALLOC = 1, FAULT_UPLOAD = 2, FAULT_BADARG = 3 };
int injected_fault();

// Launch geometry shared by host and kernels.
constexpr int NT = 256;               // threads per CTA of the CUDA-core kernels
constexpr int NW = NT / 32;           // warps per CTA
constexpr int PRED_ROWS_HIDDEN = 4;   // predictor hidden units per CTA (K1)
constexpr int PRED_ROWS_LOGIT = 32;   // logits per CTA = one mask word (K2)
constexpr int RED_COLS = 128;         // output columns per CTA of the partial-sum reduction
constexpr int DOWN_GROUP_MIN = 16;    // smallest group of active neurons per fp32 partial
constexpr int MAX_GROUPS = 256;       // at most this many partials per layer (group size grows with the count)
constexpr size_t SMEM_VEC_CAP = 96 * 1024;  // shared memory for one staged batch tile of input vectors

// Persistent decode-step kernel (batch 1): one CTA of STACK_NT threads per SM.
constexpr int STACK_NT = 512;
constexpr int STACK_SLICE = 32;           // output columns per reduction slice
constexpr int STACK_MAX_CHUNK = 512;      // neurons one CTA may own (f <= 512 * grid)
constexpr int STACK_MAX_SLOTS = 16;       // shared-memory ring slots (one neuron's rows each)
constexpr int STACK_MAX_P1_ROWS = 8;      // predictor hidden units one CTA owns (r <= 8 * SMs)
constexpr int STACK_P2_TILES = 16;        // ring slots for 16-row tiles of owned P2 rows, at most

struct StackLayer {
    const void *wg, *wu, *wd;     // [f x d] gate (W1), up (NULL if non-gated), W_down transposed
    const void *sg, *su, *sd;     // int4 scales or NULL
    const float *bg;              // gate bias or NULL
    const void *p1, *p2;          // predictor [r x d], [f x r]
    const float *bp;              // predictor bias or NULL
};

// Byte stride of the P2 rows the persistent step stages in shared memory: the row plus 16 or
// 32 bytes, so that the stride is an odd number of 16-byte units and eight consecutive rows
// start in eight different bank groups.
__host__ __device__ inline int stack_p2_stride(int row_bytes)
{
    return row_bytes + ((row_bytes >> 4) & 1 ? 32 : 16);
}

struct StackArgs {
    const StackLayer *layers;     // device array [L]
    int L, d, f, r;
    float tau, eps;
    const float *x0;
    float *xa, *xb, *x_out;       // ping-pong layer outputs, final output
    float *hp;                    // [r]
    uint32_t *maskw;              // [L x ceil(f/32)], zeroed by the kernel
    float *part;                  // [grid x d] one fp32 partial per CTA
    float *sumsq;                 // [ceil(d/STACK_SLICE)]
    int32_t *counts, *idx_out;    // optional outputs
    unsigned long long *bar;      // monotonic grid-barrier counter (zeroed at create and after a timeout)
    uint32_t *status;
    int slots, slot_bytes;
    unsigned nblocks;             // CTAs expected at every grid barrier
    long long pf_bytes;           // next-layer predictor bytes to prefetch into L2
    int off_hp, off_scr, off_flags, off_mbar, off_ring;   // dynamic shared-memory layout
    int ring_bytes;               // ring region: the neuron slots
    int bias_bulk;                // gate biases ride in the row copies (every layer has one and f % 4 == 0)
    int hot_k;                    // ring slots per CTA held by hot owned neurons (loaded a layer ahead), <= slots - 2
    int hot_prefix;               // neurons below this are active without a logit
    int p2_tiles;                 // ring slots for 16-row tiles of owned P2 rows (0: none)
    int p2_stage_tiles;           // of which filled between layers, at most (the rest as the logits start)
    int pf_p1;                    // the next layer's P1 rows into L2: 1 during the grid barrier after the FFN, 2 a layer ahead
    int pf_p2;                    // the next layer's unstaged P2 rows into L2 a layer ahead
    int pf_p2_ffn;                // the next layer's unstaged P2 rows into L2 during this layer's FFN, the first pf_p2_frac / 256 of them
    int pf_p2_frac;
    int balance;                  // spread the FFN's neurons evenly: 1 over all CTAs (one more grid barrier per layer), 2/4/8 within groups of as many CTAs
    int32_t *glist, *gcount;      // [grid x STACK_MAX_CHUNK] published lists, [grid] their counts
    unsigned long long *gflag;    // [grid] per CTA: the last (launch, layer) epoch whose list it published
    float *x_layers;              // optional [L x d]: row l = x_{l+1} (every layer's output), or NULL
    unsigned long long *stamps;   // optional [L x STACK_PHASES x grid] %globaltimer stamps, or NULL
};

// Phase boundaries the persistent step can stamp per layer and CTA (pi_ffn_set_phase_trace).
constexpr int STACK_PHASES = 8;

template <int WT>
cudaError_t launch_stack_wt(int pdt, int kind, const StackArgs &a, int grid, size_t smem, cudaStream_t s);
extern template cudaError_t launch_stack_wt<0>(int, int, const StackArgs &, int, size_t, cudaStream_t);
extern template cudaError_t launch_stack_wt<1>(int, int, const StackArgs &, int, size_t, cudaStream_t);
extern template cudaError_t launch_stack_wt<2>(int, int, const StackArgs &, int, size_t, cudaStream_t);
extern template cudaError_t launch_stack_wt<3>(int, int, const StackArgs &, int, size_t, cudaStream_t);

// Tensor-core path (batch >= 16): modes of the one kernel template k_tc.
constexpr int TC_PRED_HIDDEN = 0, TC_LOGITS = 1, TC_GATED = 2, TC_RELU = 3, TC_DOWN = 4;
constexpr int TC_MAX_STAGES = 8;

struct TcArgs {
    const uint16_t *w0, *w1;      // weight rows [.. x K] (w1: up rows, gated only); TC_DOWN: W_down^T [f x d]
    const int32_t *idx, *count;   // gathered row list and its device count (NULL, NULL: rows 0..n_static-1)
    int n_static;
    int f;                        // row ids must lie in [0, f)
    int K, d;                     // contraction length (row modes); model width (TC_DOWN)
    const uint16_t *xhi, *xlo;    // activations hi/lo [NB x ldx], rows >= B zero
    int ldx, B;
    const float *bias;            // per-row bias indexed by row id, or NULL
    float tau;
    int row0;                     // row id of row 0 when there is no list (TC_LOGITS: start of the tiles)
    int hot;                      // TC_LOGITS: row ids below this are active without a logit (hot prefix)
    uint16_t *ohi, *olo;          // outputs hi/lo [NB x ldo] (hidden / h)
    int ldo;
    uint32_t *maskw;              // TC_LOGITS: mask words, then ascending idx_out, count_out
    int32_t *idx_out, *count_out;
    const float *xin;             // TC_DOWN: residual input or NULL
    float *out;                   // TC_DOWN: [B x d]
    float *part;                  // stream-K partials [grid x 2 x ACC x 128]
    uint32_t *tile_cnt, *done_cnt, *status;   // counters zero on entry, left zero
    int stages;
};

// w: 64-wide K blocks per pipeline step (row modes), or 128-column slices per W_down^T
// tile (TC_DOWN); 1 or 2.
template <int WT, int MODE>
cudaError_t launch_tc_mode(int nb, int w, const TcArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl);
#define PI_TC_EXTERN(WT, MODE) \
    extern template cudaError_t launch_tc_mode<WT, MODE>(int, int, const TcArgs &, int, size_t, cudaStream_t, bool);
PI_TC_EXTERN(1, 0) PI_TC_EXTERN(1, 1) PI_TC_EXTERN(1, 2) PI_TC_EXTERN(1, 3) PI_TC_EXTERN(1, 4)
PI_TC_EXTERN(2, 0) PI_TC_EXTERN(2, 1) PI_TC_EXTERN(2, 2) PI_TC_EXTERN(2, 3) PI_TC_EXTERN(2, 4)
#undef PI_TC_EXTERN
template <int WT>
cudaError_t launch_tc_split_wt(const float *x, int d, int B, int nb, int ld, int rms, float eps, uint16_t *hi,
                               uint16_t *lo, cudaStream_t s, bool pdl);
extern template cudaError_t launch_tc_split_wt<1>(const float *, int, int, int, int, int, float, uint16_t *,
                                                  uint16_t *, cudaStream_t, bool);
extern template cudaError_t launch_tc_split_wt<2>(const float *, int, int, int, int, int, float, uint16_t *,
                                                  uint16_t *, cudaStream_t, bool);

struct Launch {
    dim3 grid, block;     // grid.x == 0: persistent grid, one wave of resident CTAs over nsm SMs
    size_t smem;
    cudaStream_t stream;
    bool pdl;             // programmatic dependent launch after the previous kernel in the stream
    int nsm;
};

// K1: hp[b,k] = max(0, (x_b * inv_rms_b) . p1_t[k])  for all k < r, b < B.
cudaError_t launch_pred_hidden(const Launch &L, int pdt, int bt, const void *p1t, int d, int r,
                               const float *x, const float *inv_rms, int B, float *hp);

// K2: z = hp . p2_t[i] + b_pred[i]; mask bit i = OR_b (z > tau), and 1 without a logit for
// i < hot (hot prefix); the last CTA compacts the mask words into ascending idx[] and *count.
// ticket must be 0 on entry (left 0).
cudaError_t launch_pred_logits(const Launch &L, int pdt, int bt, const void *p2t, int r, int f,
                               const float *b_pred, float tau, const float *hp, int B,
                               uint32_t *maskw, uint32_t *ticket, int32_t *idx, int32_t *count, int hot);

// Fused predictor for small batches (one cooperative launch per layer, grid = one CTA per SM):
// hp = max(0, inv_rms_b * (P1T . x_b)) over all CTAs, one bounded grid barrier, then the logits
// and union mask of 32-neuron words (a contiguous range of words per CTA) and the compaction
// of the mask by the last CTA (as K1 + K2). inv_rms: given per row, or computed here from x
// (rms_self), or neither (x is u). hp is [B x r] workspace; bar a 64-bit grid-barrier counter
// of its own; ticket 0 on entry (left 0).
constexpr int FP_NT = 512;              // threads per CTA of the fused predictor
constexpr int FP_MAX_WORDS = 64;        // mask words per CTA (f <= 2048 * grid)
struct FusedPredArgs {
    const void *p1t, *p2t;
    const float *b_pred;
    int d, r, f, B, hot, rms_self;
    float tau, eps;
    const float *x, *inv_rms;
    float *hp;
    uint32_t *maskw, *ticket, *status;
    unsigned long long *bar;
    int32_t *idx, *count;
};
cudaError_t launch_pred_fused(int pdt, int bt, const FusedPredArgs &a, int grid, size_t smem, cudaStream_t s);

// K3: h[b,j] for the listed neurons j < *count.
cudaError_t launch_ffn_h(const Launch &L, int wdt, int kind, int bt, const void *wg, const void *wu,
                         const void *sg, const void *su, const float *bg, int d, int f,
                         const float *x, const float *inv_rms, int B,
                         const int32_t *idx, const int32_t *count, float *h, int ldh, uint32_t *status);

// K4a: part[g,b,:] = sum_{j in group g} h[b,j] * w_down_t[idx[j],:]
cudaError_t launch_ffn_down(const Launch &L, int wdt, int bt, const void *wd, const void *sd, int d, int f,
                            const int32_t *idx, const int32_t *count, const float *h, int ldh, int B,
                            float *part, uint32_t *status);

// K4b: y = sum_g part[g] (fixed order). With xin: out = xin + y, and inv_rms of out
// (last CTA) for the next layer. ticket must be 0 on entry (left 0).
cudaError_t launch_reduce(const Launch &L, const float *part, int d, int B, int f, const int32_t *count,
                          const float *xin, float *out, float *sumsq, uint32_t *ticket, float *inv_rms,
                          float eps);

// inv_rms[b] = 1 / sqrt(mean(x_b^2) + eps)
cudaError_t launch_rms(const Launch &L, const float *x, int d, int B, float *inv_rms, float eps);

// offline order
cudaError_t launch_hot_first(const uint32_t *counts, int f, int32_t *perm, cudaStream_t s);
cudaError_t launch_permute_rows(const void *src, void *dst, const int32_t *perm, int64_t rows, int64_t row_bytes,
                                int32_t *err, cudaStream_t s);

// groups of the down projection for a given active count (device and host agree)
__host__ __device__ inline int down_group_size(int n)
{
    int g = (n + MAX_GROUPS - 1) / MAX_GROUPS;
    return g < DOWN_GROUP_MIN ? DOWN_GROUP_MIN : g;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(const Launch &L, Kern kern, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = L.grid;
    if (cfg.gridDim.x == 0) {
        int occ = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, (int)(L.block.x * L.block.y),
                                                                      L.smem);
        if (e != cudaSuccess) return e;
        cfg.gridDim.x = (unsigned)(L.nsm * (occ > 0 ? occ : 1));
    }
    cfg.blockDim = L.block;
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Opt a kernel in to its dynamic shared memory when dynamic + static shared memory
// could pass the default 48 KB limit (remembered per kernel).
template <typename Kern>
cudaError_t ensure_smem(Kern kern, size_t bytes)
{
    static std::unordered_map<const void *, size_t> done;
    if (bytes + 8 * 1024 <= 48 * 1024) return cudaSuccess;
    auto it = done.find((const void *)kern);
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done[(const void *)kern] = bytes;
    return e;
}

}  // namespace pi
