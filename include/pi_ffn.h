/*
 * pi_ffn.h -- C ABI of libpi_ffn.so: activation-sparse FFN decode on one GB300 (sm_103a).
 *
 * The method is the one the PowerInfer pages describe: per layer, a small
 * predictor decides which FFN neurons will be non-zero, and only those neurons'
 * weight rows are read ("PowerInfer" paper walk-through page, section
 * "inference flow": input reaches a layer -> predictor -> compute the predicted
 * neurons -> merge -> next layer; summary page, Methodology: neuron-aware sparse
 * operators that do matrix-vector products at neuron granularity).
 * Here the whole model is resident in HBM; nothing runs on the CPU at inference.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers (cudaMalloc'd or managed), borrowed:
 *    the caller owns them and keeps them alive while the library may read them.
 *    Host pointers are rejected with PI_ERR_INVALID_ARG before any launch.
 *  - Matrices are row-major. Every FFN matrix is stored neuron-major: row i of
 *    w_gate / w_up / w_down_t holds the d weights of neuron i (w_down_t is the
 *    transpose of the down projection). Neurons are expected in hot-first order
 *    (pi_hot_first_order), which keeps frequently active rows contiguous.
 *  - Element types: PI_F32 (fp32), PI_BF16, PI_F16, PI_INT4_G128. INT4_G128:
 *    per-row groups of 128 consecutive elements share one fp16 scale s; the
 *    value is q*s with q a signed 4-bit two's-complement integer; element 2k is
 *    the low nibble of byte k. Scales are [rows x d/128] fp16.
 *  - Activations and outputs are fp32; every dot product accumulates in fp32.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). All calls after
 *    pi_ffn_create are asynchronous on `stream`; they validate arguments on the
 *    host first and return an error without launching anything if one is bad.
 *  - Errors found by the kernels (an active index outside [0, f), a count
 *    outside [0, f]) are recorded in a device status word and the offending
 *    entry is skipped; pi_get_status() reports them. No kernel traps.
 *  - No C++ exception crosses this boundary. Not thread-safe per handle.
 *
 * Environment, read at pi_ffn_create (all optional; the defaults are the tuned paths):
 *  - PI_FFN_STACK_KERNEL=0  batch-1 steps use the multi-kernel chain instead of the
 *                           persistent one-kernel step.
 *  - PI_FFN_STACK_P2=0      the persistent step reads the predictor's P2 rows from memory
 *                           instead of passing them through its shared-memory ring.
 *  - PI_FFN_STACK_BALANCE=n the persistent step spreads the layer's active neurons evenly: 1
 *                           over all CTAs (one more grid barrier per layer), 2, 4 or 8 within
 *                           groups of as many consecutive CTAs (the members exchange their lists
 *                           through memory, no grid barrier); 0: each CTA computes its own active
 *                           neurons. Default 8 for gated 16-bit layers with d >= 5120 (~7% faster
 *                           on Llama2-13B-like layers), else 0 (slower on the OPT-175B- and
 *                           ReluLLaMA-7B-like ones).
 *  - PI_FFN_STACK_PF=n      L2 prefetches of the persistent step, a bit mask: 1 = the next
 *                           layer's P1 rows (during the grid barrier after the FFN, or a whole
 *                           layer ahead with 4), 2 = the next layer's P2 rows that the ring does
 *                           not hold, a whole layer ahead, 8 = those rows during this layer's
 *                           FFN (the first PI_FFN_STACK_PF_P2_FRAC / 256 of them, default all).
 *                           Default 7 while one layer's predictor is at most 40 MB, else 1.
 *  - PI_FFN_STACK_P2_STAGE=n  at most n P2 tiles are copied into the ring between layers (the
 *                           rest as the logits start); default all that fit.
 *  - PI_FFN_TC=0            every batch > 1 stays on the CUDA-core kernels.
 *  - PI_FFN_TC_MIN_BATCH=n  smallest batch for the tensor-core path (default 3 for
 *                           d >= 5120, else 6).
 *  - PI_FFN_PRED_FUSED=1    the predictor of batches up to 8 (pi_predict, the multi-kernel and
 *                           tensor-core steps) runs as one cooperative launch (hidden layer over
 *                           all SMs, a grid barrier, logits, mask and compaction) instead of two
 *                           kernels; off by default (slower on a GB300, see the design notes).
 *  - PI_FFN_PRED_FUSED_MAXB=n  largest batch for the one-launch predictor (default 8; also
 *                           bounded by B * max(d, r) * 4 bytes of shared memory).
 *  - PI_FFN_TC_KW, PI_FFN_TC_DS, PI_FFN_TC_STAGES, PI_FFN_TC_HIDDEN_CPT: tensor-core step
 *    widths (64-wide K blocks per step, 128-column W_down slices per tile: 1 or 2, default
 *    2), ring depth cap, and CTAs per predictor-hidden tile (default 8).
 * They change speed and, for some, the order of floating-point additions (so the output
 * bits), not what is computed.
 *  - PI_FAULT=alloc|upload|badarg  host-side fault injection for failure-path tests:
 *    pi_ffn_create then fails its workspace allocation (PI_ERR_OOM, nothing allocated),
 *    fails after the workspace exists (PI_ERR_CUDA, the workspace is freed again), or
 *    rejects the descriptor (PI_ERR_INVALID_ARG). *out is NULL in every case.
 */
#ifndef PI_FFN_H
#define PI_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PI_FFN_ABI_VERSION 1

typedef enum {
    PI_OK = 0,
    PI_ERR_INVALID_ARG = 1,   /* bad size, NULL / misaligned / host pointer, layer or batch out of range */
    PI_ERR_UNSUPPORTED = 2,   /* a valid request the library does not implement (e.g. int4 with d % 128 != 0) */
    PI_ERR_CUDA = 3,          /* a CUDA runtime call failed */
    PI_ERR_OOM = 4,           /* workspace allocation failed */
    PI_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up */
    PI_ERR_DEVICE_CHECK = 6   /* a kernel rejected an input entry (see conventions) */
} pi_status_t;

typedef enum {
    PI_FFN_GATED_RELU = 0,    /* LLaMA-style: h_i = ReLU(u.Wg_i + bg_i) * (u.Wu_i) */
    PI_FFN_RELU = 1           /* OPT/Falcon-style: h_i = ReLU(u.W1_i + b1_i); w_gate holds W1 */
} pi_ffn_kind_t;

typedef enum { PI_F32 = 0, PI_BF16 = 1, PI_F16 = 2, PI_INT4_G128 = 3 } pi_dtype_t;

/* Shape and numerics of a layer stack. All layers share it. */
typedef struct {
    int32_t d;          /* model width; multiple of 8 (of 128 for PI_INT4_G128) */
    int32_t f;          /* FFN width (neurons), >= 1 */
    int32_t r;          /* predictor rank, multiple of 8 */
    int32_t n_layers;   /* >= 1 */
    int32_t max_batch;  /* largest B any call will pass, 1..256; sizes the workspace */
    int32_t kind;       /* pi_ffn_kind_t */
    int32_t wdtype;     /* pi_dtype_t of w_gate / w_up / w_down_t */
    int32_t pdtype;     /* pi_dtype_t of p1_t / p2_t: PI_F32, PI_BF16 or PI_F16 */
    float tau_logit;    /* threshold on the predictor logit; neuron active iff z > tau (0 <=> sigmoid > 0.5) */
} pi_ffn_desc_t;

/* One layer's weights (device pointers, borrowed; 16-byte aligned). */
typedef struct {
    const void *w_gate;    /* [f x d] Wg (gated) or W1 (non-gated) */
    const void *w_up;      /* [f x d] Wu; NULL for PI_FFN_RELU */
    const void *w_down_t;  /* [f x d] W_down transposed */
    const void *s_gate;    /* int4 only: fp16 [f x d/128]; else NULL */
    const void *s_up;      /* int4 + gated only; else NULL */
    const void *s_down;    /* int4 only; else NULL */
    const float *b_gate;   /* [f] fp32 gate / fc1 bias, or NULL (zero) */
    const void *p1_t;      /* [r x d] predictor first layer, transposed (row k = weights of hidden unit k) */
    const void *p2_t;      /* [f x r] predictor second layer, transposed (row i = weights of neuron i's logit) */
    const float *b_pred;   /* [f] fp32 predictor bias, or NULL (zero) */
} pi_layer_weights_t;

typedef struct pi_ffn pi_ffn_t;

/*
 * Create a handle for a stack of desc->n_layers layers. `layers` (host array of
 * n_layers descriptors) is copied; the weight memory it points to is borrowed.
 * Allocates the workspace (predictor hidden state, mask words, active indices,
 * h, fp32 partial sums, stack buffers, status word) on the current device.
 * Returns PI_ERR_INVALID_ARG / PI_ERR_UNSUPPORTED / PI_ERR_OOM / PI_ERR_CUDA with
 * *out = NULL on failure.
 */
pi_status_t pi_ffn_create(pi_ffn_t **out, const pi_ffn_desc_t *desc, const pi_layer_weights_t *layers);

/* Free the workspace and the handle (waits for the device first). NULL is a no-op. */
void pi_ffn_destroy(pi_ffn_t *h);

/*
 * Activation predictor of layer `layer` ("PowerInfer" walk-through page, section
 * "activation predictor", eq. a = sigmoid(x Wp + b_p), neuron i active when
 * a_i > tau; read as a two-layer low-rank MLP):
 *   hp[b,k] = max(0, u[b,:] . p1_t[k,:])               k < r
 *   z[b,i]  = hp[b,:] . p2_t[i,:] + b_pred[i]          i < f
 *   neuron i is active iff z[b,i] > tau_logit for at least one row b (union over the batch).
 * u:     [B x d] fp32 device, the layer input (already normalised).
 * idx:   [f] int32 device, out: the active neurons in ascending order (entries >= *count unspecified).
 * count: one int32 device, out: number of active neurons.
 * 1 <= B <= max_batch.
 */
pi_status_t pi_predict(pi_ffn_t *h, int32_t layer, const float *u, int32_t B,
                       int32_t *idx, int32_t *count, void *stream);

/*
 * Neuron-sparse FFN of layer `layer` over a given active list (same page, section
 * "technical details", eq. FFN(x) = sigma(x W1) (.) (x W2) W3, sigma = ReLU), reading
 * only the listed neurons' rows:
 *   gated:     h[b,j] = max(0, u_b . Wg_i + bg_i) * (u_b . Wu_i),    i = idx[j], j < *count
 *   non-gated: h[b,j] = max(0, u_b . W1_i + b1_i)
 *   y[b,:]     = sum_j h[b,j] * w_down_t[i,:]
 * The sum is deterministic: fixed groups of consecutive list entries are summed in
 * list order into fp32 partials, and the partials are added in a fixed order, so the
 * bits of y depend only on the inputs. Any index list is accepted (ascending or not,
 * empty when *count == 0); entries outside [0, f) are skipped and flagged.
 * u: [B x d] fp32; idx: [>= *count] int32; count: one int32 (device); y: [B x d] fp32 out.
 * Argument errors are found before any launch. If the CUDA runtime refuses a later launch of
 * the chain (not an argument error), PI_ERR_CUDA is returned with the earlier kernels already
 * enqueued; they write only the workspace, and y is then not written.
 */
pi_status_t pi_sparse_ffn(pi_ffn_t *h, int32_t layer, const float *u, int32_t B,
                          const int32_t *idx, const int32_t *count, float *y, void *stream);

/*
 * One decode step through all n_layers layers (the walk-through page's per-layer
 * inference flow, merge -> next layer), with a parameter-free pre-norm residual
 * between layers (the pages are silent about non-FFN layers):
 *   x_0 = x0;  u_l = x_l / sqrt(mean(x_l^2) + 1e-6);  x_{l+1} = x_l + FFN_l(u_l over predict_l(u_l))
 * x0: [B x d] fp32 device; x_out: [B x d] fp32 device, out (= x_L).
 * counts: [n_layers] int32 device out (active count per layer), or NULL.
 * idx_out: [n_layers x f] int32 device out (layer l's ascending active list in row l), or NULL.
 * No host synchronisation inside. B = 1 steps (element-type pairs f32/f32, bf16/bf16,
 * f16/f16, int4/f16, int4/bf16, when the shapes fit its shared-memory plan) run as ONE
 * persistent cooperative kernel, one CTA per SM, whose layers are separated by bounded
 * grid barriers; a barrier that gives up records PI_ERR_TIMEOUT. Its partial sums are
 * one per CTA, so the output bits depend on the SM count (and nothing else).
 * PI_FFN_STACK_KERNEL=0 in the environment at pi_ffn_create turns it off;
 * PI_FFN_STACK_P2=0 keeps the predictor's P2 rows out of its shared memory (the logits
 * then run on the CUDA cores from memory). Other steps
 * run as a chain of kernels, recorded once outside stream capture into a CUDA graph
 * per (B, pointer set) and replayed.
 */
pi_status_t pi_decode_stack(pi_ffn_t *h, const float *x0, int32_t B, float *x_out,
                            int32_t *counts, int32_t *idx_out, void *stream);

/*
 * pi_decode_stack that also keeps every layer's output, for checking a step layer by layer
 * (the walk-through page's inference flow hands each layer's merged output to the next
 * layer; this exposes those hand-offs). Computes exactly what pi_decode_stack computes, on
 * the same kernels, and writes x_{l+1} to row l of x_layers.
 * x_layers: [n_layers x B x d] fp32 device, out (row n_layers - 1 equals x_out); not NULL.
 * The multi-kernel chain then runs without its recorded graph. Other arguments and errors
 * as pi_decode_stack.
 */
pi_status_t pi_decode_stack_layers(pi_ffn_t *h, const float *x0, int32_t B, float *x_out,
                                   int32_t *counts, int32_t *idx_out, float *x_layers, void *stream);

/*
 * Phase timing of the persistent batch-1 step (tracing aid; off by default). With a buffer
 * set, every later pi_decode_stack / pi_decode_stack_layers call that runs the persistent
 * kernel writes, per layer l, phase boundary p < PI_STACK_PHASES and CTA c (one CTA per SM),
 * the GPU's nanosecond global timer to stamps[(l * PI_STACK_PHASES + p) * n_sm + c].
 * Boundaries: 0 layer start (predictor hidden layer), 1 hidden layer done, 2 after the grid
 * barrier (logits start), 3 active list ready, 4 first batch of active rows landed (= 3 when
 * the CTA has no active neuron), 5 the CTA's FFN partial written, 6 after the grid barrier
 * (reduction start), 7 reduction done. Only thread 0 of each CTA writes; one store per
 * boundary. stamps: device, 8-byte aligned, n_stamps >= n_layers * PI_STACK_PHASES * n_sm
 * (n_sm = the device's multiprocessor count), borrowed until it is replaced or cleared.
 * NULL clears it. Returns PI_ERR_INVALID_ARG for a short or non-device buffer.
 */
#define PI_STACK_PHASES 8
pi_status_t pi_ffn_set_phase_trace(pi_ffn_t *h, uint64_t *stamps, int64_t n_stamps);

/*
 * Offline hot-first order (walk-through page, section "offline profiling", code
 * block: per-neuron activation counts sorted in descending order). perm[k] = the
 * neuron that moves to position k: counts descending, equal counts keep their
 * original (ascending) order. counts: [f] uint32 device; perm: [f] int32 device out.
 */
pi_status_t pi_hot_first_order(const uint32_t *counts, int32_t f, int32_t *perm, void *stream);

/*
 * Apply an order to a row-major matrix: row k of dst = row perm[k] of src.
 * rows rows of row_bytes bytes each; src and dst must not overlap.
 * err: one int32 device counter (or NULL), incremented per perm entry outside
 * [0, rows); such destination rows are left unwritten.
 */
pi_status_t pi_permute_rows(const void *src, void *dst, const int32_t *perm, int64_t rows,
                            int64_t row_bytes, int32_t *err, void *stream);

/*
 * Per-kernel timing (tracing aid). Between pi_profile_begin and pi_profile_end, every
 * kernel the handle launches is bracketed by two CUDA events on its stream, and
 * pi_decode_stack runs without its CUDA graph and without programmatic overlap, so
 * each bracket is that kernel's own duration. pi_profile_end waits for the device and
 * writes, per kernel kind k < n_kinds (pi_kernel_kind_t), the summed milliseconds
 * ms[k] and the number of launches launches[k] (either array may be NULL).
 */
typedef enum {
    PI_K_RMS = 0,          /* RMS scale of the stack input */
    PI_K_PRED_HIDDEN = 1,  /* predictor hidden layer */
    PI_K_PRED_LOGITS = 2,  /* predictor logits, union mask, compaction */
    PI_K_FFN_H = 3,        /* gate/up gather-GEMV */
    PI_K_FFN_DOWN = 4,     /* row-sparse W_down axpy into fp32 partials */
    PI_K_REDUCE = 5,       /* deterministic reduction (+ residual, next RMS scale) */
    PI_K_STACK = 6,        /* persistent decode step, all layers in one kernel (batch 1) */
    PI_K_PRED_FUSED = 7,   /* predictor hidden layer + logits + union mask + compaction, one launch (small batches) */
    PI_K_COUNT = 8
} pi_kernel_kind_t;

pi_status_t pi_profile_begin(pi_ffn_t *h);
pi_status_t pi_profile_end(pi_ffn_t *h, float *ms, int32_t *launches, int32_t n_kinds);

/*
 * Allocation-free variant of pi_sparse_ffn for callers that cannot call cudaMalloc
 * (code inside an allocator callback, a plugin whose host owns all device memory,
 * a runtime that forbids allocation after start-up), and so cannot create a handle.
 * The pages have no counterpart: this is a deployment convenience, not a step of
 * the method.
 *
 * Computes exactly what pi_sparse_ffn computes for one layer described by `desc`
 * (only d, f, r, kind, wdtype are read) and `layer`, with the same kernels. Its
 * scratch memory (h and the fp32 partial sums) is a static device array inside the
 * library, PI_NOALLOC_SCRATCH_BYTES per GPU, held from the library's load on that GPU
 * until process exit. The call needs (B*f rounded up to 64 + 256*B*d) * 4 bytes of it
 * and returns PI_ERR_UNSUPPORTED, launching nothing, when that exceeds the array.
 * Set-up: the first call on each device looks up the array's device address with
 * that device current (again after the device's context changes, e.g. after a
 * cudaDeviceReset); make that first call before any stream capture. The lookup is
 * guarded by a mutex, so first calls from several host threads are safe.
 * Every call shares the array and it keeps the previous call's contents (this path
 * needs none of it zeroed); calls whose kernels overlap on the GPU race on it, so
 * order them on one stream. u and y must hold B*d floats, idx and count as for
 * pi_sparse_ffn; pointers are checked like a handle's (inside their allocations).
 * status: optional int32 device word; a kernel that
 * rejects a list entry or count sets it to PI_ERR_DEVICE_CHECK if it is 0 (clear it
 * before the call). No cudaMalloc, cudaFree or other allocating call is made.
 * The three kernels are launched one after another: every argument error is found
 * before the first launch, but if the CUDA runtime refuses the second or third
 * launch, the call returns PI_ERR_CUDA with the earlier kernels already enqueued
 * (they write only the scratch array), and y is not written.
 */
#define PI_NOALLOC_SCRATCH_BYTES (16u << 20)

pi_status_t pi_sparse_ffn_noalloc(const pi_ffn_desc_t *desc, const pi_layer_weights_t *layer,
                                  const float *u, int32_t B, const int32_t *idx, const int32_t *count,
                                  float *y, int32_t *status, void *stream);

/*
 * Failure-detection self-test of the bounded grid barrier used by pi_decode_stack.
 * work: 4 zeroed uint32 words of device memory, 8-byte aligned: [0..1] barrier counter, [2] number of
 * CTAs that passed the barrier, [3] status out. A cooperative grid of 2 CTAs meets at
 * the barrier expecting 2 + extra CTAs. extra = 0: both pass, work[2] = 2, work[3] = 0.
 * extra > 0: no CTA can pass; each gives up after the barrier's limit (200 ms),
 * work[3] = PI_ERR_TIMEOUT, and the kernel returns (no trap, the context stays usable).
 */
pi_status_t pi_selftest_grid_barrier(uint32_t *work, int32_t extra, void *stream);

/*
 * Check of the tensor-core (tcgen05) operand layouts used by the batched path: one
 * CTA stages A and B in shared memory the way those kernels do, multiplies them on the
 * tensor cores with an fp32 accumulator in tensor memory, and writes
 * d[128 x n] = A * B^T (row-major fp32, device).
 *   a: device, 16-bit elements of `dtype` (PI_BF16 or PI_F16). mode 0: A as [128 x k]
 *      row-major (staged K-major). mode 1: A^T as [k x 128] row-major (staged MN-major).
 *   b: device, [n x k] row-major (staged K-major).
 *   n in {16, 32, 64, 128}; k in {64, 128}. a, b, d 16-byte aligned.
 *   status: device uint32, set to PI_ERR_TIMEOUT if the product's completion is not
 *   signalled within 200 ms (the kernel then returns without writing d).
 * Returns PI_ERR_INVALID_ARG for other shapes or non-device pointers.
 */
pi_status_t pi_selftest_umma(const void *a, const void *b, float *d, int32_t mode, int32_t n, int32_t k,
                             int32_t dtype, uint32_t *status, void *stream);

/*
 * Hot prefix (a variant of the method). The pages split neurons into hot ones, which fire on
 * most inputs and are served without question, and cold ones, which the predictor decides
 * ("PowerInfer" paper walk-through page, hot/cold neurons and inference flow; summary page,
 * Methodology). With hot_prefix = H, neurons [0, H) of the hot-first order are active on
 * every token without a logit (their P2 rows are not read), and the predictor decides only
 * [H, f). pi_predict returns [0, H) followed by the predicted tail, ascending; pi_decode_stack
 * computes both. The result differs from H = 0 only where the predictor would have dropped a
 * hot neuron whose gate is positive: it is then closer to the dense FFN. 0 (the default) is
 * the plain method. Returns PI_ERR_INVALID_ARG unless 0 <= H <= f. Takes effect from the next call.
 */
pi_status_t pi_ffn_set_hot_prefix(pi_ffn_t *h, int32_t hot_prefix);

/*
 * Hot neurons of the batch-1 decode step. The offline profile ("PowerInfer" paper
 * walk-through, offline profiling code block; summary page, Methodology: a small set of
 * hot neurons fires on most inputs) orders neurons hot-first; n_hot says that neurons
 * [0, n_hot) fire on most tokens. The persistent batch-1 kernel of pi_decode_stack then
 * requests those neurons' rows one layer ahead, before their predictor has run, into ring
 * slots of their own (at most ring slots - 2 per SM). A hot neuron that the predictor
 * rejects costs its bytes but does not change the result. With hot slots every CTA computes
 * the FFN of its own neurons (the even spread of the neurons over the CTAs is off), and the
 * output is bit-identical for every n_hot > 0 to the output with PI_FFN_STACK_BALANCE=0.
 * 0 (the default) turns this off. Other paths ignore it.
 * Returns PI_ERR_INVALID_ARG unless 0 <= n_hot <= f. Takes effect from the next call.
 */
pi_status_t pi_ffn_set_hot_neurons(pi_ffn_t *h, int32_t n_hot);

/* Wait for all work on the device, return the first kernel-recorded error and clear it. */
pi_status_t pi_get_status(pi_ffn_t *h);

/* Static text for a status code. */
const char *pi_status_string(pi_status_t s);

/* PI_FFN_ABI_VERSION of the loaded library. */
int32_t pi_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PI_FFN_H */
