// pi_api.cu -- host side of the C ABI declared in include/pi_ffn.h.
//
// Validates every argument before launching anything, owns the workspace, and
// chains the kernels of one decode step on the caller's stream: predictor
// (K1 hidden, K2 logits + compaction) -> gate/up gather (K3) -> W_down axpy (K4a)
// -> deterministic reduction (K4b). Kernels after the first of a call use
// programmatic dependent launch so that their weight loads overlap the
// previous kernel's tail. The layer stack is recorded into a CUDA graph.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <new>
#include <vector>

#include "pi_ffn.h"
#include "pi_internal.h"

using namespace pi;

namespace {

constexpr float RMS_EPS = 1e-6f;

typedef CUresult (*GetRangeFn)(CUdeviceptr *, size_t *, CUdeviceptr);

GetRangeFn get_range_fn()
{
    static GetRangeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (GetRangeFn)p;
        else
            cudaGetLastError();
    }
    return fn;
}

}  // namespace

namespace pi {

pi_status_t check_ptr(const void *p, size_t bytes, size_t align, int dev)
{
    if (!p || ((uintptr_t)p % align) != 0) return PI_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return PI_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return PI_ERR_INVALID_ARG;
    if (a.type == cudaMemoryTypeDevice && a.device != dev) return PI_ERR_INVALID_ARG;
    if (GetRangeFn fn = get_range_fn()) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (fn(&base, &size, (CUdeviceptr)(uintptr_t)p) == CUDA_SUCCESS) {
            if ((uintptr_t)p + bytes > (uintptr_t)base + size) return PI_ERR_INVALID_ARG;
        }
    }
    return PI_OK;
}

int injected_fault()
{
    const char *v = std::getenv("PI_FAULT");
    if (!v) return FAULT_NONE;
    if (!std::strcmp(v, "alloc")) return FAULT_ALLOC;
    if (!std::strcmp(v, "upload")) return FAULT_UPLOAD;
    if (!std::strcmp(v, "badarg")) return FAULT_BADARG;
    return FAULT_NONE;
}

}  // namespace pi

namespace {

pi_status_t check_opt(const void *p, size_t bytes, size_t align, int dev)
{
    return p ? check_ptr(p, bytes, align, dev) : PI_OK;
}

size_t elt_row_bytes(int dt, int64_t n)
{
    switch (dt) {
    case PI_F32: return (size_t)n * 4;
    case PI_BF16:
    case PI_F16: return (size_t)n * 2;
    case PI_INT4_G128: return (size_t)n / 2;
    }
    return 0;
}

pi_status_t validate_desc(const pi_ffn_desc_t *d)
{
    if (!d || injected_fault() == FAULT_BADARG) return PI_ERR_INVALID_ARG;
    if (d->d < 8 || d->d % 8 || d->f < 1 || d->r < 8 || d->r % 8 || d->n_layers < 1 || d->max_batch < 1 ||
        d->max_batch > 256)
        return PI_ERR_INVALID_ARG;
    if (d->kind != PI_FFN_GATED_RELU && d->kind != PI_FFN_RELU) return PI_ERR_INVALID_ARG;
    if (d->wdtype < PI_F32 || d->wdtype > PI_INT4_G128) return PI_ERR_INVALID_ARG;
    if (d->pdtype < PI_F32 || d->pdtype > PI_F16) return PI_ERR_INVALID_ARG;
    if (!std::isfinite(d->tau_logit)) return PI_ERR_INVALID_ARG;
    if (d->wdtype == PI_INT4_G128 && d->d % 128) return PI_ERR_UNSUPPORTED;
    // one batch row of the staged input vector must fit the shared-memory budget
    if ((size_t)d->d * 4 > SMEM_VEC_CAP || (size_t)d->r * 4 > SMEM_VEC_CAP) return PI_ERR_UNSUPPORTED;
    if (d->f > (1 << 26)) return PI_ERR_UNSUPPORTED;
    return PI_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

namespace pi {

int pick_bt(int B, int K, int cap)
{
    int fit = (int)(SMEM_VEC_CAP / ((size_t)K * 4));
    int bt = 1;
    while (bt * 2 <= cap && bt * 2 <= fit && bt < B) bt *= 2;
    return bt;
}

pi_status_t check_layer(const pi_ffn_desc_t &D, const pi_layer_weights_t &w, int dev, bool predictor)
{
    const size_t wrow = elt_row_bytes(D.wdtype, D.d), prow = elt_row_bytes(D.pdtype, D.d),
                 p2row = elt_row_bytes(D.pdtype, D.r);
    const size_t srow = (size_t)(D.d / 128) * 2;
    const bool gated = D.kind == PI_FFN_GATED_RELU, int4 = D.wdtype == PI_INT4_G128;
    pi_status_t s;
    if ((s = check_ptr(w.w_gate, wrow * D.f, 16, dev))) return s;
    if ((s = check_ptr(w.w_down_t, wrow * D.f, 16, dev))) return s;
    if (gated) {
        if ((s = check_ptr(w.w_up, wrow * D.f, 16, dev))) return s;
    } else if (w.w_up || w.s_up) {
        return PI_ERR_INVALID_ARG;
    }
    if (int4) {
        if ((s = check_ptr(w.s_gate, srow * D.f, 2, dev))) return s;
        if ((s = check_ptr(w.s_down, srow * D.f, 2, dev))) return s;
        if (gated && (s = check_ptr(w.s_up, srow * D.f, 2, dev))) return s;
    } else if (w.s_gate || w.s_up || w.s_down) {
        return PI_ERR_INVALID_ARG;
    }
    if ((s = check_opt(w.b_gate, (size_t)D.f * 4, 4, dev))) return s;
    if (!predictor) return PI_OK;
    if ((s = check_ptr(w.p1_t, prow * D.r, 16, dev))) return s;
    if ((s = check_ptr(w.p2_t, p2row * D.f, 16, dev))) return s;
    if ((s = check_opt(w.b_pred, (size_t)D.f * 4, 4, dev))) return s;
    return PI_OK;
}

}  // namespace pi

struct pi_ffn {
    pi_ffn_desc_t desc;
    std::vector<pi_layer_weights_t> layers;
    int dev = 0, nsm = 0;
    void *ws = nullptr;
    float *xbuf[2] = {nullptr, nullptr};
    float *inv_rms = nullptr, *sumsq = nullptr, *hp = nullptr, *hbuf = nullptr, *part = nullptr;
    uint32_t *maskw = nullptr, *tickets = nullptr, *status = nullptr;
    int32_t *idx_ws = nullptr, *count_ws = nullptr, *counts_ws = nullptr;
    // per-kernel event brackets (pi_profile_begin / pi_profile_end)
    bool prof = false;
    std::vector<cudaEvent_t> prof_ev;   // pairs: [2k] before, [2k+1] after launch k
    std::vector<int> prof_kind;
    size_t prof_n = 0;
    // persistent decode-step kernel (batch 1)
    bool stack_ok = false;
    int n_hot = 0;                     // neurons [0, n_hot) expected to fire on most tokens
    int hot_prefix = 0;                // neurons [0, hot_prefix) computed on every token
    int stack_p2 = 0;                  // ring slots of the persistent step for 16-row tiles of owned P2 rows
    StackLayer *stack_layers = nullptr;
    uint32_t *stack_mask = nullptr;
    float *stack_sumsq = nullptr;
    int stack_slots = 0, stack_slot_bytes = 0;
    size_t stack_smem = 0;
    unsigned long long *phase_stamps = nullptr;   // pi_ffn_set_phase_trace (borrowed device buffer)
    int stack_p2_stage = STACK_P2_TILES;   // P2 tiles filled between layers, at most (PI_FFN_STACK_P2_STAGE)
    int stack_balance = 0;             // persistent step: FFN neurons spread evenly over the CTAs (PI_FFN_STACK_BALANCE)
    int32_t *stack_glist = nullptr, *stack_gcount = nullptr;
    unsigned long long *stack_gflag = nullptr;
    int stack_pf = 1;                  // L2 prefetch of the persistent step: bit 0 P1, bit 1 unstaged P2 rows (PI_FFN_STACK_PF)
    int stack_pf_frac = 256;           // share (of 256) of the unstaged P2 rows prefetched during the FFN (PI_FFN_STACK_PF_P2_FRAC)
    int off_ring = 0, off_flags = 0, off_mbar = 0, off_hp = 0, off_scr = 0, stack_ring = 0;
    // fused predictor for batches up to pf_maxb (set by plan_pred_fused)
    int pf_maxb = 0;
    // tensor-core path (batch >= tc_min_b, set by plan_tc)
    bool tc_ok = false;
    int tc_min_b = 16, tc_nbmax = 0, tc_rpad = 0, tc_fpad = 0;
    int tc_stages[5][4][2] = {};       // [mode][log2(NB / 16)][log2(w)]
    size_t tc_smem[5][4][2] = {};
    int tc_kw = 1, tc_ds = 1, tc_stage_cap = TC_MAX_STAGES;   // tuning (PI_FFN_TC_KW / _DS / _STAGES)
    int tc_hidden_cpt = 8;             // CTAs per predictor-hidden tile (PI_FFN_TC_HIDDEN_CPT)
    uint16_t *tc_uhi = nullptr, *tc_ulo = nullptr, *tc_hphi = nullptr, *tc_hplo = nullptr, *tc_hhi = nullptr,
             *tc_hlo = nullptr;
    float *tc_part = nullptr;
    uint32_t *tc_cnt = nullptr;        // [tc_ntiles] tile tickets, then one done counter
    int tc_ntiles = 0;
    // recorded decode step (multi-kernel path)
    cudaGraphExec_t gexec = nullptr;
    int g_B = 0;
    const float *g_x0 = nullptr;
    float *g_xout = nullptr;
    int32_t *g_counts = nullptr, *g_idx = nullptr;
};

namespace {

pi_status_t cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return PI_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? PI_ERR_OOM : PI_ERR_CUDA;
}

Launch mk(const pi_ffn_t *h, dim3 grid, size_t smem, cudaStream_t s, bool pdl)
{
    Launch L;
    L.grid = grid;
    L.block = dim3(NT);
    L.smem = smem;
    L.stream = s;
    L.pdl = pdl;
    L.nsm = h->nsm;
    return L;
}

// Event bracket around one launch when profiling (no-op otherwise).
struct ProfScope {
    pi_ffn_t *h;
    cudaStream_t s;
    size_t slot;
    ProfScope(const pi_ffn_t *hc, cudaStream_t st, int kind) : h(const_cast<pi_ffn_t *>(hc)), s(st), slot(0)
    {
        if (!h->prof) return;
        slot = h->prof_n++;
        while (h->prof_ev.size() < 2 * h->prof_n) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) {
                cudaGetLastError();
                h->prof = false;
                return;
            }
            h->prof_ev.push_back(e);
        }
        if (h->prof_kind.size() < h->prof_n) h->prof_kind.resize(h->prof_n);
        h->prof_kind[slot] = kind;
        cudaEventRecord(h->prof_ev[2 * slot], s);
    }
    ~ProfScope()
    {
        if (h->prof && 2 * slot + 1 < h->prof_ev.size()) cudaEventRecord(h->prof_ev[2 * slot + 1], s);
    }
};

// A positive integer from the environment, else def.
int env_int(const char *name, int def)
{
    const char *v = std::getenv(name);
    return v && std::atoi(v) > 0 ? std::atoi(v) : def;
}

// Whether the fused predictor serves batch B on this handle.
bool pf_use(const pi_ffn_t *h, int B) { return B >= 1 && B <= h->pf_maxb; }

// The fused predictor (K1 + K2 in one cooperative launch) for one layer: u = x * inv_rms (inv_rms
// per row when given, else computed from x when rms_self, else u = x).
cudaError_t fused_predict(const pi_ffn_t *h, int layer, const float *x, const float *inv_rms, int rms_self, int B,
                          int32_t *idx, int32_t *count, cudaStream_t s)
{
    const pi_ffn_desc_t &D = h->desc;
    const pi_layer_weights_t &w = h->layers[layer];
    FusedPredArgs a;
    a.p1t = w.p1_t;
    a.p2t = w.p2_t;
    a.b_pred = w.b_pred;
    a.d = D.d;
    a.r = D.r;
    a.f = D.f;
    a.B = B;
    a.hot = h->hot_prefix;
    a.rms_self = rms_self;
    a.tau = D.tau_logit;
    a.eps = RMS_EPS;
    a.x = x;
    a.inv_rms = inv_rms;
    a.hp = h->hp;
    a.maskw = h->maskw;
    a.ticket = h->tickets + 0;
    a.status = h->status;
    a.bar = reinterpret_cast<unsigned long long *>(h->tickets + 4);
    a.idx = idx;
    a.count = count;
    const int bt = B <= 2 ? 2 : (B <= 4 ? 4 : 8);
    const size_t smem = (size_t)B * std::max(D.d, D.r) * 4;
    ProfScope p(h, s, PI_K_PRED_FUSED);
    return launch_pred_fused(D.pdtype, bt, a, h->nsm, smem, s);
}

// K1 + K2 for one layer. pdl_first: whether the first kernel may overlap its predecessor.
cudaError_t enqueue_predict(const pi_ffn_t *h, int layer, const float *x, const float *inv_rms, int B,
                            int32_t *idx, int32_t *count, cudaStream_t s, bool pdl_first)
{
    if (pf_use(h, B)) return fused_predict(h, layer, x, inv_rms, 0, B, idx, count, s);
    const pi_ffn_desc_t &D = h->desc;
    const pi_layer_weights_t &w = h->layers[layer];
    const int bt1 = pick_bt(B, D.d), bt2 = pick_bt(B, D.r);
    const bool pdl = !h->prof;
    cudaError_t e;
    {
        ProfScope p(h, s, PI_K_PRED_HIDDEN);
        e = launch_pred_hidden(
            mk(h, dim3((D.r + PRED_ROWS_HIDDEN - 1) / PRED_ROWS_HIDDEN), (size_t)bt1 * D.d * 4, s, pdl && pdl_first),
            D.pdtype, bt1, w.p1_t, D.d, D.r, x, inv_rms, B, h->hp);
    }
    if (e != cudaSuccess) return e;
    ProfScope p(h, s, PI_K_PRED_LOGITS);
    return launch_pred_logits(
        mk(h, dim3((D.f + PRED_ROWS_LOGIT - 1) / PRED_ROWS_LOGIT), (size_t)bt2 * D.r * 4, s, pdl), D.pdtype, bt2,
        w.p2_t, D.r, D.f, w.b_pred, D.tau_logit, h->hp, B, h->maskw, h->tickets + 0, idx, count, h->hot_prefix);
}

// K3 + K4a + K4b for one layer. xin != NULL: stack glue (out = xin + y, inv_rms for the next layer).
cudaError_t enqueue_ffn(const pi_ffn_t *h, int layer, const float *x, const float *inv_rms, int B,
                        const int32_t *idx, const int32_t *count, const float *xin, float *out, cudaStream_t s,
                        bool pdl_first)
{
    const pi_ffn_desc_t &D = h->desc;
    const pi_layer_weights_t &w = h->layers[layer];
    const int bt = pick_bt(B, D.d);
    const bool pdl = !h->prof;
    cudaError_t e;
    {
        ProfScope p(h, s, PI_K_FFN_H);
        e = launch_ffn_h(mk(h, dim3(0), (size_t)bt * D.d * 4, s, pdl && pdl_first), D.wdtype, D.kind, bt, w.w_gate,
                         w.w_up, w.s_gate, w.s_up, w.b_gate, D.d, D.f, x, inv_rms, B, idx, count, h->hbuf, D.f,
                         h->status);
    }
    if (e != cudaSuccess) return e;
    const int btd = pick_bt(B, 1, D.wdtype == PI_INT4_G128 ? 2 : 8);
    {
        ProfScope p(h, s, PI_K_FFN_DOWN);
        e = launch_ffn_down(mk(h, dim3(0), 0, s, pdl), D.wdtype, btd, w.w_down_t, w.s_down, D.d, D.f, idx, count,
                            h->hbuf, D.f, B, h->part, h->status);
    }
    if (e != cudaSuccess) return e;
    const dim3 rg((D.d + RED_COLS - 1) / RED_COLS, B);
    ProfScope p(h, s, PI_K_REDUCE);
    return launch_reduce(mk(h, rg, 0, s, pdl), h->part, D.d, B, D.f, count, xin, out, h->sumsq, h->tickets + 1,
                         h->inv_rms, RMS_EPS);
}

// ---------------------------------------------------------------- tensor-core path ----------

int tc_nb(int B) { return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : 128; }
int tc_nbi(int nb) { return nb == 16 ? 0 : nb == 32 ? 1 : nb == 64 ? 2 : 3; }

bool tc_use(const pi_ffn_t *h, int B) { return h->tc_ok && B >= h->tc_min_b && B <= h->tc_nbmax; }

// Whether the tensor-core kernels serve batches >= tc_min_b on this handle (16-bit weights
// and predictor of one type, d % 128 == 0, r % 64 == 0), and their shared-memory rings.
// The CUDA-core chain's time grows with the batch (one FMA chain per row and neuron) while
// the tensor-core kernels cost about the same for any batch up to their 16-row tile, so
// the crossover moves down as rows get longer: measured on a GB300 at batch 3 for d 5120
// and d 7168 (batch 2 still faster on the chain), between batches 4 and 6 for d 4096.
// PI_FFN_TC=0 turns the path off; PI_FFN_TC_MIN_BATCH moves its lower batch bound.
void plan_tc(pi_ffn_t *h)
{
    h->tc_ok = false;
    const pi_ffn_desc_t &D = h->desc;
    h->tc_min_b = D.d >= 5120 ? 3 : 6;
    const char *env = std::getenv("PI_FFN_TC");
    if (env && env[0] == '0') return;
    if (const char *mb = std::getenv("PI_FFN_TC_MIN_BATCH")) {
        const int v = std::atoi(mb);
        if (v >= 1) h->tc_min_b = v;
    }
    if (!((D.wdtype == PI_BF16 && D.pdtype == PI_BF16) || (D.wdtype == PI_F16 && D.pdtype == PI_F16))) return;
    if (D.d % 128 || D.r % 64 || D.max_batch < h->tc_min_b) return;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    h->tc_kw = env_int("PI_FFN_TC_KW", 2) >= 2 ? 2 : 1;
    h->tc_ds = env_int("PI_FFN_TC_DS", 2) >= 2 ? 2 : 1;
    h->tc_hidden_cpt = std::max(1, env_int("PI_FFN_TC_HIDDEN_CPT", 8));
    h->tc_stage_cap = std::min(TC_MAX_STAGES, env_int("PI_FFN_TC_STAGES", TC_MAX_STAGES));
    const size_t avail = (size_t)optin > 2048 ? (size_t)optin - 2048 : 0;   // alignment slack + static barriers
    for (int mode = 0; mode < 5; ++mode)
        for (int i = 0; i < 4; ++i)
            for (int wi = 0; wi < 2; ++wi) {
                const int nb = 16 << i, w = 1 << wi;
                const size_t stage = mode == TC_DOWN ? (size_t)w * 16384 + 2 * (size_t)nb * 128
                                                     : (mode == TC_GATED ? 2 : 1) * (size_t)w * 16384 +
                                                           2 * (size_t)w * nb * 128;
                const int st = (int)std::min<size_t>((size_t)h->tc_stage_cap, avail / stage);
                h->tc_stages[mode][i][wi] = st;
                h->tc_smem[mode][i][wi] = 1024 + (size_t)st * stage;
            }
    for (int mode = 0; mode < 5; ++mode)   // every mode must fit with w = 1
        for (int i = 0; i < 4; ++i)
            if (h->tc_stages[mode][i][0] < 2) return;
    h->tc_nbmax = tc_nb(std::min(D.max_batch, 128));
    h->tc_rpad = (D.r + 127) / 128 * 128;
    h->tc_fpad = (D.f + 127) / 128 * 128;
    h->tc_ntiles = std::max(h->tc_fpad / 128, std::max(h->tc_rpad / 128, D.d / 128));
    h->tc_ok = true;
}

// Width of one pipeline step (row modes: 64-wide K blocks; TC_DOWN: 128-column slices).
int tc_width(const pi_ffn_t *h, int mode, int nb, int K)
{
    if (mode == TC_DOWN) {
        int w = h->tc_ds;
        while (w > 1 && h->desc.d % (128 * w)) w /= 2;
        return w;
    }
    return h->tc_kw == 2 && K % 128 == 0 ? 2 : 1;
}

template <int WT>
cudaError_t tc_dispatch(int mode, int nb, int w, const TcArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl)
{
    switch (mode) {
    case TC_PRED_HIDDEN: return launch_tc_mode<WT, TC_PRED_HIDDEN>(nb, w, a, grid, smem, s, pdl);
    case TC_LOGITS: return launch_tc_mode<WT, TC_LOGITS>(nb, w, a, grid, smem, s, pdl);
    case TC_GATED: return launch_tc_mode<WT, TC_GATED>(nb, w, a, grid, smem, s, pdl);
    case TC_RELU: return launch_tc_mode<WT, TC_RELU>(nb, w, a, grid, smem, s, pdl);
    case TC_DOWN: return launch_tc_mode<WT, TC_DOWN>(nb, w, a, grid, smem, s, pdl);
    }
    return cudaErrorInvalidValue;
}

cudaError_t tc_launch(const pi_ffn_t *h, int mode, int nb, const TcArgs &a0, cudaStream_t s, bool pdl)
{
    TcArgs a = a0;
    const int i = tc_nbi(nb);
    int w = tc_width(h, mode, nb, a.K);
    int wi = w == 1 ? 0 : 1;
    if (h->tc_stages[mode][i][wi] < 2) {   // that width does not fit shared memory: one block per step
        w = 1;
        wi = 0;
    }
    a.stages = h->tc_stages[mode][i][wi];
    a.part = h->tc_part;
    a.tile_cnt = h->tc_cnt;
    a.done_cnt = h->tc_cnt + h->tc_ntiles;
    a.status = h->status;
    const size_t smem = h->tc_smem[mode][i][wi];
    // The predictor's hidden layer has few tiles (r / 128) and a long K: spread over every SM,
    // each tile's k range is cut into ~19 parts whose partials one CTA adds at the end. A few
    // CTAs per tile stream the same bytes with far fewer partials to add.
    int grid = h->nsm;
    if (mode == TC_PRED_HIDDEN && a.count == nullptr)
        grid = std::min(h->nsm, std::max(1, (a.n_static + 127) / 128) * h->tc_hidden_cpt);
    return h->desc.wdtype == PI_BF16 ? tc_dispatch<1>(mode, nb, w, a, grid, smem, s, pdl)
                                     : tc_dispatch<2>(mode, nb, w, a, grid, smem, s, pdl);
}

// u (or x_l with rms) -> uhi, ulo [NB x d]
cudaError_t tc_split(const pi_ffn_t *h, const float *x, int B, int rms, cudaStream_t s, bool pdl)
{
    const pi_ffn_desc_t &D = h->desc;
    const int nb = tc_nb(B);
    ProfScope p(h, s, PI_K_RMS);
    return D.wdtype == PI_BF16
               ? launch_tc_split_wt<1>(x, D.d, B, nb, D.d, rms, RMS_EPS, h->tc_uhi, h->tc_ulo, s, pdl && !h->prof)
               : launch_tc_split_wt<2>(x, D.d, B, nb, D.d, rms, RMS_EPS, h->tc_uhi, h->tc_ulo, s, pdl && !h->prof);
}

TcArgs tc_args()
{
    TcArgs a;
    std::memset(&a, 0, sizeof(a));
    return a;
}

// predictor on the tensor cores: hidden (P1T rows, K = d) then logits + mask + compaction (P2T rows, K = r)
cudaError_t tc_predict(const pi_ffn_t *h, int layer, int B, int32_t *idx, int32_t *count, cudaStream_t s)
{
    const pi_ffn_desc_t &D = h->desc;
    const pi_layer_weights_t &w = h->layers[layer];
    const int nb = tc_nb(B);
    const bool pdl = !h->prof;
    cudaError_t e;
    {
        TcArgs a = tc_args();
        a.w0 = (const uint16_t *)w.p1_t;
        a.n_static = D.r;
        a.f = D.r;
        a.K = D.d;
        a.d = D.d;
        a.xhi = h->tc_uhi;
        a.xlo = h->tc_ulo;
        a.ldx = D.d;
        a.B = B;
        a.ohi = h->tc_hphi;
        a.olo = h->tc_hplo;
        a.ldo = h->tc_rpad;
        ProfScope p(h, s, PI_K_PRED_HIDDEN);
        e = tc_launch(h, TC_PRED_HIDDEN, nb, a, s, pdl);
    }
    if (e != cudaSuccess) return e;
    TcArgs a = tc_args();
    // the tiles start at the last 128-row boundary inside the hot prefix (keeping one tile)
    a.hot = h->hot_prefix;
    a.row0 = std::min(h->hot_prefix / 128, (D.f - 1) / 128) * 128;
    a.w0 = (const uint16_t *)w.p2_t;
    a.n_static = D.f - a.row0;
    a.f = D.f;
    a.K = D.r;
    a.d = D.d;
    a.xhi = h->tc_hphi;
    a.xlo = h->tc_hplo;
    a.ldx = h->tc_rpad;
    a.B = B;
    a.bias = w.b_pred;
    a.tau = D.tau_logit;
    a.maskw = h->maskw;
    a.idx_out = idx;
    a.count_out = count;
    ProfScope p(h, s, PI_K_PRED_LOGITS);
    return tc_launch(h, TC_LOGITS, nb, a, s, pdl);
}

// FFN on the tensor cores: h for the listed neurons (gate/up or fc1 rows, K = d), then
// out = xin + h . WdT[idx] (xin NULL: out = y).
cudaError_t tc_ffn(const pi_ffn_t *h, int layer, int B, const int32_t *idx, const int32_t *count, const float *xin,
                   float *out, cudaStream_t s)
{
    const pi_ffn_desc_t &D = h->desc;
    const pi_layer_weights_t &w = h->layers[layer];
    const int nb = tc_nb(B);
    const bool pdl = !h->prof;
    cudaError_t e;
    {
        TcArgs a = tc_args();
        a.w0 = (const uint16_t *)w.w_gate;
        a.w1 = (const uint16_t *)w.w_up;
        a.idx = idx;
        a.count = count;
        a.f = D.f;
        a.K = D.d;
        a.d = D.d;
        a.xhi = h->tc_uhi;
        a.xlo = h->tc_ulo;
        a.ldx = D.d;
        a.B = B;
        a.bias = w.b_gate;
        a.ohi = h->tc_hhi;
        a.olo = h->tc_hlo;
        a.ldo = h->tc_fpad;
        ProfScope p(h, s, PI_K_FFN_H);
        e = tc_launch(h, D.kind == PI_FFN_GATED_RELU ? TC_GATED : TC_RELU, nb, a, s, pdl);
    }
    if (e != cudaSuccess) return e;
    TcArgs a = tc_args();
    a.w0 = (const uint16_t *)w.w_down_t;
    a.idx = idx;
    a.count = count;
    a.f = D.f;
    a.d = D.d;
    a.xhi = h->tc_hhi;
    a.xlo = h->tc_hlo;
    a.ldx = h->tc_fpad;
    a.B = B;
    a.xin = xin;
    a.out = out;
    ProfScope p(h, s, PI_K_FFN_DOWN);
    return tc_launch(h, TC_DOWN, nb, a, s, pdl);
}

// Layer l's output buffer: x_out for the last layer, else row l of x_layers when it is
// given, else one of the two ping-pong buffers.
float *layer_out(const pi_ffn_t *h, int l, int B, float *x_out, float *x_layers)
{
    if (l == h->desc.n_layers - 1) return x_out;
    return x_layers ? x_layers + (size_t)l * B * h->desc.d : h->xbuf[l & 1];
}

// The last layer's output also into the last row of x_layers (when given).
cudaError_t copy_last_layer(const pi_ffn_t *h, int B, const float *x_out, float *x_layers, cudaStream_t s)
{
    if (!x_layers) return cudaSuccess;
    const size_t n = (size_t)B * h->desc.d;
    return cudaMemcpyAsync(x_layers + (size_t)(h->desc.n_layers - 1) * n, x_out, n * 4, cudaMemcpyDeviceToDevice, s);
}

cudaError_t enqueue_stack_tc(const pi_ffn_t *h, const float *x0, int B, float *x_out, int32_t *counts,
                             int32_t *idx_out, float *x_layers, cudaStream_t s)
{
    const pi_ffn_desc_t &D = h->desc;
    cudaError_t e;
    const float *xl = x0;
    for (int l = 0; l < D.n_layers; ++l) {
        float *xn = layer_out(h, l, B, x_out, x_layers);
        int32_t *idx = idx_out ? idx_out + (size_t)l * D.f : h->idx_ws;
        int32_t *cnt = counts ? counts + l : h->counts_ws + l;
        if ((e = tc_split(h, xl, B, 1, s, l > 0)) != cudaSuccess) return e;
        if ((e = pf_use(h, B) ? fused_predict(h, l, xl, nullptr, 1, B, idx, cnt, s) : tc_predict(h, l, B, idx, cnt, s)) !=
            cudaSuccess)
            return e;
        if ((e = tc_ffn(h, l, B, idx, cnt, xl, xn, s)) != cudaSuccess) return e;
        xl = xn;
    }
    return copy_last_layer(h, B, x_out, x_layers, s);
}

cudaError_t enqueue_stack(const pi_ffn_t *h, const float *x0, int B, float *x_out, int32_t *counts,
                          int32_t *idx_out, float *x_layers, cudaStream_t s)
{
    const pi_ffn_desc_t &D = h->desc;
    if (tc_use(h, B)) return enqueue_stack_tc(h, x0, B, x_out, counts, idx_out, x_layers, s);
    cudaError_t e;
    {
        ProfScope p(h, s, PI_K_RMS);
        e = launch_rms(mk(h, dim3(B), 0, s, false), x0, D.d, B, h->inv_rms, RMS_EPS);
    }
    if (e != cudaSuccess) return e;
    const float *xl = x0;
    for (int l = 0; l < D.n_layers; ++l) {
        float *xn = layer_out(h, l, B, x_out, x_layers);
        int32_t *idx = idx_out ? idx_out + (size_t)l * D.f : h->idx_ws;
        int32_t *cnt = counts ? counts + l : h->counts_ws + l;
        if ((e = enqueue_predict(h, l, xl, h->inv_rms, B, idx, cnt, s, true)) != cudaSuccess) return e;
        if ((e = enqueue_ffn(h, l, xl, h->inv_rms, B, idx, cnt, xl, xn, s, true)) != cudaSuccess) return e;
        xl = xn;
    }
    return copy_last_layer(h, B, x_out, x_layers, s);
}

bool legacy_stream(cudaStream_t s) { return s == nullptr || s == cudaStreamLegacy; }

// The largest batch the fused predictor serves on this handle (0: none): its shared memory holds
// B rows of max(d, r) floats, each CTA at most FP_MAX_WORDS mask words. Off unless
// PI_FFN_PRED_FUSED=1 in the environment: measured on a GB300 it is slower than the two
// predictor kernels at batches 1-8 (those overlap their weight loads with the previous kernel
// through programmatic dependent launch; a cooperative launch cannot). PI_FFN_PRED_FUSED_MAXB
// lowers its batch bound (default 8).
void plan_pred_fused(pi_ffn_t *h)
{
    h->pf_maxb = 0;
    const char *env = std::getenv("PI_FFN_PRED_FUSED");
    if (!env || env[0] != '1') return;
    const pi_ffn_desc_t &D = h->desc;
    if (D.pdtype != PI_F32 && D.pdtype != PI_BF16 && D.pdtype != PI_F16) return;
    const int V = D.pdtype == PI_F32 ? 4 : 8;
    if (D.d % V || D.r % V) return;
    const int W = (D.f + 31) / 32;
    if ((W + h->nsm - 1) / h->nsm > FP_MAX_WORDS) return;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    const long long row = (long long)std::max(D.d, D.r) * 4;
    const long long fit = (optin - 8 * 1024) / row;   // static shared memory and slack
    h->pf_maxb = (int)std::min<long long>({8, fit, (long long)D.max_batch, (long long)env_int("PI_FFN_PRED_FUSED_MAXB", 8)});
    if (h->pf_maxb < 1) h->pf_maxb = 0;
}

// Whether the persistent decode-step kernel serves this handle at batch 1, and its
// shared-memory layout. PI_FFN_STACK_KERNEL=0 in the environment turns it off.
void plan_stack(pi_ffn_t *h)
{
    h->stack_ok = false;
    const char *env = std::getenv("PI_FFN_STACK_KERNEL");
    if (env && env[0] == '0') return;
    const pi_ffn_desc_t &D = h->desc;
    const bool combo = (D.wdtype == PI_F32 && D.pdtype == PI_F32) || (D.wdtype == PI_BF16 && D.pdtype == PI_BF16) ||
                       (D.wdtype == PI_F16 && D.pdtype == PI_F16) ||
                       (D.wdtype == PI_INT4_G128 && (D.pdtype == PI_F16 || D.pdtype == PI_BF16));
    if (!combo) return;
    const int V = D.wdtype == PI_F32 ? 4 : 8;                      // columns per unit of the FFN's thread mapping
    const int cpt = D.wdtype == PI_INT4_G128 ? 4 : 3;                  // units per thread (kernel instances)
    if (D.d % V || D.d / V > cpt * STACK_NT) return;
    if (D.wdtype == PI_INT4_G128) {
        if (D.d % 1024) return;                                    // scale rows must be 16-byte multiples
        for (const pi_layer_weights_t &w : h->layers)              // and start 16-byte aligned (bulk copies)
            if ((uintptr_t)w.s_gate % 16 || (uintptr_t)w.s_up % 16 || (uintptr_t)w.s_down % 16) return;
    }
    const int P = h->nsm;
    if (P > MAX_GROUPS) return;                                   // one fp32 partial per CTA
    if ((D.f + P - 1) / P > STACK_MAX_CHUNK) return;
    if ((D.r + P - 1) / P > STACK_MAX_P1_ROWS) return;
    for (const pi_layer_weights_t &w : h->layers)                  // gate bias may travel as a 16-byte chunk
        if ((uintptr_t)w.b_gate % 16) return;
    const int rows = D.kind == PI_FFN_GATED_RELU ? 3 : 2;
    const size_t rowb = elt_row_bytes(D.wdtype, D.d);
    const size_t sclb = D.wdtype == PI_INT4_G128 ? (size_t)(D.d / 128) * 2 : 0;
    const size_t slot = align_up(rows * (rowb + sclb) + 16, 128);
    const size_t own = (size_t)(D.f + P - 1) / P;
    // hp (phase BC, also as its hi/lo halves), the reduction scratch (BC and D), the logit flags
    const size_t off_hp = 0;
    const size_t off_scr = align_up((size_t)D.r * 4, 128);
    const size_t off_flags = off_scr + 8192;
    const size_t off_mbar = align_up(off_flags + own, 16);
    const size_t off_ring = align_up(off_mbar + 8 * STACK_MAX_SLOTS, 128);
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    const size_t cap = (size_t)optin > 8192 ? ((size_t)optin - 8192) / 128 * 128 : 0;   // room for static arrays
    if (off_ring + 2 * slot > cap) return;
    const size_t ring = cap - off_ring;
    h->stack_slots = (int)std::min((size_t)STACK_MAX_SLOTS, ring / slot);
    h->stack_slot_bytes = (int)slot;
    h->stack_ring = (int)((size_t)h->stack_slots * slot);
    h->off_hp = (int)off_hp;
    h->off_scr = (int)off_scr;
    h->off_ring = (int)off_ring;
    h->off_flags = (int)off_flags;
    h->off_mbar = (int)off_mbar;
    // The owned P2 rows pass through the ring in 16-row tiles: the first ones are copied in while
    // the ring is idle between one layer's FFN and the next layer's logits, and the logits stream
    // the rest through the same slots. A tile slot may reach past the last FFN slot, into the rest
    // of the shared memory (PI_FFN_STACK_P2=0: no tiles, the logits read P2 from memory).
    const char *p2env = std::getenv("PI_FFN_STACK_P2");
    const size_t p2row = elt_row_bytes(D.pdtype, D.r), p2st = (size_t)stack_p2_stride((int)p2row);
    h->stack_p2 = 0;
    if (!(p2env && p2env[0] == '0') && p2row % 16 == 0)
        h->stack_p2 = (int)std::min({(size_t)STACK_P2_TILES, ring / (16 * p2st), (own + 15) / 16});
    h->stack_smem = off_ring + std::max((size_t)h->stack_ring, (size_t)h->stack_p2 * 16 * p2st);
    // While one layer's predictor is small next to L2 (129 MB), the next layer's P1 rows and the P2
    // rows that the ring does not hold go to L2 a whole layer ahead. A larger predictor would be
    // evicted by the layer's own traffic before it is read (measured on the OPT-175B shape: 1.31x
    // the algorithmic DRAM bytes, 13% slower), so only its P1 rows go, during the grid barrier
    // after the FFN, landing during the reduction just before the predictor reads them.
    const size_t pred_bytes = elt_row_bytes(D.pdtype, D.d) * D.r + p2row * D.f;
    h->stack_pf = pred_bytes <= (40u << 20) ? 7 : 1;
    if (const char *pf = std::getenv("PI_FFN_STACK_PF")) h->stack_pf = std::max(0, std::min(15, std::atoi(pf)));
    if (const char *pr = std::getenv("PI_FFN_STACK_PF_P2_FRAC")) h->stack_pf_frac = std::max(0, std::min(256, std::atoi(pr)));
    // The FFN's active neurons spread within groups of 8 CTAs: measured on a GB300, +7% for gated
    // 16-bit layers of d 5120 (13B-like), -6% at d 4096 and -1.5% for int4 non-gated d 12288 (the
    // exchange costs the same, the spread it removes grows with the per-neuron work).
    h->stack_balance = D.kind == PI_FFN_GATED_RELU && (D.wdtype == PI_BF16 || D.wdtype == PI_F16) && D.d >= 5120 ? 8 : 0;
    if (const char *bl = std::getenv("PI_FFN_STACK_BALANCE")) {
        const int v = std::atoi(bl);
        h->stack_balance = v == 2 || v == 4 || v == 8 ? v : (v ? 1 : 0);
    }
    if (const char *ps = std::getenv("PI_FFN_STACK_P2_STAGE")) h->stack_p2_stage = std::max(0, std::atoi(ps));
    h->stack_ok = true;
}

cudaError_t launch_stack(const pi_ffn_t *h, const float *x0, float *x_out, int32_t *counts, int32_t *idx_out,
                         float *x_layers, cudaStream_t st)
{
    const pi_ffn_desc_t &D = h->desc;
    StackArgs a;
    a.layers = h->stack_layers;
    a.L = D.n_layers;
    a.d = D.d;
    a.f = D.f;
    a.r = D.r;
    a.tau = D.tau_logit;
    a.eps = RMS_EPS;
    a.x0 = x0;
    a.xa = h->xbuf[0];
    a.xb = h->xbuf[1];
    a.x_out = x_out;
    a.hp = h->hp;
    a.maskw = h->stack_mask;
    a.part = h->part;
    a.sumsq = h->stack_sumsq;
    a.counts = counts;
    a.idx_out = idx_out;
    a.bar = reinterpret_cast<unsigned long long *>(h->tickets + 2);
    a.status = h->status;
    a.slots = h->stack_slots;
    a.slot_bytes = h->stack_slot_bytes;
    a.nblocks = (unsigned)h->nsm;
    const long long pbytes = (D.pdtype == PI_F32 ? 4LL : 2LL) * ((long long)D.r * D.d + (long long)D.f * D.r);
    a.pf_bytes = std::min(pbytes, 48LL << 20);
    a.off_hp = h->off_hp;
    a.off_scr = h->off_scr;
    a.off_ring = h->off_ring;
    a.off_flags = h->off_flags;
    a.off_mbar = h->off_mbar;
    a.ring_bytes = h->stack_ring;
    a.hot_prefix = h->hot_prefix;
    a.hot_k = h->n_hot > 0 ? std::min((h->n_hot + h->nsm - 1) / h->nsm, h->stack_slots - 2) : 0;
    if (a.hot_k < 0) a.hot_k = 0;
    a.p2_tiles = a.hot_k > 0 ? 0 : h->stack_p2;   // the hot slots hold the ring between layers
    a.p2_stage_tiles = h->stack_p2_stage;
    a.pf_p1 = (h->stack_pf & 4) ? 2 : (h->stack_pf & 1);   // 2: a layer ahead, 1: just in time
    a.pf_p2 = (h->stack_pf >> 1) & 1;
    a.pf_p2_ffn = (h->stack_pf >> 3) & 1;
    a.pf_p2_frac = h->stack_pf_frac;
    a.balance = a.hot_k == 0 && (h->stack_balance == 1 || (h->stack_balance > 1 && h->nsm % h->stack_balance == 0))
                    ? h->stack_balance : 0;
    a.glist = h->stack_glist;
    a.gcount = h->stack_gcount;
    a.gflag = h->stack_gflag;
    a.x_layers = x_layers;
    a.stamps = h->phase_stamps;
    a.bias_bulk = D.f % 4 == 0 ? 1 : 0;
    for (const pi_layer_weights_t &w : h->layers)
        if (!w.b_gate) a.bias_bulk = 0;
    switch (D.wdtype) {
    case PI_F32: return launch_stack_wt<0>(D.pdtype, D.kind, a, h->nsm, h->stack_smem, st);
    case PI_BF16: return launch_stack_wt<1>(D.pdtype, D.kind, a, h->nsm, h->stack_smem, st);
    case PI_F16: return launch_stack_wt<2>(D.pdtype, D.kind, a, h->nsm, h->stack_smem, st);
    case PI_INT4_G128: return launch_stack_wt<3>(D.pdtype, D.kind, a, h->nsm, h->stack_smem, st);
    }
    return cudaErrorNotSupported;
}

}  // namespace

extern "C" {

int32_t pi_abi_version(void) { return PI_FFN_ABI_VERSION; }

const char *pi_status_string(pi_status_t s)
{
    switch (s) {
    case PI_OK: return "ok";
    case PI_ERR_INVALID_ARG: return "invalid argument";
    case PI_ERR_UNSUPPORTED: return "unsupported";
    case PI_ERR_CUDA: return "CUDA error";
    case PI_ERR_OOM: return "out of device memory";
    case PI_ERR_TIMEOUT: return "device-side wait timed out";
    case PI_ERR_DEVICE_CHECK: return "device-side input check failed";
    }
    return "unknown status";
}

pi_status_t pi_ffn_create(pi_ffn_t **out, const pi_ffn_desc_t *desc, const pi_layer_weights_t *layers)
{
    if (!out) return PI_ERR_INVALID_ARG;
    *out = nullptr;
    pi_status_t s = validate_desc(desc);
    if (s != PI_OK) return s;
    if (!layers) return PI_ERR_INVALID_ARG;

    pi_ffn_t *h = new (std::nothrow) pi_ffn_t();
    if (!h) return PI_ERR_OOM;
    h->desc = *desc;
    h->layers.assign(layers, layers + desc->n_layers);
    if ((s = cuda_status(cudaGetDevice(&h->dev))) != PI_OK ||
        (s = cuda_status(cudaDeviceGetAttribute(&h->nsm, cudaDevAttrMultiProcessorCount, h->dev))) != PI_OK) {
        delete h;
        return s;
    }
    for (int l = 0; l < desc->n_layers; ++l) {
        if ((s = check_layer(h->desc, h->layers[l], h->dev, true)) != PI_OK) {
            delete h;
            return s;
        }
    }

    plan_tc(h);
    plan_pred_fused(h);
    const pi_ffn_desc_t &D = h->desc;
    const size_t mb = (size_t)D.max_batch;
    const size_t tnb = h->tc_ok ? (size_t)h->tc_nbmax : 0;
    const size_t nred = (size_t)(D.d + RED_COLS - 1) / RED_COLS;
    const size_t sizes[] = {
        mb * D.d * 4, mb * D.d * 4,                    // xbuf[2]
        mb * 4,                                        // inv_rms
        nred * mb * 4,                                 // sumsq
        mb * D.r * 4,                                  // hp
        mb * D.f * 4,                                  // hbuf
        (size_t)MAX_GROUPS * mb * D.d * 4,             // part
        (size_t)(D.f + 31) / 32 * 4,                   // maskw
        8 * 4,                                         // tickets: [0] logits, [1] reduce, [2..3] stack barrier, [4..5] fused predictor barrier
        4,                                             // status
        (size_t)D.f * 4,                               // idx_ws
        4,                                             // count_ws
        (size_t)D.n_layers * 4,                        // counts_ws
        (size_t)D.n_layers * sizeof(StackLayer),       // stack_layers
        (size_t)D.n_layers * ((D.f + 31) / 32) * 4,    // stack_mask
        (size_t)(D.d + STACK_SLICE - 1) / STACK_SLICE * 4,  // stack_sumsq
        tnb * D.d * 2, tnb * D.d * 2,                  // tc_uhi, tc_ulo
        tnb * h->tc_rpad * 2, tnb * h->tc_rpad * 2,    // tc_hphi, tc_hplo
        tnb * h->tc_fpad * 2, tnb * h->tc_fpad * 2,    // tc_hhi, tc_hlo
        (size_t)h->nsm * 2 * 256 * 128 * 4 * (tnb ? 1 : 0),   // tc_part: two slots of up to 256 accumulator columns
        h->tc_ok ? (size_t)(h->tc_ntiles + 1) * 4 : 0, // tc_cnt
        (size_t)h->nsm * STACK_MAX_CHUNK * 4,          // stack_glist
        (size_t)h->nsm * 4,                            // stack_gcount
        (size_t)h->nsm * 8,                            // stack_gflag
    };
    const int nbuf = sizeof(sizes) / sizeof(sizes[0]);
    size_t off[32], total = 0;
    for (int i = 0; i < nbuf; ++i) {
        off[i] = total;
        total = align_up(total + sizes[i], 256);
    }
    const int fault = injected_fault();
    if ((s = cuda_status(fault == FAULT_ALLOC ? cudaErrorMemoryAllocation : cudaMalloc(&h->ws, total))) != PI_OK) {
        delete h;
        return s;
    }
    if ((s = cuda_status(cudaMemset(h->ws, 0, total))) != PI_OK) {
        cudaFree(h->ws);
        delete h;
        return s;
    }
    char *base = (char *)h->ws;
    h->xbuf[0] = (float *)(base + off[0]);
    h->xbuf[1] = (float *)(base + off[1]);
    h->inv_rms = (float *)(base + off[2]);
    h->sumsq = (float *)(base + off[3]);
    h->hp = (float *)(base + off[4]);
    h->hbuf = (float *)(base + off[5]);
    h->part = (float *)(base + off[6]);
    h->maskw = (uint32_t *)(base + off[7]);
    h->tickets = (uint32_t *)(base + off[8]);
    h->status = (uint32_t *)(base + off[9]);
    h->idx_ws = (int32_t *)(base + off[10]);
    h->count_ws = (int32_t *)(base + off[11]);
    h->counts_ws = (int32_t *)(base + off[12]);
    h->stack_layers = (StackLayer *)(base + off[13]);
    h->stack_mask = (uint32_t *)(base + off[14]);
    h->stack_sumsq = (float *)(base + off[15]);
    if (h->tc_ok) {
        h->tc_uhi = (uint16_t *)(base + off[16]);
        h->tc_ulo = (uint16_t *)(base + off[17]);
        h->tc_hphi = (uint16_t *)(base + off[18]);
        h->tc_hplo = (uint16_t *)(base + off[19]);
        h->tc_hhi = (uint16_t *)(base + off[20]);
        h->tc_hlo = (uint16_t *)(base + off[21]);
        h->tc_part = (float *)(base + off[22]);
        h->tc_cnt = (uint32_t *)(base + off[23]);
    }
    h->stack_glist = (int32_t *)(base + off[24]);
    h->stack_gcount = (int32_t *)(base + off[25]);
    h->stack_gflag = (unsigned long long *)(base + off[26]);
    {
        std::vector<StackLayer> sl(D.n_layers);
        for (int l = 0; l < D.n_layers; ++l) {
            const pi_layer_weights_t &w = h->layers[l];
            sl[l] = StackLayer{w.w_gate, w.w_up, w.w_down_t, w.s_gate, w.s_up, w.s_down, w.b_gate, w.p1_t, w.p2_t,
                               w.b_pred};
        }
        if ((s = cuda_status(fault == FAULT_UPLOAD ? cudaErrorInvalidValue
                                                   : cudaMemcpy(h->stack_layers, sl.data(),
                                                                sl.size() * sizeof(StackLayer),
                                                                cudaMemcpyHostToDevice))) != PI_OK) {
            cudaFree(h->ws);
            delete h;
            return s;
        }
    }
    plan_stack(h);
    *out = h;
    return PI_OK;
}

void pi_ffn_destroy(pi_ffn_t *h)
{
    if (!h) return;
    cudaDeviceSynchronize();
    if (h->gexec) cudaGraphExecDestroy(h->gexec);
    for (cudaEvent_t e : h->prof_ev) cudaEventDestroy(e);
    if (h->ws) cudaFree(h->ws);
    cudaGetLastError();
    delete h;
}

pi_status_t pi_predict(pi_ffn_t *h, int32_t layer, const float *u, int32_t B, int32_t *idx, int32_t *count,
                       void *stream)
{
    if (!h || layer < 0 || layer >= h->desc.n_layers || B < 1 || B > h->desc.max_batch) return PI_ERR_INVALID_ARG;
    const pi_ffn_desc_t &D = h->desc;
    pi_status_t s;
    if ((s = check_ptr(u, (size_t)B * D.d * 4, 16, h->dev))) return s;
    if ((s = check_ptr(idx, (size_t)D.f * 4, 4, h->dev))) return s;
    if ((s = check_ptr(count, 4, 4, h->dev))) return s;
    if (tc_use(h, B) && !pf_use(h, B)) {
        cudaError_t e = tc_split(h, u, B, 0, (cudaStream_t)stream, false);
        if (e == cudaSuccess) e = tc_predict(h, layer, B, idx, count, (cudaStream_t)stream);
        return cuda_status(e);
    }
    return cuda_status(enqueue_predict(h, layer, u, nullptr, B, idx, count, (cudaStream_t)stream, false));
}

pi_status_t pi_sparse_ffn(pi_ffn_t *h, int32_t layer, const float *u, int32_t B, const int32_t *idx,
                          const int32_t *count, float *y, void *stream)
{
    if (!h || layer < 0 || layer >= h->desc.n_layers || B < 1 || B > h->desc.max_batch) return PI_ERR_INVALID_ARG;
    const pi_ffn_desc_t &D = h->desc;
    pi_status_t s;
    if ((s = check_ptr(u, (size_t)B * D.d * 4, 16, h->dev))) return s;
    if ((s = check_ptr(idx, 4, 4, h->dev))) return s;      // length is *count, checked on the device
    if ((s = check_ptr(count, 4, 4, h->dev))) return s;
    if ((s = check_ptr(y, (size_t)B * D.d * 4, 16, h->dev))) return s;
    if (tc_use(h, B)) {
        cudaError_t e = tc_split(h, u, B, 0, (cudaStream_t)stream, false);
        if (e == cudaSuccess) e = tc_ffn(h, layer, B, idx, count, nullptr, y, (cudaStream_t)stream);
        return cuda_status(e);
    }
    return cuda_status(enqueue_ffn(h, layer, u, nullptr, B, idx, count, nullptr, y, (cudaStream_t)stream, false));
}

}  // extern "C"

namespace {

pi_status_t decode_stack(pi_ffn_t *h, const float *x0, int32_t B, float *x_out, int32_t *counts, int32_t *idx_out,
                         float *x_layers, void *stream)
{
    if (!h || B < 1 || B > h->desc.max_batch) return PI_ERR_INVALID_ARG;
    const pi_ffn_desc_t &D = h->desc;
    pi_status_t s;
    if ((s = check_ptr(x0, (size_t)B * D.d * 4, 16, h->dev))) return s;
    if ((s = check_ptr(x_out, (size_t)B * D.d * 4, 16, h->dev))) return s;
    if ((s = check_opt(counts, (size_t)D.n_layers * 4, 4, h->dev))) return s;
    if ((s = check_opt(idx_out, (size_t)D.n_layers * D.f * 4, 4, h->dev))) return s;
    if ((s = check_opt(x_layers, (size_t)D.n_layers * B * D.d * 4, 16, h->dev))) return s;
    cudaStream_t st = (cudaStream_t)stream;

    if (B == 1 && h->stack_ok) {
        ProfScope p(h, st, PI_K_STACK);
        cudaError_t e = launch_stack(h, x0, x_out, counts, idx_out, x_layers, st);
        if (e == cudaSuccess) return PI_OK;
        cudaGetLastError();
        if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge) return cuda_status(e);
        h->stack_ok = false;   // not launchable here: use the multi-kernel path from now on
    }

    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (!legacy_stream(st) && cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cuda_status(cudaGetLastError());
    if (legacy_stream(st) || cs != cudaStreamCaptureStatusNone || h->prof || x_layers)
        return cuda_status(enqueue_stack(h, x0, B, x_out, counts, idx_out, x_layers, st));

    if (!(h->gexec && h->g_B == B && h->g_x0 == x0 && h->g_xout == x_out && h->g_counts == counts &&
          h->g_idx == idx_out)) {
        if (h->gexec) {
            cudaGraphExecDestroy(h->gexec);
            h->gexec = nullptr;
        }
        cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed);
        if (e != cudaSuccess) return cuda_status(e);
        cudaError_t el = enqueue_stack(h, x0, B, x_out, counts, idx_out, nullptr, st);
        cudaGraph_t g = nullptr;
        e = cudaStreamEndCapture(st, &g);
        if (el != cudaSuccess || e != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            return cuda_status(el != cudaSuccess ? el : e);
        }
        e = cudaGraphInstantiate(&h->gexec, g, 0);
        cudaGraphDestroy(g);
        if (e != cudaSuccess) {
            h->gexec = nullptr;
            return cuda_status(e);
        }
        h->g_B = B;
        h->g_x0 = x0;
        h->g_xout = x_out;
        h->g_counts = counts;
        h->g_idx = idx_out;
    }
    return cuda_status(cudaGraphLaunch(h->gexec, st));
}

}  // namespace

extern "C" {

pi_status_t pi_decode_stack(pi_ffn_t *h, const float *x0, int32_t B, float *x_out, int32_t *counts,
                            int32_t *idx_out, void *stream)
{
    return decode_stack(h, x0, B, x_out, counts, idx_out, nullptr, stream);
}

pi_status_t pi_decode_stack_layers(pi_ffn_t *h, const float *x0, int32_t B, float *x_out, int32_t *counts,
                                   int32_t *idx_out, float *x_layers, void *stream)
{
    if (!x_layers) return PI_ERR_INVALID_ARG;
    return decode_stack(h, x0, B, x_out, counts, idx_out, x_layers, stream);
}

pi_status_t pi_ffn_set_phase_trace(pi_ffn_t *h, uint64_t *stamps, int64_t n_stamps)
{
    if (!h) return PI_ERR_INVALID_ARG;
    if (!stamps) {
        h->phase_stamps = nullptr;
        return PI_OK;
    }
    const int64_t need = (int64_t)h->desc.n_layers * STACK_PHASES * h->nsm;
    if (n_stamps < need) return PI_ERR_INVALID_ARG;
    pi_status_t s;
    if ((s = check_ptr(stamps, (size_t)need * 8, 8, h->dev))) return s;
    h->phase_stamps = reinterpret_cast<unsigned long long *>(stamps);
    return PI_OK;
}

pi_status_t pi_ffn_set_hot_prefix(pi_ffn_t *h, int32_t n_hot)
{
    if (!h || n_hot < 0 || n_hot > h->desc.f) return PI_ERR_INVALID_ARG;
    h->hot_prefix = n_hot;
    return PI_OK;
}

pi_status_t pi_ffn_set_hot_neurons(pi_ffn_t *h, int32_t n_hot)
{
    if (!h || n_hot < 0 || n_hot > h->desc.f) return PI_ERR_INVALID_ARG;
    h->n_hot = n_hot;
    return PI_OK;
}

pi_status_t pi_profile_begin(pi_ffn_t *h)
{
    if (!h) return PI_ERR_INVALID_ARG;
    h->prof = true;
    h->prof_n = 0;
    return PI_OK;
}

pi_status_t pi_profile_end(pi_ffn_t *h, float *ms, int32_t *launches, int32_t n_kinds)
{
    if (!h || n_kinds < 0) return PI_ERR_INVALID_ARG;
    const bool was = h->prof;
    h->prof = false;
    for (int k = 0; k < n_kinds; ++k) {
        if (ms) ms[k] = 0.f;
        if (launches) launches[k] = 0;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_status(cudaGetLastError());
    if (!was) return PI_OK;
    for (size_t i = 0; i < h->prof_n && 2 * i + 1 < h->prof_ev.size(); ++i) {
        const int k = h->prof_kind[i];
        float t = 0.f;
        if (cudaEventElapsedTime(&t, h->prof_ev[2 * i], h->prof_ev[2 * i + 1]) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (k >= 0 && k < n_kinds) {
            if (ms) ms[k] += t;
            if (launches) launches[k] += 1;
        }
    }
    h->prof_n = 0;
    return PI_OK;
}

pi_status_t pi_get_status(pi_ffn_t *h)
{
    if (!h) return PI_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_status(cudaGetLastError());
    uint32_t v = 0;
    if (cudaMemcpy(&v, h->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_status(cudaGetLastError());
    if (v && cudaMemset(h->status, 0, 4) != cudaSuccess) return cuda_status(cudaGetLastError());
    // a grid barrier that gave up leaves its arrival count (and the compaction ticket behind it)
    // behind: start the next step clean
    if (v == PI_ERR_TIMEOUT && cudaMemset(h->tickets, 0, 8 * 4) != cudaSuccess) return cuda_status(cudaGetLastError());
    // the group exchange's epochs derive from the barrier counter: restart them with it
    if (v == PI_ERR_TIMEOUT && h->stack_gflag && cudaMemset(h->stack_gflag, 0, (size_t)h->nsm * 8) != cudaSuccess)
        return cuda_status(cudaGetLastError());
    // so does a tensor-core kernel that gave up between its tile tickets
    if (v == PI_ERR_TIMEOUT && h->tc_cnt &&
        cudaMemset(h->tc_cnt, 0, (size_t)(h->tc_ntiles + 1) * 4) != cudaSuccess)
        return cuda_status(cudaGetLastError());
    return (pi_status_t)v;
}

pi_status_t pi_hot_first_order(const uint32_t *counts, int32_t f, int32_t *perm, void *stream)
{
    if (f < 0) return PI_ERR_INVALID_ARG;
    if (f == 0) return PI_OK;
    int dev = 0;
    pi_status_t s;
    if ((s = cuda_status(cudaGetDevice(&dev)))) return s;
    if ((s = check_ptr(counts, (size_t)f * 4, 4, dev))) return s;
    if ((s = check_ptr(perm, (size_t)f * 4, 4, dev))) return s;
    return cuda_status(launch_hot_first(counts, f, perm, (cudaStream_t)stream));
}

pi_status_t pi_permute_rows(const void *src, void *dst, const int32_t *perm, int64_t rows, int64_t row_bytes,
                            int32_t *err, void *stream)
{
    if (rows < 0 || row_bytes < 0) return PI_ERR_INVALID_ARG;
    if (rows == 0 || row_bytes == 0) return PI_OK;
    const size_t n = (size_t)rows * (size_t)row_bytes;
    int dev = 0;
    pi_status_t s;
    if ((s = cuda_status(cudaGetDevice(&dev)))) return s;
    if ((s = check_ptr(src, n, 1, dev))) return s;
    if ((s = check_ptr(dst, n, 1, dev))) return s;
    if ((s = check_ptr(perm, (size_t)rows * 4, 4, dev))) return s;
    if ((s = check_opt(err, 4, 4, dev))) return s;
    const uintptr_t a = (uintptr_t)src, b = (uintptr_t)dst;
    if (a < b + n && b < a + n) return PI_ERR_INVALID_ARG;
    return cuda_status(launch_permute_rows(src, dst, perm, rows, row_bytes, err, (cudaStream_t)stream));
}

}  // extern "C"
