// pi_predict.cu -- activation predictor kernels (sm_103a, CUDA cores).
//
// "PowerInfer" paper walk-through page, section "activation predictor": every
// layer has a small predictor that says, from the layer input, which FFN
// neurons will fire (eq. a = sigmoid(x Wp + b_p), active where a_i > tau).
// Read here as a two-layer low-rank MLP, thresholded on the logit:
//   K1  hp[b,k] = max(0, u_b . P1T[k])                 (dense GEMV, r rows of d)
//   K2  z[b,i]  = hp_b . P2T[i] + b_pred[i];  active_i = OR_b (z[b,i] > tau)
//       followed by compaction of the active bits into an ascending index list.
// Both are HBM-bound streams of the predictor weights. The weight loads of the
// first chunk batch are issued before waiting for the producer of u / hp
// (programmatic dependent launch), so they overlap the previous kernel's tail.
#include "pi_async.cuh"
#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_rowdot.cuh"

namespace pi {

// ---------------------------------------------------------------- K1 -------------------------
// CTA: 8 warps, PRED_ROWS_HIDDEN rows; warp w takes the w-th eighth of every row.
template <int PT, int BT>
__global__ void __launch_bounds__(NT, 2)
k_pred_hidden(const uint4 *__restrict__ P1, int d, int r, const float *__restrict__ x,
              const float *__restrict__ inv_rms, int B, float *__restrict__ hp)
{
    constexpr int RW = PRED_ROWS_HIDDEN, U = 4, V = Vec<PT>::N;
    extern __shared__ float4 su4[];                 // [BT][d/4] planar
    __shared__ float red[NW][RW][BT];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = d / V;
    const int per = (nch + NW - 1) / NW;
    const int cb = warp * per, ce = min(nch, cb + per);
    const int row0 = blockIdx.x * RW;

    const uint4 *row[RW];
    const __half *srow[RW];
#pragma unroll
    for (int k = 0; k < RW; ++k) {
        row[k] = row0 + k < r ? P1 + (size_t)(row0 + k) * nch : nullptr;
        srow[k] = nullptr;
    }

    RowChunks<PT, RW, U> rc;
    rows_issue(rc, row, srow, cb + lane, ce);   // input-independent: before the wait
    pdl_launch_dependents();
    pdl_wait();

    for (int b0 = 0; b0 < B; b0 += BT) {
        const int bt = min(BT, B - b0);
        __syncthreads();
        stage_planar<PT, BT>(su4, x + (size_t)b0 * d, d, bt, inv_rms ? inv_rms + b0 : nullptr);
        __syncthreads();
        if (b0 > 0) rows_issue(rc, row, srow, cb + lane, ce);
        float acc[RW][BT];
#pragma unroll
        for (int k = 0; k < RW; ++k)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[k][b] = 0.f;
        for (int c = cb + lane;;) {
            rows_consume<PT, RW, U, BT>(rc, c, ce, su4, d, acc);
            c += 32 * U;
            if (c >= ce) break;
            rows_issue(rc, row, srow, c, ce);
        }
#pragma unroll
        for (int k = 0; k < RW; ++k)
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                const float s = warp_sum(acc[k][b]);
                if (lane == 0) red[warp][k][b] = s;
            }
        __syncthreads();
        if (threadIdx.x < RW * BT) {
            const int k = threadIdx.x / BT, b = threadIdx.x - k * BT;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += red[w][k][b];   // fixed order
            if (row0 + k < r && b < bt) hp[(size_t)(b0 + b) * r + row0 + k] = fmaxf(s, 0.f);
        }
    }
}

// ---------------------------------------------------------------- K2 -------------------------
// CTA: 8 warps, 32 consecutive neurons (one mask word); warp w takes neurons w, w+8, w+16, w+24.
template <int PT, int BT>
__global__ void __launch_bounds__(NT, 2)
k_pred_logits(const uint4 *__restrict__ P2, int r, int f, const float *__restrict__ b_pred, float tau,
              const float *__restrict__ hp, int B, uint32_t *__restrict__ maskw, uint32_t *__restrict__ ticket,
              int32_t *__restrict__ idx, int32_t *__restrict__ count, int hot)
{
    constexpr int RW = PRED_ROWS_LOGIT / NW, U = 4, V = Vec<PT>::N;
    extern __shared__ float4 su4[];                 // [BT][r/4] planar
    __shared__ uint32_t word;
    __shared__ bool last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = r / V;
    const int n0 = blockIdx.x * PRED_ROWS_LOGIT;

    const uint4 *row[RW];
    const __half *srow[RW];
#pragma unroll
    for (int k = 0; k < RW; ++k) {
        const int i = n0 + warp + NW * k;
        row[k] = (i < f && i >= hot) ? P2 + (size_t)i * nch : nullptr;   // hot prefix: no logit needed
        srow[k] = nullptr;
    }
    if (threadIdx.x == 0) word = 0u;

    RowChunks<PT, RW, U> rc;
    rows_issue(rc, row, srow, lane, nch);        // input-independent: before the wait
    pdl_launch_dependents();
    pdl_wait();

    uint32_t bits = 0u;
    for (int b0 = 0; b0 < B; b0 += BT) {
        const int bt = min(BT, B - b0);
        __syncthreads();
        stage_planar<PT, BT>(su4, hp + (size_t)b0 * r, r, bt, nullptr);
        __syncthreads();
        if (b0 > 0) rows_issue(rc, row, srow, lane, nch);
        float acc[RW][BT];
#pragma unroll
        for (int k = 0; k < RW; ++k)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[k][b] = 0.f;
        for (int c = lane;;) {
            rows_consume<PT, RW, U, BT>(rc, c, nch, su4, r, acc);
            c += 32 * U;
            if (c >= nch) break;
            rows_issue(rc, row, srow, c, nch);
        }
#pragma unroll
        for (int k = 0; k < RW; ++k) {
            const int i = n0 + warp + NW * k;
            const float bias = (i < f && b_pred) ? __ldg(b_pred + i) : 0.f;
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                const float z = warp_sum(acc[k][b]) + bias;
                if (i < f && b < bt && (i < hot || z > tau)) bits |= 1u << (warp + NW * k);
            }
        }
    }
    if (lane == 0 && bits) atomicOr(&word, bits);
    __syncthreads();
    if (threadIdx.x == 0) {
        maskw[blockIdx.x] = word;
        last = ticket_acq_rel(ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __shared__ int wsum[NW];
    compact_words<NW>(maskw, gridDim.x, 0, idx, count, wsum, [] { __syncthreads(); });
    if (threadIdx.x == 0) *ticket = 0u;
}

// ---------------------------------------------------------------- fused predictor ------------
// Small batches: K1 and K2 as one cooperative launch over every SM. Each CTA stages the B input
// rows in shared memory, takes r / grid rows of P1 (thread t: chunks t, t + 512, ... of RG rows
// at once, the rows' dot products with every input row), and after one bounded grid barrier
// the logits of a contiguous range of 32-neuron mask words: warp w takes NPW neurons at a time,
// all their P2 chunks in flight, and the union over the rows sets the neuron's bit. The last
// CTA to finish compacts the mask words into the ascending list.
template <int PT, int BT>
__global__ void __launch_bounds__(FP_NT, 1) k_pred_fused(FusedPredArgs a)
{
    constexpr int V = Vec<PT>::N, FW = FP_NT / 32;
    constexpr int RG = BT >= 4 ? 32 / BT : 8;   // P1 rows per pass: RG * BT <= 32 sums per thread
    constexpr int NPW = BT <= 4 ? 3 : 2;        // neurons per warp in flight in the logits
    constexpr int QC = 4;                       // P2 chunks per lane and neuron in flight
    extern __shared__ float4 fsm4[];
    float *xs = reinterpret_cast<float *>(fsm4);   // [B][d] the inputs, then [B][r] hp
    __shared__ float red[FW][32];
    __shared__ float sinv[BT];
    __shared__ uint32_t sword[FP_MAX_WORDS];
    __shared__ unsigned long long s_base;
    __shared__ int s_flag, wsum[FW];
    __shared__ bool s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x, B = a.B, d = a.d, r = a.r, f = a.f;
    if (tid == 0) s_base = barrier_base(a.bar, (unsigned long long)P);

    // the input rows into shared memory, and their RMS scales
    float ssq[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        ssq[b] = 0.f;
        if (b < B)
            for (int j = tid; j < d / 4; j += FP_NT) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.x + (size_t)b * d) + j);
                reinterpret_cast<float4 *>(xs + (size_t)b * d)[j] = v;
                ssq[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
    }
    if (a.rms_self) {
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const float t = warp_sum(ssq[b]);
            if (lane == 0) red[warp][b] = t;
        }
        __syncthreads();
        if (tid < BT) {
            float t = 0.f;
            for (int w = 0; w < FW; ++w) t += red[w][tid];   // fixed order
            sinv[tid] = 1.f / sqrtf(t / (float)d + a.eps);
        }
    } else if (tid < BT) {
        sinv[tid] = (a.inv_rms && tid < B) ? a.inv_rms[tid] : 1.f;
    }
    __syncthreads();

    // hidden layer: rows [k0, k1) of P1T
    const int k0 = (int)((long long)c * r / P), k1 = (int)((long long)(c + 1) * r / P);
    const int nch = d / V;
    const uint4 *p1 = reinterpret_cast<const uint4 *>(a.p1t);
    for (int kb = k0; kb < k1; kb += RG) {
        float acc[RG][BT];
#pragma unroll
        for (int g = 0; g < RG; ++g)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[g][b] = 0.f;
        for (int j = tid; j < nch; j += FP_NT) {
            uint4 wv[RG];
#pragma unroll
            for (int g = 0; g < RG; ++g)
                wv[g] = kb + g < k1 ? __ldg(p1 + (size_t)(kb + g) * nch + j) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                if (b >= B) break;
                float xv[V];
#pragma unroll
                for (int e4 = 0; e4 < V / 4; ++e4) {
                    const float4 t = reinterpret_cast<const float4 *>(xs + (size_t)b * d + (size_t)j * V)[e4];
                    xv[4 * e4] = t.x; xv[4 * e4 + 1] = t.y; xv[4 * e4 + 2] = t.z; xv[4 * e4 + 3] = t.w;
                }
#pragma unroll
                for (int g = 0; g < RG; ++g) {
                    float wf[V];
                    unpack<PT>(wv[g], wf);
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[g][b] = fmaf(wf[e], xv[e], acc[g][b]);
                }
            }
        }
#pragma unroll
        for (int g = 0; g < RG; ++g)
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                const float t = warp_sum(acc[g][b]);
                if (lane == 0) red[warp][g * BT + b] = t;
            }
        __syncthreads();
        if (tid < RG * BT) {
            const int g = tid / BT, b = tid - g * BT;
            float t = 0.f;
            for (int w = 0; w < FW; ++w) t += red[w][tid];   // fixed order
            if (kb + g < k1 && b < B) a.hp[(size_t)b * r + kb + g] = fmaxf(t * sinv[b], 0.f);
        }
        __syncthreads();
    }
    if (!grid_sync_to(a.bar, s_base + (unsigned long long)P, a.status, &s_flag)) return;

    // logits of the words [w0, w1): hp into shared memory first
    float *hs = xs;
#pragma unroll
    for (int b = 0; b < BT; ++b)
        if (b < B)
            for (int j = tid; j < r / 4; j += FP_NT)
                reinterpret_cast<float4 *>(hs + (size_t)b * r)[j] = __ldcg(reinterpret_cast<const float4 *>(a.hp + (size_t)b * r) + j);
    const int W = (f + 31) / 32;
    const int w0 = (int)((long long)c * W / P), w1 = (int)((long long)(c + 1) * W / P);
    for (int i = tid; i < w1 - w0; i += FP_NT) sword[i] = 0u;
    __syncthreads();
    const int n0 = 32 * w0, n1 = min(f, 32 * w1), nchr = r / V;
    const uint4 *p2 = reinterpret_cast<const uint4 *>(a.p2t);
    for (int nb = n0 + warp * NPW; nb < n1; nb += FW * NPW) {
        float acc[NPW][BT];
#pragma unroll
        for (int p = 0; p < NPW; ++p)
#pragma unroll
            for (int b = 0; b < BT; ++b) acc[p][b] = 0.f;
        for (int q0 = lane; q0 < nchr; q0 += 32 * QC) {
            uint4 wv[NPW][QC];
#pragma unroll
            for (int p = 0; p < NPW; ++p) {
                const int i = nb + p;
                const bool need = i < n1 && i >= a.hot;   // the hot prefix needs no logit
#pragma unroll
                for (int u = 0; u < QC; ++u) {
                    const int q = q0 + 32 * u;
                    wv[p][u] = need && q < nchr ? __ldg(p2 + (size_t)i * nchr + q) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < QC; ++u) {
                const int q = q0 + 32 * u;
                if (q >= nchr) break;
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    if (b >= B) break;
                    float hv[V];
#pragma unroll
                    for (int e4 = 0; e4 < V / 4; ++e4) {
                        const float4 t = reinterpret_cast<const float4 *>(hs + (size_t)b * r + (size_t)q * V)[e4];
                        hv[4 * e4] = t.x; hv[4 * e4 + 1] = t.y; hv[4 * e4 + 2] = t.z; hv[4 * e4 + 3] = t.w;
                    }
#pragma unroll
                    for (int p = 0; p < NPW; ++p) {
                        float wf[V];
                        unpack<PT>(wv[p][u], wf);
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[p][b] = fmaf(wf[e], hv[e], acc[p][b]);
                    }
                }
            }
        }
#pragma unroll
        for (int p = 0; p < NPW; ++p) {
            const int i = nb + p;
            const float bias = (i < n1 && a.b_pred) ? __ldg(a.b_pred + i) : 0.f;
            bool act = false;
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                const float z = warp_sum(acc[p][b]) + bias;
                act = act || (b < B && z > a.tau);
            }
            if (lane == 0 && i < n1 && (i < a.hot || act)) atomicOr(&sword[(i >> 5) - w0], 1u << (i & 31));
        }
    }
    __syncthreads();
    for (int i = tid; i < w1 - w0; i += FP_NT) a.maskw[w0 + i] = sword[i];
    __syncthreads();
    if (tid == 0) s_last = ticket_acq_rel(a.ticket, 1u) == (unsigned)P - 1u;
    __syncthreads();
    if (!s_last) return;
    compact_words<FW>(a.maskw, W, 0, a.idx, a.count, wsum, [] { __syncthreads(); });
    if (tid == 0) *a.ticket = 0u;
}

// ---------------------------------------------------------------- launchers ------------------

template <int PT>
static cudaError_t hidden_bt(const Launch &L, int bt, const void *p1t, int d, int r, const float *x,
                             const float *inv_rms, int B, float *hp)
{
    auto go = [&](auto kern) {
        cudaError_t e = ensure_smem(kern, L.smem);
        return e != cudaSuccess ? e : launch_ex(L, kern, (const uint4 *)p1t, d, r, x, inv_rms, B, hp);
    };
    switch (bt) {
    case 1: return go(k_pred_hidden<PT, 1>);
    case 2: return go(k_pred_hidden<PT, 2>);
    case 4: return go(k_pred_hidden<PT, 4>);
    case 8: return go(k_pred_hidden<PT, 8>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_pred_hidden(const Launch &L, int pdt, int bt, const void *p1t, int d, int r,
                               const float *x, const float *inv_rms, int B, float *hp)
{
    switch (pdt) {
    case DT_F32: return hidden_bt<DT_F32>(L, bt, p1t, d, r, x, inv_rms, B, hp);
    case DT_BF16: return hidden_bt<DT_BF16>(L, bt, p1t, d, r, x, inv_rms, B, hp);
    case DT_F16: return hidden_bt<DT_F16>(L, bt, p1t, d, r, x, inv_rms, B, hp);
    }
    return cudaErrorInvalidValue;
}

template <int PT>
static cudaError_t logits_bt(const Launch &L, int bt, const void *p2t, int r, int f, const float *b_pred,
                             float tau, const float *hp, int B, uint32_t *maskw, uint32_t *ticket,
                             int32_t *idx, int32_t *count, int hot)
{
    auto go = [&](auto kern) {
        cudaError_t e = ensure_smem(kern, L.smem);
        return e != cudaSuccess ? e
                                : launch_ex(L, kern, (const uint4 *)p2t, r, f, b_pred, tau, hp, B, maskw, ticket,
                                            idx, count, hot);
    };
    switch (bt) {
    case 1: return go(k_pred_logits<PT, 1>);
    case 2: return go(k_pred_logits<PT, 2>);
    case 4: return go(k_pred_logits<PT, 4>);
    case 8: return go(k_pred_logits<PT, 8>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_pred_logits(const Launch &L, int pdt, int bt, const void *p2t, int r, int f,
                               const float *b_pred, float tau, const float *hp, int B,
                               uint32_t *maskw, uint32_t *ticket, int32_t *idx, int32_t *count, int hot)
{
    switch (pdt) {
    case DT_F32: return logits_bt<DT_F32>(L, bt, p2t, r, f, b_pred, tau, hp, B, maskw, ticket, idx, count, hot);
    case DT_BF16: return logits_bt<DT_BF16>(L, bt, p2t, r, f, b_pred, tau, hp, B, maskw, ticket, idx, count, hot);
    case DT_F16: return logits_bt<DT_F16>(L, bt, p2t, r, f, b_pred, tau, hp, B, maskw, ticket, idx, count, hot);
    }
    return cudaErrorInvalidValue;
}

template <int PT>
static cudaError_t fused_bt(int bt, const FusedPredArgs &a, int grid, size_t smem, cudaStream_t s)
{
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, FP_NT, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorNotSupported;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(FP_NT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a);
    };
    switch (bt) {
    case 2: return go(k_pred_fused<PT, 2>);
    case 4: return go(k_pred_fused<PT, 4>);
    case 8: return go(k_pred_fused<PT, 8>);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_pred_fused(int pdt, int bt, const FusedPredArgs &a, int grid, size_t smem, cudaStream_t s)
{
    switch (pdt) {
    case DT_F32: return fused_bt<DT_F32>(bt, a, grid, smem, s);
    case DT_BF16: return fused_bt<DT_BF16>(bt, a, grid, smem, s);
    case DT_F16: return fused_bt<DT_F16>(bt, a, grid, smem, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pi
