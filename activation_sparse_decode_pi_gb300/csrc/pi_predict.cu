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
        __threadfence();
        last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    __shared__ int wsum[NW];
    compact_words<NW>(maskw, gridDim.x, 0, idx, count, wsum, [] { __syncthreads(); });
    if (threadIdx.x == 0) *ticket = 0u;
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

}  // namespace pi
