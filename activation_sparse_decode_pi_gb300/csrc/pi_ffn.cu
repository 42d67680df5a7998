// pi_ffn.cu -- neuron-sparse FFN kernels (sm_103a, CUDA cores).
//
// "PowerInfer" paper walk-through page, section "technical details":
// FFN(x) = sigma(x W1) (.) (x W2) W3 with sigma = ReLU; the summary page
// (Methodology) computes it with neuron-aware sparse operators, i.e. only the
// neurons the predictor marked are touched:
//   K3   gate/up gather-GEMV: h[b,j] = ReLU(u_b . Wg_i + bg_i) * (u_b . Wu_i), i = idx[j]
//        (non-gated: ReLU(u_b . W1_i + b1_i)). Rows are 16-byte vector loads,
//        u is staged in shared memory, warp-shuffle + fixed-order CTA reduction.
//   K4a  row-sparse W_down axpy: part[g,b,:] = sum_{j in group g} h[b,j] * WdT[idx_j,:]
//        fp32 accumulators in registers, each thread owning a fixed column chunk.
//   K4b  deterministic reduction y = sum_g part[g] in a fixed order; in the layer
//        stack it also applies the residual and the next layer's RMS scale.
// The group size depends only on the active count, never on the GPU, so the
// result's bits depend only on the inputs.
#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_rowdot.cuh"

namespace pi {

__device__ __forceinline__ int clamp_count(const int32_t *count, int f, uint32_t *status)
{
    int n = __ldcg(count);
    if (n < 0 || n > f) {
        set_status(status, ST_DEVICE_CHECK);
        n = n < 0 ? 0 : f;
    }
    return n;
}

// ---------------------------------------------------------------- K3 -------------------------
template <int WT, int KIND, int BT>
__global__ void __launch_bounds__(NT, 2)
k_ffn_h(const uint4 *__restrict__ Wg, const uint4 *__restrict__ Wu, const __half *__restrict__ Sg,
        const __half *__restrict__ Su, const float *__restrict__ bg, int d, int f,
        const float *__restrict__ x, const float *__restrict__ inv_rms, int B,
        const int32_t *__restrict__ idx, const int32_t *__restrict__ count, float *__restrict__ h, int ldh,
        uint32_t *__restrict__ status)
{
    constexpr int RW = 4, U = (WT == DT_INT4) ? 2 : 4, V = Vec<WT>::N;
    constexpr int NPI = KIND == KIND_GATED ? RW / 2 : RW;   // neurons per CTA iteration
    extern __shared__ float4 su4[];                        // [BT][d/4] planar
    __shared__ float red[NW][RW][BT];
    __shared__ int sidx[NPI];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = d / V;
    const int per = (nch + NW - 1) / NW;
    const int cb = warp * per, ce = min(nch, cb + per);
    const int gpr = d / 128;                               // int4 groups per row

    pdl_launch_dependents();
    pdl_wait();
    const int n = clamp_count(count, f, status);
    const int nblk = (n + NPI - 1) / NPI;
    if ((int)blockIdx.x >= nblk) return;

    for (int b0 = 0; b0 < B; b0 += BT) {
        const int bt = min(BT, B - b0);
        __syncthreads();
        stage_planar<WT, BT>(su4, x + (size_t)b0 * d, d, bt, inv_rms ? inv_rms + b0 : nullptr);
        for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
            if (threadIdx.x < NPI) {
                const int j = blk * NPI + threadIdx.x;
                int i = -1;
                if (j < n) {
                    i = __ldcg(idx + j);
                    if (i < 0 || i >= f) {
                        set_status(status, ST_DEVICE_CHECK);
                        i = -1;
                    }
                }
                sidx[threadIdx.x] = i;
            }
            __syncthreads();
            const uint4 *row[RW];
            const __half *srow[RW];
#pragma unroll
            for (int k = 0; k < RW; ++k) {
                const int q = KIND == KIND_GATED ? k >> 1 : k;
                const int i = sidx[q];
                const bool up = KIND == KIND_GATED && (k & 1);
                row[k] = i >= 0 ? (up ? Wu : Wg) + (size_t)i * nch : nullptr;
                srow[k] = (WT == DT_INT4 && i >= 0) ? (up ? Su : Sg) + (size_t)i * gpr : nullptr;
            }
            RowChunks<WT, RW, U> rc;
            float acc[RW][BT];
#pragma unroll
            for (int k = 0; k < RW; ++k)
#pragma unroll
                for (int b = 0; b < BT; ++b) acc[k][b] = 0.f;
            rows_issue(rc, row, srow, cb + lane, ce);
            for (int c = cb + lane;;) {
                rows_consume<WT, RW, U, BT>(rc, c, ce, su4, d, acc);
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
            if (threadIdx.x < NPI * BT) {
                const int q = threadIdx.x / BT, b = threadIdx.x - q * BT;
                const int j = blk * NPI + q;
                const int i = sidx[q];
                if (j < n && b < bt) {
                    float hv = 0.f;
                    if (i >= 0) {
                        const int kg = KIND == KIND_GATED ? 2 * q : q;
                        float g = 0.f;
#pragma unroll
                        for (int w = 0; w < NW; ++w) g += red[w][kg][b];   // fixed order
                        g += bg ? __ldg(bg + i) : 0.f;
                        hv = fmaxf(g, 0.f);
                        if (KIND == KIND_GATED) {
                            float u = 0.f;
#pragma unroll
                            for (int w = 0; w < NW; ++w) u += red[w][kg + 1][b];
                            hv *= u;
                        }
                    }
                    h[(size_t)(b0 + b) * ldh + j] = hv;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------- K4a ------------------------
template <int WT, int BT>
__global__ void __launch_bounds__(NT)
k_ffn_down(const uint4 *__restrict__ Wd, const __half *__restrict__ Sd, int d, int f,
           const int32_t *__restrict__ idx, const int32_t *__restrict__ count, const float *__restrict__ h,
           int ldh, int B, float *__restrict__ part, uint32_t *__restrict__ status)
{
    constexpr int V = Vec<WT>::N, U = (WT == DT_INT4) ? 4 : 8, SUB = 32;
    __shared__ int sidx[SUB];
    __shared__ float sh[BT][SUB];

    const int nch = d / V;
    const int ncb = (nch + NT - 1) / NT;
    const int gpr = d / 128;

    pdl_launch_dependents();
    pdl_wait();
    const int n = clamp_count(count, f, status);
    const int G = down_group_size(n);
    const int ngroups = (n + G - 1) / G;
    const int tasks = ngroups * ncb;

    for (int task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int g = task / ncb;
        const int c = (task - g * ncb) * NT + threadIdx.x;
        const bool cok = c < nch;
        const int j0 = g * G, j1 = min(n, j0 + G);
        for (int b0 = 0; b0 < B; b0 += BT) {
            const int bt = min(BT, B - b0);
            float acc[BT][V];
#pragma unroll
            for (int b = 0; b < BT; ++b)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[b][e] = 0.f;
            for (int js = j0; js < j1; js += SUB) {
                const int jn = min(SUB, j1 - js);
                __syncthreads();
                if (threadIdx.x < SUB) {
                    int i = -1;
                    if ((int)threadIdx.x < jn) {
                        i = __ldcg(idx + js + threadIdx.x);
                        if (i < 0 || i >= f) i = -1;
                    }
                    sidx[threadIdx.x] = i;
                }
                for (int t = threadIdx.x; t < BT * SUB; t += NT) {
                    const int b = t / SUB, q = t - b * SUB;
                    sh[b][q] = (q < jn && b < bt) ? __ldcg(h + (size_t)(b0 + b) * ldh + js + q) : 0.f;
                }
                __syncthreads();
                for (int q0 = 0; q0 < jn; q0 += U) {
                    uint4 w[U];
                    float s[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int q = q0 + u;
                        const int i = q < jn ? sidx[q] : -1;
                        const bool ok = cok && i >= 0;
                        w[u] = ok ? ld_stream(Wd + (size_t)i * nch + c) : make_uint4(0u, 0u, 0u, 0u);
                        if (WT == DT_INT4) s[u] = ok ? ld_scale(Sd + (size_t)i * gpr + (c >> 2)) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int q = q0 + u;
                        if (q >= jn) break;
                        if constexpr (WT == DT_INT4) {
                            const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                            for (int a = 0; a < 4; ++a)
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float wv = nib(ww[a], e) * s[u];
#pragma unroll
                                    for (int b = 0; b < BT; ++b) acc[b][8 * a + e] = fmaf(sh[b][q], wv, acc[b][8 * a + e]);
                                }
                        } else {
                            float wf[V];
                            unpack<WT>(w[u], wf);
#pragma unroll
                            for (int b = 0; b < BT; ++b) {
                                const float hb = sh[b][q];
#pragma unroll
                                for (int e = 0; e < V; ++e) acc[b][e] = fmaf(hb, wf[e], acc[b][e]);
                            }
                        }
                    }
                }
            }
            if (cok) {
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    if (b >= bt) break;
                    float4 *dst = reinterpret_cast<float4 *>(part + ((size_t)g * B + b0 + b) * d + (size_t)c * V);
#pragma unroll
                    for (int e = 0; e < V / 4; ++e)
                        dst[e] = make_float4(acc[b][4 * e], acc[b][4 * e + 1], acc[b][4 * e + 2], acc[b][4 * e + 3]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- K4b ------------------------
// grid (ceil(d/RED_COLS), B). Warp w adds groups w, w+8, ... in order; the 8 warp sums
// are then added in warp order.
template <bool GLUE>
__global__ void __launch_bounds__(NT)
k_reduce(const float *__restrict__ part, int d, int B, int f, const int32_t *__restrict__ count,
         const float *__restrict__ xin, float *__restrict__ out, float *__restrict__ sumsq,
         uint32_t *__restrict__ ticket, float *__restrict__ inv_rms, float eps)
{
    static_assert(RED_COLS == 4 * 32, "one float4 per lane");
    __shared__ float4 red[NW][32];
    __shared__ bool last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int col4 = blockIdx.x * 32 + lane;
    const int d4 = d / 4;
    const bool ok = col4 < d4;

    pdl_launch_dependents();
    pdl_wait();
    const int n = clamp_count(count, f, nullptr);
    const int G = down_group_size(n);
    const int ngroups = (n + G - 1) / G;

    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
#pragma unroll 4
        for (int g = warp; g < ngroups; g += NW) {
            const float4 v = __ldcg(p4 + ((size_t)g * B + b) * d4 + col4);
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0) {
        float4 y = red[0][lane];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
            const float4 v = red[w][lane];
            y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
        }
        float ss = 0.f;
        if (GLUE && ok) {
            const float4 xv = __ldcg(reinterpret_cast<const float4 *>(xin) + (size_t)b * d4 + col4);
            y.x += xv.x; y.y += xv.y; y.z += xv.z; y.w += xv.w;
            ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
        }
        if (ok) reinterpret_cast<float4 *>(out)[(size_t)b * d4 + col4] = y;
        if (GLUE) {
            ss = warp_sum(ss);
            if (lane == 0) sumsq[(size_t)b * gridDim.x + blockIdx.x] = ss;
        }
    }
    if (!GLUE) return;
    __syncthreads();
    if (threadIdx.x == 0) last = ticket_acq_rel(ticket, 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!last) return;
    for (int bb = warp; bb < B; bb += NW) {
        float t = 0.f;
        for (int k = lane; k < (int)gridDim.x; k += 32) t += __ldcg(sumsq + (size_t)bb * gridDim.x + k);
        t = warp_sum(t);
        if (lane == 0) inv_rms[bb] = 1.0f / sqrtf(t / (float)d + eps);
    }
    if (threadIdx.x == 0) *ticket = 0u;
}

// ---------------------------------------------------------------- RMS of the stack input ----
__global__ void __launch_bounds__(NT) k_rms(const float *__restrict__ x, int d, float *__restrict__ inv_rms, float eps)
{
    __shared__ float ws[NW];
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();
    float t = 0.f;
    for (int i = threadIdx.x; i < d; i += NT) {
        const float v = __ldcg(x + (size_t)b * d + i);
        t = fmaf(v, v, t);
    }
    t = warp_sum(t);
    if (lane == 0) ws[warp] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < NW; ++w) s += ws[w];
        inv_rms[b] = 1.0f / sqrtf(s / (float)d + eps);
    }
}

// ---------------------------------------------------------------- launchers ------------------

template <int WT, int KIND>
static cudaError_t ffn_h_bt(const Launch &L, int bt, const void *wg, const void *wu, const void *sg,
                            const void *su, const float *bg, int d, int f, const float *x, const float *inv_rms,
                            int B, const int32_t *idx, const int32_t *count, float *h, int ldh, uint32_t *status)
{
    auto go = [&](auto kern) {
        cudaError_t e = ensure_smem(kern, L.smem);
        return e != cudaSuccess ? e
                                : launch_ex(L, kern, (const uint4 *)wg, (const uint4 *)wu, (const __half *)sg,
                                            (const __half *)su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    };
    switch (bt) {
    case 1: return go(k_ffn_h<WT, KIND, 1>);
    case 2: return go(k_ffn_h<WT, KIND, 2>);
    case 4: return go(k_ffn_h<WT, KIND, 4>);
    case 8: return go(k_ffn_h<WT, KIND, 8>);
    }
    return cudaErrorInvalidValue;
}

template <int WT>
static cudaError_t ffn_h_kind(const Launch &L, int kind, int bt, const void *wg, const void *wu, const void *sg,
                              const void *su, const float *bg, int d, int f, const float *x, const float *inv_rms,
                              int B, const int32_t *idx, const int32_t *count, float *h, int ldh, uint32_t *status)
{
    if (kind == KIND_GATED)
        return ffn_h_bt<WT, KIND_GATED>(L, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    return ffn_h_bt<WT, KIND_RELU>(L, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
}

cudaError_t launch_ffn_h(const Launch &L, int wdt, int kind, int bt, const void *wg, const void *wu,
                         const void *sg, const void *su, const float *bg, int d, int f,
                         const float *x, const float *inv_rms, int B,
                         const int32_t *idx, const int32_t *count, float *h, int ldh, uint32_t *status)
{
    switch (wdt) {
    case DT_F32: return ffn_h_kind<DT_F32>(L, kind, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    case DT_BF16: return ffn_h_kind<DT_BF16>(L, kind, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    case DT_F16: return ffn_h_kind<DT_F16>(L, kind, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    case DT_INT4: return ffn_h_kind<DT_INT4>(L, kind, bt, wg, wu, sg, su, bg, d, f, x, inv_rms, B, idx, count, h, ldh, status);
    }
    return cudaErrorInvalidValue;
}

template <int WT>
static cudaError_t down_bt(const Launch &L, int bt, const void *wd, const void *sd, int d, int f, const int32_t *idx,
                           const int32_t *count, const float *h, int ldh, int B, float *part, uint32_t *status)
{
    auto go = [&](auto kern) {
        return launch_ex(L, kern, (const uint4 *)wd, (const __half *)sd, d, f, idx, count, h, ldh, B, part, status);
    };
    switch (bt) {
    case 1: return go(k_ffn_down<WT, 1>);
    case 2: return go(k_ffn_down<WT, 2>);
    case 4: if constexpr (WT != DT_INT4) return go(k_ffn_down<WT, 4>); break;
    case 8: if constexpr (WT != DT_INT4) return go(k_ffn_down<WT, 8>); break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_ffn_down(const Launch &L, int wdt, int bt, const void *wd, const void *sd, int d, int f,
                            const int32_t *idx, const int32_t *count, const float *h, int ldh, int B,
                            float *part, uint32_t *status)
{
    switch (wdt) {
    case DT_F32: return down_bt<DT_F32>(L, bt, wd, sd, d, f, idx, count, h, ldh, B, part, status);
    case DT_BF16: return down_bt<DT_BF16>(L, bt, wd, sd, d, f, idx, count, h, ldh, B, part, status);
    case DT_F16: return down_bt<DT_F16>(L, bt, wd, sd, d, f, idx, count, h, ldh, B, part, status);
    case DT_INT4: return down_bt<DT_INT4>(L, bt, wd, sd, d, f, idx, count, h, ldh, B, part, status);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(const Launch &L, const float *part, int d, int B, int f, const int32_t *count,
                          const float *xin, float *out, float *sumsq, uint32_t *ticket, float *inv_rms, float eps)
{
    if (xin) return launch_ex(L, k_reduce<true>, part, d, B, f, count, xin, out, sumsq, ticket, inv_rms, eps);
    return launch_ex(L, k_reduce<false>, part, d, B, f, count, xin, out, sumsq, ticket, inv_rms, eps);
}

cudaError_t launch_rms(const Launch &L, const float *x, int d, int B, float *inv_rms, float eps)
{
    (void)B;
    return launch_ex(L, k_rms, x, d, inv_rms, eps);
}

}  // namespace pi
