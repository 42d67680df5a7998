// pi_rowdot.cuh -- dot products of several weight rows with a small batch of fp32 vectors.
//
// Used by the predictor (dense rows) and by the gate/up gather (rows picked by
// the active list). Each lane walks 16-byte chunks of its rows with a stride of
// 32 chunks and keeps RW rows x U chunks of loads in flight; the fp32 vectors
// live in shared memory in a *planar* layout so that lane-consecutive chunk
// reads are conflict-free:  float4 plane q of chunk ci of batch row b sits at
//   su4[b * K/4 + q * nch + ci],   nch = K / V,  q < V/4.
#pragma once

#include "pi_common.cuh"

namespace pi {

template <int DT, int RW, int U>
struct RowChunks {
    uint4 w[RW][U];
    float s[RW][U];  // group scale of the chunk (int4 only)
};

// Issue the loads of chunks c, c+32, ..., c+32(U-1) (< ce) of each row.
template <int DT, int RW, int U>
__device__ __forceinline__ void rows_issue(RowChunks<DT, RW, U> &rc, const uint4 *const (&row)[RW],
                                           const __half *const (&srow)[RW], int c, int ce)
{
#pragma unroll
    for (int i = 0; i < U; ++i) {
        const int ci = c + 32 * i;
#pragma unroll
        for (int k = 0; k < RW; ++k) {
            const bool ok = ci < ce && row[k] != nullptr;
            rc.w[k][i] = ok ? ld_stream(row[k] + ci) : make_uint4(0u, 0u, 0u, 0u);
            if (DT == DT_INT4) rc.s[k][i] = ok ? ld_scale(srow[k] + (ci >> 2)) : 0.f;
        }
    }
}

// acc[k][b] += row_k[chunk] . u_b[chunk] for the chunks held in rc.
template <int DT, int RW, int U, int BT>
__device__ __forceinline__ void rows_consume(const RowChunks<DT, RW, U> &rc, int c, int ce,
                                             const float4 *__restrict__ su4, int K, float (&acc)[RW][BT])
{
    constexpr int V = Vec<DT>::N;
    constexpr int Q = V / 4;
    const int nch = K / V;
#pragma unroll
    for (int i = 0; i < U; ++i) {
        const int ci = c + 32 * i;
        if (ci >= ce) continue;
        if constexpr (DT == DT_INT4) {
            float part[RW][BT];
#pragma unroll
            for (int k = 0; k < RW; ++k)
#pragma unroll
                for (int b = 0; b < BT; ++b) part[k][b] = 0.f;
            const uint32_t *wk[RW];
#pragma unroll
            for (int k = 0; k < RW; ++k) wk[k] = reinterpret_cast<const uint32_t *>(&rc.w[k][i]);
#pragma unroll
            for (int a = 0; a < 4; ++a) {        // 32-bit word a holds elements 8a .. 8a+7
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    const float4 u0 = su4[b * (K / 4) + (2 * a) * nch + ci];
                    const float4 u1 = su4[b * (K / 4) + (2 * a + 1) * nch + ci];
                    const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int k = 0; k < RW; ++k) {
                        const uint32_t w = wk[k][a];
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[k][b] = fmaf(nib(w, e), uu[e], part[k][b]);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < RW; ++k)
#pragma unroll
                for (int b = 0; b < BT; ++b) acc[k][b] = fmaf(rc.s[k][i], part[k][b], acc[k][b]);
        } else if constexpr (RW > BT) {
            // more rows than batch rows: hold the chunk of u, stream the rows through one at a time
            float uv[BT][V];
#pragma unroll
            for (int b = 0; b < BT; ++b)
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const float4 u = su4[b * (K / 4) + q * nch + ci];
                    uv[b][4 * q + 0] = u.x;
                    uv[b][4 * q + 1] = u.y;
                    uv[b][4 * q + 2] = u.z;
                    uv[b][4 * q + 3] = u.w;
                }
#pragma unroll
            for (int k = 0; k < RW; ++k) {
                float wf[V];
                unpack<DT>(rc.w[k][i], wf);
#pragma unroll
                for (int b = 0; b < BT; ++b) {
                    float a = acc[k][b];
#pragma unroll
                    for (int e = 0; e < V; ++e) a = fmaf(wf[e], uv[b][e], a);
                    acc[k][b] = a;
                }
            }
        } else {
            float wf[RW][V];
#pragma unroll
            for (int k = 0; k < RW; ++k) unpack<DT>(rc.w[k][i], wf[k]);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const float4 u = su4[b * (K / 4) + q * nch + ci];
#pragma unroll
                    for (int k = 0; k < RW; ++k) {
                        float a = acc[k][b];
                        a = fmaf(wf[k][4 * q + 0], u.x, a);
                        a = fmaf(wf[k][4 * q + 1], u.y, a);
                        a = fmaf(wf[k][4 * q + 2], u.z, a);
                        a = fmaf(wf[k][4 * q + 3], u.w, a);
                        acc[k][b] = a;
                    }
                }
            }
        }
    }
}

// Stage bt (<= BT) rows of a [*, K] fp32 matrix, times an optional per-row scale,
// into the planar layout. Rows bt..BT-1 are zero-filled. Reads bypass L1 (the
// vector was written by the previous kernel).
template <int DT, int BT>
__device__ __forceinline__ void stage_planar(float4 *__restrict__ su4, const float *__restrict__ src, int K, int bt,
                                             const float *__restrict__ row_scale)
{
    constexpr int Q = Vec<DT>::N / 4;
    const int nch = K / Vec<DT>::N;
    const int k4 = K / 4;
    for (int t = threadIdx.x; t < BT * k4; t += blockDim.x) {
        const int b = t / k4, j = t - b * k4;       // float4 j of row b
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < bt) {
            v = __ldcg(reinterpret_cast<const float4 *>(src + (size_t)b * K) + j);
            if (row_scale) {
                const float s = __ldcg(row_scale + b);
                v.x *= s; v.y *= s; v.z *= s; v.w *= s;
            }
        }
        const int ci = j / Q, q = j - ci * Q;
        su4[b * k4 + q * nch + ci] = v;
    }
}

}  // namespace pi
