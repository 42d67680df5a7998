// pi_stack.cuh -- one decode step through every layer in a single persistent kernel (batch 1).
//
// "PowerInfer" paper walk-through page, section "inference flow": the input reaches
// a layer, the predictor marks the neurons that will fire, only those are computed,
// the result is merged and passed to the next layer. Here every SM runs one CTA of
// 512 threads that walks all layers; the dependent steps of a layer are separated
// by four bounded grid barriers:
//
//   A  hp[k] = ReLU(u . P1T[k])           CTA c: hidden units [c*r/P, (c+1)*r/P)
//   -- barrier
//   B  z[i] = hp . P2T[i] + b_p[i] > tau   CTA c: neurons [c*f/P, (c+1)*f/P) -> mask bits
//   -- barrier
//   C  active list = set bits of the mask, cut into NCHUNK fixed chunks of consecutive
//      list entries; for each neuron of its chunk a CTA bulk-copies the gate(/up) and
//      W_down rows into a shared-memory ring (cp.async.bulk + mbarrier), reduces
//      h = ReLU(u.Wg + bg) * (u.Wu) over the CTA, and accumulates h * WdT into fp32
//      registers (each thread owns fixed columns). One fp32 partial per chunk.
//   -- barrier
//   D  x_{l+1} = x_l + sum over the chunk partials in a fixed order, per 32-column slice,
//      plus that slice's sum of squares for the next layer's RMS scale.
//   -- barrier
//
// The predictor weights do not depend on the input, so each CTA fetches its slice of
// the next layer's predictor while the current layer is still running: its P1 rows
// are loaded into registers before the last barrier of the layer, and its P2 rows
// (and the rest of its P1 rows) are prefetched into L2 at the start of the layer.
// The HBM stream thus continues across the barriers.
// The chunking depends only on the active count, so the bits of the result do not
// depend on the number of SMs.
#pragma once

#include "pi_async.cuh"
#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_rowdot.cuh"

namespace pi {

constexpr int SNW = STACK_NT / 32;

template <int WT>
__host__ __device__ constexpr int weight_row_bytes(int d)
{
    return WT == DT_F32 ? d * 4 : (WT == DT_INT4 ? d / 2 : d * 2);
}

// j-th set bit (0-based) of the mask words, given their exclusive popcount prefix.
__device__ __forceinline__ int select_active(const uint32_t *words, const int *pre, int W, int j)
{
    int lo = 0, hi = W - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= j) lo = mid;
        else hi = mid - 1;
    }
    uint32_t m = words[lo];
    for (int k = j - pre[lo]; k > 0; --k) m &= m - 1;
    return lo * 32 + __ffs(m) - 1;
}

template <int WT, int PT, int KIND>
__global__ void __launch_bounds__(STACK_NT, 1) k_decode_stack(const StackArgs a)
{
    constexpr int VW = Vec<WT>::N;
    constexpr int CPT = (WT == DT_INT4) ? 1 : 3;            // weight chunks per thread per row (max)
    constexpr int ROWS = KIND == KIND_GATED ? 3 : 2;         // rows staged per neuron
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem + a.off_ring;                 // phase C: row slots
    uint32_t *swords = reinterpret_cast<uint32_t *>(smem + a.off_words);
    int *spre = reinterpret_cast<int *>(smem + a.off_pre);
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + a.off_mbar);   // [S] row slots
    float4 *ua4 = reinterpret_cast<float4 *>(smem + a.off_ua);         // phase A: u (planar, predictor type)
    float4 *hp4 = reinterpret_cast<float4 *>(smem + a.off_hp);         // phase B: hp (planar)
    float4 *scr4 = reinterpret_cast<float4 *>(smem + a.off_scr);       // phase D: partial sums

    __shared__ float red[2][SNW][8];
    __shared__ unsigned long long s_base;
    __shared__ int wsum[SNW];
    __shared__ int sneur[STACK_MAX_CHUNK];
    __shared__ uint32_t sbits[STACK_MAX_BITWORDS];
    __shared__ float s_inv;
    __shared__ int s_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x;
    const int d = a.d, f = a.f, r = a.r, S = a.slots;
    const int W = (f + 31) >> 5;
    const int nchw = d / VW;
    const int rowb = weight_row_bytes<WT>(d);
    const int sclb = WT == DT_INT4 ? (d / 128) * 2 : 0;
    const int pb = PT == DT_F32 ? 4 : 2;
    const int k0 = (int)((long long)c * r / P), k1 = (int)((long long)(c + 1) * r / P);
    const int i0 = (int)((long long)c * f / P), i1 = (int)((long long)(c + 1) * f / P);
    uint32_t seq = 0;   // neurons staged by this CTA so far: slot seq % S, phase (seq / S) & 1
    unsigned kb = 0;    // grid barriers passed in this launch
    auto sync_grid = [&]() -> bool {
        ++kb;
        return grid_sync_to(a.bar, s_base + (unsigned long long)kb * a.nblocks, a.status, &s_flag);
    };
    // first chunk of this CTA's P1 rows (one per lane and row) into registers
    constexpr int VPA = Vec<PT>::N;
    const int nchp = d / VPA;
    const int pa_per = (nchp + SNW - 1) / SNW, pa_cb = warp * pa_per, pa_ce = min(nchp, pa_cb + pa_per);
    RowChunks<PT, 8, 1> pa;
    auto load_p1 = [&](const StackLayer &L) {
        const uint4 *row[8];
        const __half *srow[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            row[k] = k0 + k < k1 ? reinterpret_cast<const uint4 *>(L.p1) + (size_t)(k0 + k) * nchp : nullptr;
            srow[k] = nullptr;
        }
        rows_issue(pa, row, srow, pa_cb + lane, pa_ce);
    };

    // the parts of this CTA's predictor slice that are not staged otherwise, into L2
    auto prefetch_predictor = [&](const StackLayer &L) {
        const size_t per_cta = (size_t)(a.pf_bytes / P);
        const size_t b1 = (size_t)(k1 - k0) * d * pb;
        prefetch_l2_range((const char *)L.p1 + (size_t)k0 * d * pb, b1 < per_cta ? b1 : per_cta);
        const size_t b2 = (size_t)(i1 - i0) * r * pb;
        const size_t left = per_cta > b1 ? per_cta - b1 : 0;
        prefetch_l2_range((const char *)L.p2 + (size_t)i0 * r * pb, b2 < left ? b2 : left);
    };

    // ---------------------------------------------------------------- phase 0
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 1);
        fence_mbar_init();
        s_base = barrier_base(a.bar, (unsigned long long)(4 * a.L) * a.nblocks);
        prefetch_predictor(a.layers[0]);
    }
    load_p1(a.layers[0]);
    for (int i = c * STACK_NT + tid; i < a.L * W; i += P * STACK_NT) a.maskw[i] = 0u;
    {
        float t = 0.f;
        for (int i = tid; i < d; i += STACK_NT) {
            const float v = __ldcg(a.x0 + i);
            t = fmaf(v, v, t);
        }
        t = warp_sum(t);
        if (lane == 0) red[0][warp][0] = t;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < SNW; ++w) s += red[0][w][0];
            s_inv = 1.0f / sqrtf(s / (float)d + a.eps);
        }
    }
    if (!sync_grid()) return;

    for (int l = 0; l < a.L; ++l) {
        const StackLayer Lw = a.layers[l];
        const float *xl = l == 0 ? a.x0 : (((l - 1) & 1) ? a.xb : a.xa);
        float *xn = l == a.L - 1 ? a.x_out : ((l & 1) ? a.xb : a.xa);
        if (tid == 0 && l + 1 < a.L) prefetch_predictor(a.layers[l + 1]);
        const float inv = s_inv;

        // ------------------------------------------------------------ A: predictor hidden layer
        {
            constexpr int QP = VPA / 4;
            for (int t = tid; t < d / 4; t += STACK_NT) {
                float4 v = __ldcg(reinterpret_cast<const float4 *>(xl) + t);
                v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
                const int ci = t / QP, q = t - ci * QP;
                ua4[q * nchp + ci] = v;
            }
            __syncthreads();
            const uint4 *row[8];
            const __half *srow[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                row[k] = k0 + k < k1 ? reinterpret_cast<const uint4 *>(Lw.p1) + (size_t)(k0 + k) * nchp : nullptr;
                srow[k] = nullptr;
            }
            float acc[8][1];
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k][0] = 0.f;
            rows_consume<PT, 8, 1, 1>(pa, pa_cb + lane, pa_ce, ua4, d, acc);   // loaded before the barrier
            for (int cc = pa_cb + lane + 32; cc < pa_ce; cc += 32) {
                rows_issue(pa, row, srow, cc, pa_ce);
                rows_consume<PT, 8, 1, 1>(pa, cc, pa_ce, ua4, d, acc);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float sm_ = warp_sum(acc[k][0]);
                if (lane == 0) red[0][warp][k] = sm_;
            }
            __syncthreads();
            if (tid < 8 && k0 + tid < k1) {
                float sm_ = 0.f;
                for (int w = 0; w < SNW; ++w) sm_ += red[0][w][tid];   // fixed order
                a.hp[k0 + tid] = fmaxf(sm_, 0.f);
            }
        }
        if (!sync_grid()) return;

        // ------------------------------------------------------------ B: logits and mask bits
        {
            constexpr int VP = Vec<PT>::N;
            const int nchr = r / VP;
            stage_planar<PT, 1>(hp4, a.hp, r, 1, nullptr);
            const int w0 = i0 >> 5;
            for (int t = tid; t < STACK_MAX_BITWORDS; t += STACK_NT) sbits[t] = 0u;
            __syncthreads();
            for (int base = i0 + warp; base < i1; base += SNW * 4) {
                const uint4 *row[4];
                const __half *srow[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = base + SNW * k;
                    row[k] = i < i1 ? reinterpret_cast<const uint4 *>(Lw.p2) + (size_t)i * nchr : nullptr;
                    srow[k] = nullptr;
                }
                RowChunks<PT, 4, 4> rc;
                float acc[4][1] = {{0.f}, {0.f}, {0.f}, {0.f}};
                rows_issue(rc, row, srow, lane, nchr);
                for (int cc = lane;;) {
                    rows_consume<PT, 4, 4, 1>(rc, cc, nchr, hp4, r, acc);
                    cc += 32 * 4;
                    if (cc >= nchr) break;
                    rows_issue(rc, row, srow, cc, nchr);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = base + SNW * k;
                    const float z = warp_sum(acc[k][0]) + ((i < i1 && Lw.bp) ? __ldg(Lw.bp + i) : 0.f);
                    if (lane == 0 && i < i1 && z > a.tau) atomicOr(&sbits[(i >> 5) - w0], 1u << (i & 31));
                }
            }
            __syncthreads();
            if (i1 > i0)
                for (int w = tid; w <= ((i1 - 1) >> 5) - w0; w += STACK_NT)
                    if (sbits[w]) atomicOr(a.maskw + (size_t)l * W + w0 + w, sbits[w]);
        }
        if (!sync_grid()) return;

        // ------------------------------------------------------------ C: sparse FFN over the mask
        {
            // this thread's columns of u, scaled (issued first: independent of the mask)
            float ur[CPT][VW];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                const int ci = tid + cc * STACK_NT;
#pragma unroll
                for (int e4 = 0; e4 < VW / 4; ++e4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ci < nchw) v = __ldcg(reinterpret_cast<const float4 *>(xl + (size_t)ci * VW) + e4);
                    ur[cc][4 * e4 + 0] = v.x * inv;
                    ur[cc][4 * e4 + 1] = v.y * inv;
                    ur[cc][4 * e4 + 2] = v.z * inv;
                    ur[cc][4 * e4 + 3] = v.w * inv;
                }
            }
            for (int w = tid; w < W; w += STACK_NT) swords[w] = __ldcg(a.maskw + (size_t)l * W + w);
            __syncthreads();
            const int per = (W + STACK_NT - 1) / STACK_NT;
            const int wa = min(W, tid * per), wb = min(W, wa + per);
            int mine = 0;
            for (int w = wa; w < wb; ++w) mine += __popc(swords[w]);
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (lane == 31) wsum[warp] = incl;
            __syncthreads();
            int before = 0, total = 0;
            for (int w = 0; w < SNW; ++w) {
                before += w < warp ? wsum[w] : 0;
                total += wsum[w];
            }
            int off = before + incl - mine;
            for (int w = wa; w < wb; ++w) {
                spre[w] = off;
                off += __popc(swords[w]);
            }
            if (tid == 0) spre[W] = total;
            __syncthreads();
            const int n = total;
            if (c == 0 && tid == 0 && a.counts) a.counts[l] = n;

            for (int q = c; q < STACK_NCHUNK; q += P) {
                const int j0 = (int)((long long)q * n / STACK_NCHUNK), j1 = (int)((long long)(q + 1) * n / STACK_NCHUNK);
                const int nn = j1 - j0;
                for (int j = j0 + tid; j < j1; j += STACK_NT) {
                    const int i = select_active(swords, spre, W, j);
                    sneur[j - j0] = i;
                    if (a.idx_out) a.idx_out[(size_t)l * f + j] = i;
                }
                __syncthreads();

                auto issue = [&](uint32_t sq, int i) {
                    const int slot = (int)(sq % (uint32_t)S);
                    unsigned char *sl = ring + (size_t)slot * a.slot_bytes;
                    uint64_t *mb = &mbar[slot];
                    mbar_arrive_expect_tx(mb, (uint32_t)(ROWS * (rowb + sclb)));
                    bulk_g2s(sl, (const char *)Lw.wg + (size_t)i * rowb, rowb, mb);
                    if (KIND == KIND_GATED) bulk_g2s(sl + rowb, (const char *)Lw.wu + (size_t)i * rowb, rowb, mb);
                    bulk_g2s(sl + (ROWS - 1) * rowb, (const char *)Lw.wd + (size_t)i * rowb, rowb, mb);
                    if (WT == DT_INT4) {
                        unsigned char *ss = sl + ROWS * rowb;
                        bulk_g2s(ss, (const char *)Lw.sg + (size_t)i * sclb, sclb, mb);
                        if (KIND == KIND_GATED) bulk_g2s(ss + sclb, (const char *)Lw.su + (size_t)i * sclb, sclb, mb);
                        bulk_g2s(ss + (ROWS - 1) * sclb, (const char *)Lw.sd + (size_t)i * sclb, sclb, mb);
                    }
                };
                if (tid == 0) {
                    fence_proxy_async_smem();
                    for (int m = 0; m < nn && m < S; ++m) issue(seq + m, sneur[m]);
                }

                float yr[CPT][VW];
#pragma unroll
                for (int cc = 0; cc < CPT; ++cc)
#pragma unroll
                    for (int e = 0; e < VW; ++e) yr[cc][e] = 0.f;

                for (int m = 0; m < nn; ++m) {
                    const uint32_t sq = seq + m;
                    const int slot = (int)(sq % (uint32_t)S);
                    const unsigned char *sl = ring + (size_t)slot * a.slot_bytes;
                    const bool got = mbar_wait(&mbar[slot], (sq / (uint32_t)S) & 1u);
                    float pg = 0.f, pu = 0.f;
                    if (got) {
#pragma unroll
                        for (int cc = 0; cc < CPT; ++cc) {
                            const int ci = tid + cc * STACK_NT;
                            if (ci >= nchw) break;
                            const uint4 wg = reinterpret_cast<const uint4 *>(sl)[ci];
                            if constexpr (WT == DT_INT4) {
                                const __half *ss = reinterpret_cast<const __half *>(sl + ROWS * rowb);
                                const uint32_t ag[4] = {wg.x, wg.y, wg.z, wg.w};
                                float tg = 0.f;
#pragma unroll
                                for (int e = 0; e < 32; ++e) tg = fmaf(nib(ag[e >> 3], e & 7), ur[cc][e], tg);
                                pg = fmaf(__half2float(ss[ci >> 2]), tg, pg);
                                if (KIND == KIND_GATED) {
                                    const uint4 wu = reinterpret_cast<const uint4 *>(sl + rowb)[ci];
                                    const uint32_t au[4] = {wu.x, wu.y, wu.z, wu.w};
                                    float tu = 0.f;
#pragma unroll
                                    for (int e = 0; e < 32; ++e) tu = fmaf(nib(au[e >> 3], e & 7), ur[cc][e], tu);
                                    pu = fmaf(__half2float(ss[d / 128 + (ci >> 2)]), tu, pu);
                                }
                            } else {
                                float wf[VW];
                                unpack<WT>(wg, wf);
#pragma unroll
                                for (int e = 0; e < VW; ++e) pg = fmaf(wf[e], ur[cc][e], pg);
                                if (KIND == KIND_GATED) {
                                    unpack<WT>(reinterpret_cast<const uint4 *>(sl + rowb)[ci], wf);
#pragma unroll
                                    for (int e = 0; e < VW; ++e) pu = fmaf(wf[e], ur[cc][e], pu);
                                }
                            }
                        }
                    }
                    pg = warp_sum(pg);
                    if (KIND == KIND_GATED) pu = warp_sum(pu);
                    if (lane == 0) {
                        red[m & 1][warp][0] = pg;
                        red[m & 1][warp][1] = pu;
                    }
                    if (!__syncthreads_and(got)) {
                        // give up: wait (bounded) for this CTA's copies still in flight, then leave
                        if (tid == 0) {
                            set_status(a.status, ST_TIMEOUT);
                            for (int k = m; k < nn && k < m + S; ++k)
                                mbar_wait(&mbar[(seq + k) % (uint32_t)S], ((seq + k) / (uint32_t)S) & 1u);
                        }
                        return;
                    }
                    if (tid == 0 && m >= 1 && m - 1 + S < nn) {
                        fence_proxy_async_smem();
                        issue(seq + m - 1 + S, sneur[m - 1 + S]);
                    }
                    const int i = sneur[m];
                    float g = 0.f, up = 0.f;
                    for (int w = 0; w < SNW; ++w) {   // fixed order
                        g += red[m & 1][w][0];
                        up += red[m & 1][w][1];
                    }
                    g += Lw.bg ? __ldg(Lw.bg + i) : 0.f;
                    float hv = fmaxf(g, 0.f);
                    if (KIND == KIND_GATED) hv *= up;
                    const uint4 *wd = reinterpret_cast<const uint4 *>(sl + (ROWS - 1) * rowb);
#pragma unroll
                    for (int cc = 0; cc < CPT; ++cc) {
                        const int ci = tid + cc * STACK_NT;
                        if (ci >= nchw) break;
                        const uint4 w4 = wd[ci];
                        if constexpr (WT == DT_INT4) {
                            const __half *ss = reinterpret_cast<const __half *>(sl + ROWS * rowb + (ROWS - 1) * sclb);
                            const float hs = hv * __half2float(ss[ci >> 2]);
                            const uint32_t aw[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                            for (int e = 0; e < 32; ++e) yr[cc][e] = fmaf(hs, nib(aw[e >> 3], e & 7), yr[cc][e]);
                        } else {
                            float wf[VW];
                            unpack<WT>(w4, wf);
#pragma unroll
                            for (int e = 0; e < VW; ++e) yr[cc][e] = fmaf(hv, wf[e], yr[cc][e]);
                        }
                    }
                }
                seq += (uint32_t)nn;
                float *pq = a.part + (size_t)q * d;
#pragma unroll
                for (int cc = 0; cc < CPT; ++cc) {
                    const int ci = tid + cc * STACK_NT;
                    if (ci >= nchw) break;
#pragma unroll
                    for (int e4 = 0; e4 < VW / 4; ++e4)
                        reinterpret_cast<float4 *>(pq + (size_t)ci * VW)[e4] =
                            make_float4(yr[cc][4 * e4], yr[cc][4 * e4 + 1], yr[cc][4 * e4 + 2], yr[cc][4 * e4 + 3]);
                }
                __syncthreads();
            }
        }
        if (!sync_grid()) return;

        // ------------------------------------------------------------ D: fixed-order reduction + residual
        {
            const int nsl = (d + STACK_SLICE - 1) / STACK_SLICE;
            const int c4 = tid & 7, g = tid >> 3;   // 8 float4 per slice, 64 groups of chunks
            for (int s = c; s < nsl; s += P) {
                const int col = s * STACK_SLICE + c4 * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (col < d) {
#pragma unroll 3
                    for (int q = g; q < STACK_NCHUNK; q += STACK_NT / 8) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part + (size_t)q * d + col));
                        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
                    }
                }
                scr4[g * 8 + c4] = acc;
                __syncthreads();
                if (tid < 8) {
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int gg = 0; gg < STACK_NT / 8; ++gg) {   // fixed order
                        const float4 v = scr4[gg * 8 + tid];
                        y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
                    }
                    float ss = 0.f;
                    if (col < d) {
                        const float4 xv = __ldcg(reinterpret_cast<const float4 *>(xl + col));
                        y.x += xv.x; y.y += xv.y; y.z += xv.z; y.w += xv.w;
                        *reinterpret_cast<float4 *>(xn + col) = y;
                        ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
                    }
                    ss += __shfl_xor_sync(0xffu, ss, 1);
                    ss += __shfl_xor_sync(0xffu, ss, 2);
                    ss += __shfl_xor_sync(0xffu, ss, 4);
                    if (tid == 0) a.sumsq[s] = ss;
                }
                __syncthreads();
            }
            if (l + 1 < a.L) {
                load_p1(a.layers[l + 1]);   // input-independent: before the barrier
                if (!sync_grid()) return;
                if (warp == 0) {
                    float t = 0.f;
                    for (int s = lane; s < nsl; s += 32) t += __ldcg(a.sumsq + s);
                    t = warp_sum(t);
                    if (lane == 0) s_inv = 1.0f / sqrtf(t / (float)d + a.eps);
                }
                __syncthreads();
            }
        }
    }
}

template <int WT>
cudaError_t launch_stack_wt(int pdt, int kind, const StackArgs &a, int grid, size_t smem, cudaStream_t s)
{
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, STACK_NT, smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorNotSupported;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(STACK_NT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a);
    };
    const bool gated = kind == KIND_GATED;
    if constexpr (WT == DT_INT4) {
        if (pdt == DT_F16) return gated ? go(k_decode_stack<WT, DT_F16, KIND_GATED>) : go(k_decode_stack<WT, DT_F16, KIND_RELU>);
        if (pdt == DT_BF16) return gated ? go(k_decode_stack<WT, DT_BF16, KIND_GATED>) : go(k_decode_stack<WT, DT_BF16, KIND_RELU>);
    } else {
        if (pdt == WT) return gated ? go(k_decode_stack<WT, WT, KIND_GATED>) : go(k_decode_stack<WT, WT, KIND_RELU>);
    }
    return cudaErrorNotSupported;
}

}  // namespace pi
