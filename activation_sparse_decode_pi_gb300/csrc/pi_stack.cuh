// pi_stack.cuh -- one decode step through every layer in a single persistent kernel (batch 1).
//
// "PowerInfer" paper walk-through page, section "inference flow": the input reaches
// a layer, the predictor marks the neurons that will fire, only those are computed,
// the result is merged and passed to the next layer. Here every SM runs one CTA of
// 512 threads that walks all layers. A layer is three phases separated by bounded
// grid barriers:
//
//   A   hp[k] = ReLU(inv * P1T[k] . x)      CTA c: hidden units [c*r/P, (c+1)*r/P); each lane
//       reads the x chunks of the P1 chunks it multiplies (from L2) while the RMS scale inv is
//       summed from the slices' sums of squares
//   -- barrier
//   BC  CTA c owns the neurons i = c, c+P, c+2P, ... (hot-first order spreads the hot
//       neurons evenly). It computes their logits z[i] = hp . P2T[i] + b_p[i], keeps the
//       ones with z > tau in ascending order, bulk-copies their gate(/up) and W_down rows
//       and gate bias into a shared-memory ring (cp.async.bulk + mbarrier), reduces
//       h = ReLU(u.Wg + bg) * (u.Wu) over the CTA up to four neurons at a time, and
//       accumulates h * WdT into fp32 registers (each thread owns fixed columns). One
//       partial per CTA.
//   -- barrier (while waiting, the CTA requests the next layer's owned P2 rows into its ring)
//   D   x_{l+1} = x_l + sum of the P partials in a fixed order, per 32-column slice, plus
//       that slice's sum of squares for the next layer's RMS scale.
//   -- barrier
//
// Neither a global mask scan nor a global active list is on the critical path: each
// CTA computes the FFN of exactly the neurons whose logits it computed. The active
// counts (and, on request, the ascending active lists) are produced alongside.
// The predictor weights do not depend on the input. The ring is idle between one layer's
// FFN and the next layer's logits, so the next layer's owned P2 rows are copied into it
// then (as many as fit); with a 16-bit predictor (r % 32 == 0) the logits run as 16-row tiles
// on the tensor cores (mma.sync, hp split into hi and lo halves of the predictor's type),
// staged rows read from shared memory and the others streamed from memory; otherwise as
// CUDA-core row dot products. While one layer's predictor is small next to L2, P1 and the P2
// rows that do not fit are prefetched into L2 a layer ahead.
// Hot neurons (the first hot_k owned ones in hot-first order, typically active on most
// tokens) can have ring slots of their own: their rows are requested one layer ahead, during
// the previous layer's barrier wait, before the predictor has said whether they fire. A hot
// neuron the predictor rejects costs its bytes and nothing else: the neurons are reduced in
// the same list order either way, so the output bits do not depend on hot_k.
// The result is deterministic: every sum runs in a fixed order for a given grid size.
#pragma once

#include "pi_async.cuh"
#include "pi_common.cuh"
#include "pi_internal.h"
#include "pi_rowdot.cuh"
#include "pi_umma.cuh"

namespace pi {

constexpr int SNW = STACK_NT / 32;
static_assert(SNW == 16, "the batch reduction maps the 16 warps onto half a warp's lanes");
static_assert(STACK_MAX_CHUNK <= STACK_NT, "one owned neuron per thread");

template <int WT>
__host__ __device__ constexpr int weight_row_bytes(int d)
{
    return WT == DT_F32 ? d * 4 : (WT == DT_INT4 ? d / 2 : d * 2);
}

// First chunk (one per lane and row) of up to 8 consecutive predictor hidden rows [k0, k1).
template <int PT>
__device__ __forceinline__ void load_p1_chunk(RowChunks<PT, 8, 1> &pa, const void *p1, int k0, int k1, int nchp,
                                              int c, int ce)
{
    const uint4 *row[8];
    const __half *srow[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        row[k] = k0 + k < k1 ? reinterpret_cast<const uint4 *>(p1) + (size_t)(k0 + k) * nchp : nullptr;
        srow[k] = nullptr;
    }
    rows_issue(pa, row, srow, c, ce);
}

// Rows kbase, kbase + step, ... of the neurons a CTA owns (i = c + P * k, k < K) in a [f x r] matrix;
// none for neurons below `hot` (the hot prefix needs no logit).
template <int RW>
__device__ __forceinline__ void owned_rows(const uint4 *(&row)[RW], const void *m, int kbase, int step, int K, int c,
                                           int P, int nch, int hot)
{
#pragma unroll
    for (int q = 0; q < RW; ++q) {
        const int k = kbase + step * q;
        const int i = c + P * k;
        row[q] = (k < K && i >= hot) ? reinterpret_cast<const uint4 *>(m) + (size_t)i * nch : nullptr;
    }
}

// Sum of each of N (4 or 8) per-lane values over the warp, transposed: lane L ends with the sum
// of value L / (32 / N). The value count halves at each of the first log2(N) butterfly levels
// (lanes with the level's bit set keep the upper half), so the N sums take N - 1 + 5 - log2(N)
// shuffles instead of 5 N; the order of the additions is fixed.
template <int N>
__device__ __forceinline__ float warp_transpose_sum(const float (&v)[N], int lane)
{
    static_assert(N == 4 || N == 8, "value count");
    float w[N];
#pragma unroll
    for (int j = 0; j < N; ++j) w[j] = v[j];
    int off = 16;
#pragma unroll
    for (int h = N / 2; h >= 1; h /= 2, off /= 2) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < h; ++j) {
            const float send = up ? w[j] : w[j + h];
            const float keep = up ? w[j + h] : w[j];
            w[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (; off >= 1; off /= 2) w[0] += __shfl_xor_sync(0xffffffffu, w[0], off);
    return w[0];
}

// Four 8 x 8 tiles of 16-bit elements from shared memory (lane l gives the address of row
// l % 8 of tile l / 8), one 32-bit register per tile and lane.
__device__ __forceinline__ void ldsm_x4(uint32_t saddr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}

// D[16 x 8] += A[16 x 16] * B[16 x 8], 16-bit operands of type PT, fp32 accumulators
// (warp-level mma.sync; fragments in the m16n8k16 layouts).
template <int PT>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    if constexpr (PT == DT_BF16)
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                     "{%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                     "{%8, %9}, {%0, %1, %2, %3};"
                     : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                     : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Bulk-copy neuron i's rows of layer Lw (gate(, up), W_down; int4 scales; the 16-byte chunk
// holding its gate bias) into ring slot `slot`; completion is counted on the slot's mbarrier.
// Everything is derived from the launch arguments, so callers keep no state for it.
template <int WT, int KIND>
__device__ __forceinline__ void stage_neuron(const StackArgs &a, const StackLayer &Lw, unsigned char *ring,
                                             uint64_t *mbar, int slot, int i)
{
    constexpr int ROWS = KIND == KIND_GATED ? 3 : 2;
    const int rowb = WT == DT_F32 ? a.d * 4 : (WT == DT_INT4 ? a.d / 2 : a.d * 2);
    const int sclb = WT == DT_INT4 ? (a.d / 128) * 2 : 0;
    const int bias_off = ROWS * (rowb + sclb);
    unsigned char *sl = ring + (size_t)slot * a.slot_bytes;
    uint64_t *mb = &mbar[slot];
    mbar_arrive_expect_tx(mb, (uint32_t)(bias_off + (a.bias_bulk ? 16 : 0)));
    bulk_g2s(sl, (const char *)Lw.wg + (size_t)i * rowb, rowb, mb);
    if (KIND == KIND_GATED) bulk_g2s(sl + rowb, (const char *)Lw.wu + (size_t)i * rowb, rowb, mb);
    bulk_g2s(sl + (ROWS - 1) * rowb, (const char *)Lw.wd + (size_t)i * rowb, rowb, mb);
    if (WT == DT_INT4) {
        unsigned char *ss = sl + ROWS * rowb;
        bulk_g2s(ss, (const char *)Lw.sg + (size_t)i * sclb, sclb, mb);
        if (KIND == KIND_GATED) bulk_g2s(ss + sclb, (const char *)Lw.su + (size_t)i * sclb, sclb, mb);
        bulk_g2s(ss + (ROWS - 1) * sclb, (const char *)Lw.sd + (size_t)i * sclb, sclb, mb);
    }
    if (a.bias_bulk) bulk_g2s(sl + bias_off, Lw.bg + (i & ~3), 16, mb);
}

// Copies that make up one neuron's slot: its weight rows, (int4) their scale rows, and the
// 16-byte chunk holding its gate bias when biases travel with the rows.
template <int WT, int KIND>
__device__ __forceinline__ int stage_parts(const StackArgs &a)
{
    constexpr int ROWS = KIND == KIND_GATED ? 3 : 2;
    return ROWS * (WT == DT_INT4 ? 2 : 1) + (a.bias_bulk ? 1 : 0);
}

// Copy j (< stage_parts) of neuron i's slot; copy 0 also registers the slot's byte count. The
// copies of one slot may be issued by different threads in any order.
template <int WT, int KIND>
__device__ __forceinline__ void stage_part(const StackArgs &a, const StackLayer &Lw, unsigned char *ring,
                                           uint64_t *mbar, int slot, int i, int j)
{
    constexpr int ROWS = KIND == KIND_GATED ? 3 : 2;
    const int rowb = WT == DT_F32 ? a.d * 4 : (WT == DT_INT4 ? a.d / 2 : a.d * 2);
    const int sclb = WT == DT_INT4 ? (a.d / 128) * 2 : 0;
    const int bias_off = ROWS * (rowb + sclb);
    unsigned char *sl = ring + (size_t)slot * a.slot_bytes;
    uint64_t *mb = &mbar[slot];
    if (j == 0) mbar_arrive_expect_tx(mb, (uint32_t)(bias_off + (a.bias_bulk ? 16 : 0)));
    if (j < ROWS) {
        const void *src = j == 0 ? Lw.wg : (KIND == KIND_GATED && j == 1 ? Lw.wu : Lw.wd);
        bulk_g2s(sl + j * rowb, (const char *)src + (size_t)i * rowb, rowb, mb);
    } else if (WT == DT_INT4 && j < 2 * ROWS) {
        const int q = j - ROWS;
        const void *src = q == 0 ? Lw.sg : (KIND == KIND_GATED && q == 1 ? Lw.su : Lw.sd);
        bulk_g2s(sl + ROWS * rowb + q * sclb, (const char *)src + (size_t)i * sclb, sclb, mb);
    } else {
        bulk_g2s(sl + bias_off, Lw.bg + (i & ~3), 16, mb);
    }
}

template <int WT, int PT, int KIND, int CPT>
__global__ void __launch_bounds__(STACK_NT, 1) k_decode_stack(const StackArgs a)
{
    constexpr int VW = Vec<WT>::N;                           // CPT: weight chunks per thread per row
    constexpr int VP = Vec<PT>::N;
    constexpr int ROWS = KIND == KIND_GATED ? 3 : 2;         // weight rows staged per neuron
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem + a.off_ring;                 // neuron slots
    uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + a.off_mbar);
    float4 *hp4 = reinterpret_cast<float4 *>(smem + a.off_hp);         // phase BC: hp (planar)
    float4 *scr4 = reinterpret_cast<float4 *>(smem + a.off_scr);       // phase D: partial sums
    unsigned char *sflag = smem + a.off_flags;                          // phase BC: logit > tau per owned row

    __shared__ float red[2][SNW][8];
    __shared__ unsigned long long s_base;
    __shared__ int wsum[SNW];
    __shared__ int sneur[STACK_MAX_CHUNK];
    __shared__ float sbias[STACK_MAX_CHUNK];
    __shared__ float s_inv;
    __shared__ int s_flag;
    __shared__ uint64_t s_p2bar[STACK_P2_TILES];   // P2 tile slot j: its rows have landed
    __shared__ int s_p2use[STACK_P2_TILES];        // tiles slot j holds per layer
    __shared__ int s_p2par[STACK_P2_TILES];        // parity of slot j's copies in flight across a grid barrier (-1: none)
    __shared__ int s_p2iss[STACK_P2_TILES];        // uses of slot j issued in the current layer's logits
    __shared__ float spb[STACK_MAX_CHUNK];   // predictor bias of the owned rows, copied during phase A
    __shared__ const void *s_p2next;          // P2 of the next layer (read during phase A)
    __shared__ int s_pend;         // parity of the last hot-slot copies issued (-1: none)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x, c = blockIdx.x;
    const int d = a.d, f = a.f, r = a.r, S = a.slots;
    const int W = (f + 31) >> 5;
    const int rowb = weight_row_bytes<WT>(d);
    const int sclb = WT == DT_INT4 ? (d / 128) * 2 : 0;
    const int pb = PT == DT_F32 ? 4 : 2;
    const int k0 = (int)((long long)c * r / P), k1 = (int)((long long)(c + 1) * r / P);
    const int K = c < f ? (f - 1 - c) / P + 1 : 0;          // owned neurons: i = c + P * k, k < K
    const int bias_off = ROWS * (rowb + sclb);               // 16-byte chunk holding the gate bias
    const bool bias_bulk = a.bias_bulk != 0;                 // the chunk stays inside b_gate only if f % 4 == 0
    // The owned P2 rows pass through the ring in tiles of 16 rows: tile t (owned rows
    // [16t, 16t + 16)) in slot t % RT at ring + (t % RT) * 16 * p2st, completing on mbarrier
    // s_p2bar[t % RT]. The ring is idle from the end of one layer's FFN to the next layer's
    // logits, so the first NI = min(MT, RT) tiles of the next layer are copied into it then (they
    // land during the reduction and predictor phases). With the tensor-core logits and more tiles
    // than slots, the logits stream the rest: each slot is refilled with the tile RT further on
    // as soon as its tile has been multiplied. Rows below the hot prefix need no copy.
    const int p2b = r * pb, p2st = stack_p2_stride(p2b);
    const int MT = (K + 15) >> 4, RT = a.p2_tiles;
    bool TCL = false;   // logits on the tensor cores
    if constexpr (PT == DT_BF16 || PT == DT_F16) TCL = K > 0 && (r & 15) == 0 && (MT <= RT || RT >= 2);
    const int NR = min(MT, RT);                              // tiles in the ring at the start of the logits
    const int NI = min(NR, a.p2_stage_tiles);                // of which staged between layers
    const int MTS = TCL ? MT : NR;                           // tiles through the ring per layer
    const int KS = min(K, NR * 16);                          // rows in the ring at the start of the logits
    const int ks0 = a.hot_prefix > c ? min(K, (a.hot_prefix - c + P - 1) / P) : 0;
    // bytes of tile t's rows that are copied (past K and below the hot prefix: none)
    auto tile_bytes = [&](int t) -> uint32_t {
        const int lo = max(16 * t, ks0), hi = min(16 * t + 16, K);
        return hi > lo ? (uint32_t)((hi - lo) * p2b) : 0u;
    };
    // parity of the phase of slot t % RT that holds tile t of layer l (timeout paths only: it divides)
    auto tile_par = [&](int l, int t) -> uint32_t {
        const int j = t % RT;
        return (uint32_t)(l * s_p2use[j] + t / RT) & 1u;
    };
    // the same for one of the first RT tiles (slot t, first use in the layer)
    auto tile_par0 = [&](int l, int t) -> uint32_t { return (uint32_t)(l * s_p2use[t]) & 1u; };
    // copy rows [lo, hi) of tile t (owned rows) into its slot; the ring there is free
    auto copy_tile_rows = [&](const void *p2, int t, int j, int lo, int hi) {
        for (int k = max(lo, ks0); k < hi && k < K; ++k) {
            fence_proxy_async_smem();
            bulk_g2s(ring + (size_t)(j * 16 + (k - 16 * t)) * p2st,
                     (const char *)p2 + (size_t)(c + (size_t)P * k) * p2b, (uint32_t)p2b, &s_p2bar[j]);
        }
    };
    // Ring slots [0, HK) hold this CTA's hot owned neurons k < HK (loaded every layer before its
    // predictor runs: the copy for layer l is the slot's l-th, parity l & 1). Slots [HK, S) take
    // the other active neurons in list order: the cold neuron staged n-th in this launch goes to
    // slot HK + n % SC with parity (n / SC) & 1.
    uint32_t cseq = 0;
    unsigned kb = 0;    // grid barriers passed in this launch
    // optional %globaltimer stamp of phase boundary ph of layer l (thread 0 of each CTA)
    auto stamp = [&](int l, int ph) {
        if (a.stamps && tid == 0) a.stamps[((size_t)l * STACK_PHASES + ph) * P + c] = globaltimer_ns();
    };
    auto sync_grid = [&](auto work) -> bool {
        ++kb;
        const PendingCopies pc{s_p2bar, s_p2par, NI, mbar, min(a.hot_k, K), &s_pend};
        return grid_sync_to(a.bar, s_base + (unsigned long long)kb * a.nblocks, a.status, &s_flag, &pc, work);
    };
    const NoWork no_work;
    // the first NI tiles of layer l are about to be staged: their byte counts, and their parities
    // for a drain after a timed-out grid barrier
    auto expect_p2 = [&](int l) {
        if (tid < NI) {
            mbar_arrive_expect_tx(&s_p2bar[tid], tile_bytes(tid));
            s_p2par[tid] = (int)tile_par0(l, tid);
        }
    };
    // one copy per thread, row k = 16 * lane + warp (a warp's copies are issued one after another,
    // so every warp takes a few); the ring is free and expect_p2 ran
    auto stage_p2 = [&](const void *p2) {
        const int k = lane * SNW + warp;
        if (k < min(KS, NI * 16)) copy_tile_rows(p2, k >> 4, k >> 4, k, k + 1);   // tile k / 16 < NI sits in slot k / 16
    };
    // tiles [NI, NR) of layer l, not staged between layers, requested as the logits start
    // (thread 32 registers the bytes, one copy per thread)
    auto issue_rest = [&](const StackLayer &Lw, int l) {
        if (tid >= 32 + NI && tid < 32 + NR) mbar_arrive_expect_tx(&s_p2bar[tid - 32], tile_bytes(tid - 32));
        const int k = lane * SNW + warp + NI * 16;
        if (k < KS) copy_tile_rows(Lw.p2, k >> 4, k >> 4, k, k + 1);
    };
    // after a timeout: wait (bounded) for the copies of tiles [t0, t1) of layer l
    auto drain_tiles = [&](int l, int t0, int t1) {
        for (int t = t0; t < t1 && t < MTS; ++t) mbar_wait(&s_p2bar[t % RT], tile_par(l, t));
    };

    // this CTA's P1 rows, one chunk per lane and row at a time
    const int nchp = d / VP;
    const int pa_per = (nchp + SNW - 1) / SNW, pa_cb = warp * pa_per, pa_ce = min(nchp, pa_cb + pa_per);
    RowChunks<PT, 8, 1> pa;
    // This CTA's P1 rows of a layer into L2 (the last thread), issued inside the grid barrier that
    // follows the previous layer's FFN, so that they land during the reduction phase.
    auto prefetch_p1 = [&](const StackLayer &L) {
        if (tid == STACK_NT - 1)
            prefetch_l2_range((const char *)L.p1 + (size_t)k0 * d * pb, (size_t)(k1 - k0) * d * pb);
    };
    // The owned P2 rows that are not staged, into L2 a whole layer ahead (one row per thread):
    // only while a layer's predictor is small next to L2.
    auto prefetch_p2 = [&](const StackLayer &L) {
        if (a.pf_p2 && tid >= KS && tid < K)
            prefetch_l2((const char *)L.p2 + (size_t)(c + (size_t)P * tid) * r * pb, r * pb);
    };

    // the hot owned neurons of layer Lw into their slots, one issuing thread per neuron; the
    // slots' previous copies (parity prev, or none when prev < 0) have landed and been read
    auto issue_hot = [&](const StackLayer &Lw, int prev) {
        const int w = threadIdx.x >> 5, cb = blockIdx.x, np = gridDim.x;
        const int hk = min(a.hot_k, cb < a.f ? (a.f - 1 - cb) / np + 1 : 0);
        if ((threadIdx.x & 31) != 0 || w >= hk) return;
        unsigned char *rg = smem + a.off_ring;
        uint64_t *mbs = reinterpret_cast<uint64_t *>(smem + a.off_mbar);
        for (int k = w; k < hk; k += SNW) {
            if (prev >= 0 && !mbar_wait(&mbs[k], (uint32_t)prev & 1u)) set_status(a.status, ST_TIMEOUT);
            fence_proxy_async_smem();
            stage_neuron<WT, KIND>(a, Lw, rg, mbs, k, cb + np * k);
        }
    };

    // ---------------------------------------------------------------- phase 0
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 1);
        for (int j = 0; j < RT && j < STACK_P2_TILES; ++j) mbar_init(&s_p2bar[j], 1);
        fence_mbar_init();
        s_pend = a.hot_k > 0 ? 0 : -1;
        s_base = barrier_base(a.bar, (unsigned long long)((3 + (a.balance == 1 ? 1 : 0)) * a.L) * a.nblocks);
    }
    if (tid < STACK_P2_TILES) {
        s_p2use[tid] = tid < min(MTS, RT) ? (MTS - tid + RT - 1) / RT : 0;
        s_p2par[tid] = -1;
    }
    __syncthreads();   // the barriers are initialised and s_p2use is set
    expect_p2(0);
    if (a.pf_p1) prefetch_p1(a.layers[0]);
    prefetch_p2(a.layers[0]);
    __syncthreads();
    issue_hot(a.layers[0], -1);
    if (KS > 0) stage_p2(a.layers[0].p2);
    if (a.idx_out)
        for (int i = c * STACK_NT + tid; i < a.L * W; i += P * STACK_NT) a.maskw[i] = 0u;
    if (a.counts && c == 0)
        for (int i = tid; i < a.L; i += STACK_NT) a.counts[i] = 0;
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
    if (!sync_grid(no_work)) return;

    for (int l = 0; l < a.L; ++l) {
        const StackLayer Lw = a.layers[l];
        const float *xl = l == 0 ? a.x0 : (((l - 1) & 1) ? a.xb : a.xa);
        float *xn = l == a.L - 1 ? a.x_out : ((l & 1) ? a.xb : a.xa);
        float inv;   // RMS scale of x_l
        stamp(l, 0);

        // ------------------------------------------------------------ A: predictor hidden layer
        {
            // The first chunks of this CTA's P1 rows (prefetched into L2 a layer ago where that pays)
            // are requested with the matching chunks of x_l (read from L2, unscaled), while warp 0
            // adds up the slices' sums of squares; the RMS scale is applied to the dot products
            // (hp = ReLU(inv * P1 x)). x is not staged in shared memory: each lane reads the x chunk
            // of the P1 chunk it multiplies, which the 8 rows share.
            constexpr int QP = VP / 4;
            float4 xq[QP];
            auto load_x = [&](int ci) {
#pragma unroll
                for (int q = 0; q < QP; ++q)
                    xq[q] = ci < pa_ce ? __ldcg(reinterpret_cast<const float4 *>(xl + (size_t)ci * VP) + q)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            };
            load_p1_chunk<PT>(pa, Lw.p1, k0, k1, nchp, pa_cb + lane, pa_ce);
            load_x(pa_cb + lane);
            const int nsl = (d + STACK_SLICE - 1) / STACK_SLICE;
            float ssq = 0.f;
            if (l > 0 && warp == 0)
                for (int s = lane; s < nsl; s += 32) ssq += __ldcg(a.sumsq + s);
            if (tid < K) {   // the logits' biases, waited for before this phase's grid barrier
                if (Lw.bp) cp_async4(&spb[tid], Lw.bp + c + P * tid);
                else spb[tid] = 0.f;
            }
            if (tid == STACK_NT - 1 && l + 1 < a.L) s_p2next = a.layers[l + 1].p2;
            if (l > 0 && warp == 0) {
                ssq = warp_sum(ssq);
                if (lane == 0) s_inv = 1.0f / sqrtf(ssq / (float)d + a.eps);
            }
            if (l + 1 < a.L) prefetch_p2(a.layers[l + 1]);
            if (l + 1 < a.L && a.pf_p1 == 2) prefetch_p1(a.layers[l + 1]);   // a whole layer ahead
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
            // acc[k] += P1 row k0 + k, chunk ci . x chunk ci (the loaded ones)
            auto consume = [&](int ci) {
                if (ci >= pa_ce) return;
                float xe[VP];
#pragma unroll
                for (int q = 0; q < QP; ++q) {
                    xe[4 * q + 0] = xq[q].x;
                    xe[4 * q + 1] = xq[q].y;
                    xe[4 * q + 2] = xq[q].z;
                    xe[4 * q + 3] = xq[q].w;
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float wf[VP];
                    unpack<PT>(pa.w[k][0], wf);
                    float v = acc[k][0];
#pragma unroll
                    for (int e = 0; e < VP; ++e) v = fmaf(wf[e], xe[e], v);
                    acc[k][0] = v;
                }
            };
            consume(pa_cb + lane);
            for (int cc = pa_cb + lane + 32; cc < pa_ce; cc += 32) {
                rows_issue(pa, row, srow, cc, pa_ce);
                load_x(cc);
                consume(cc);
            }
            __syncthreads();   // s_inv
            inv = s_inv;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float v = warp_sum(acc[k][0]);
                if (lane == 0) red[0][warp][k] = v;
            }
            __syncthreads();
            if (tid < 8 && k0 + tid < k1) {
                float v = 0.f;
                for (int w = 0; w < SNW; ++w) v += red[0][w][tid];   // fixed order
                a.hp[k0 + tid] = fmaxf(inv * v, 0.f);
            }
            cp_async_wait_all();
        }
        stamp(l, 1);
        if (!sync_grid(no_work)) return;
        stamp(l, 2);

        // ------------------------------------------------------------ BC: logits, then the sparse FFN
        {
            // logits of the owned rows: warp w takes rows k = w, w + 16, ..., five at a time
            const int nchr = r / VP;
            const uint4 *row[5];
            RowChunks<PT, 5, 4> rc;
            // rows kbase + SNW * q: a staged row is read from the ring (the generic loads below
            // take either space), the others from memory
            auto rows_at = [&](int kbase) {
                owned_rows<5>(row, Lw.p2, kbase, SNW, K, c, P, nchr, a.hot_prefix);
#pragma unroll
                for (int q = 0; q < 5; ++q) {
                    const int k = kbase + SNW * q;
                    if (k < KS && row[q]) row[q] = reinterpret_cast<const uint4 *>(ring + (size_t)k * p2st);
                }
            };
            auto issue_rows = [&](int cc) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ci = cc + 32 * i;
#pragma unroll
                    for (int q = 0; q < 5; ++q)
                        rc.w[q][i] = ci < nchr && row[q] != nullptr ? row[q][ci] : make_uint4(0u, 0u, 0u, 0u);
                }
            };
            if (NI < NR) {   // the tiles not staged between layers are requested first
                fence_proxy_async_smem();
                issue_rest(Lw, l);
            }
            // hp is requested first, so its reads (L2 hits) do not queue behind the P2 rows
            const int r4 = r / 4;
            float4 hv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = tid + u * STACK_NT;
                hv[u] = t < r4 ? __ldcg(reinterpret_cast<const float4 *>(a.hp) + t) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // the staged tiles [0, nt) have landed (every thread waits); false after a timeout, when
            // the CTA leaves once its copies in flight have landed
            auto wait_staged = [&](int nt) -> bool {
                bool ok = true;
                for (int j = 0; j < nt; ++j) ok = mbar_wait(&s_p2bar[j], tile_par0(l, j)) && ok;
                if (__syncthreads_and(ok)) return true;
                if (tid == 0) {
                    set_status(a.status, ST_TIMEOUT);
                    drain_tiles(l, 0, nt);
                }
                return false;
            };
            // 16-bit predictor, r % 16 == 0: the logits are small contractions on the tensor cores,
            // [16-row tile of P2 rows] x [hp_hi hp_lo 0 ... 0] per mma.sync, hp entering as hi + lo
            // halves in the predictor's type (so ~16 bits of it, with fp32 accumulation), A read
            // from the ring with ldmatrix (the odd row stride keeps it conflict-free).
            bool act = false;   // owned neuron k = tid fires
            if (TCL) {
                uint32_t *bfr = reinterpret_cast<uint32_t *>(hp4);   // B fragments [r/16][8 lanes][2]
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int t = tid + u * STACK_NT;
                    if (t >= r4) continue;
                    const float e[4] = {hv[u].x, hv[u].y, hv[u].z, hv[u].w};
#pragma unroll
                    for (int h = 0; h < 2; ++h) {   // element pair p = 2t + h: k = 2p, 2p + 1
                        uint16_t h0, l0, h1, l1;
                        split16<PT>(e[2 * h], h0, l0);
                        split16<PT>(e[2 * h + 1], h1, l1);
                        const int p = 2 * t + h, s16 = p >> 3, w = p & 7;
                        const int ln = w & 3, reg = w >> 2;   // lane (column 0 = hi) and register of the pair
                        bfr[(s16 * 8 + ln) * 2 + reg] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                        bfr[(s16 * 8 + ln + 4) * 2 + reg] = (uint32_t)l0 | ((uint32_t)l1 << 16);
                    }
                }
                float *zp = reinterpret_cast<float *>(scr4);
                const int NKS = r >> 4;
                // the products of k16 steps [s0, s1) of the 16 rows of the tile in slot j (rows past
                // K repeat row K - 1) into two accumulators (even and odd steps)
                auto tile_mma = [&](int t, int j, int s0, int s1, float (&acc)[2][4]) {
                    const int rw = min(t * 16 + (lane & 15), K - 1) - t * 16;
                    const uint32_t ab = smem_u32(ring) + (uint32_t)((j * 16 + rw) * p2st) + (uint32_t)(lane >> 4) * 16u;
                    for (int s16 = s0; s16 < s1; s16 += 2) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if (s16 + e >= s1) break;
                            uint32_t af[4];
                            ldsm_x4(ab + (uint32_t)(s16 + e) * 32u, af);
                            const uint2 bf = lane < 8 ? reinterpret_cast<const uint2 *>(bfr)[(s16 + e) * 8 + lane]
                                                      : make_uint2(0u, 0u);
                            mma_16816<PT>(acc[e], af, bf.x, bf.y);
                        }
                    }
                };
                if (MT <= RT) {
                    // every tile was staged between layers: one pass, units (tile t, k part g), G warps
                    // sharing a tile when there are fewer tiles than warps
                    if (!wait_staged(MT)) return;   // MT == NR here
                    const int G = MT >= SNW ? 1 : SNW / MT;
                    for (int u = warp; u < MT * G; u += SNW) {
                        const int t = u / G, g = u - t * G;
                        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        tile_mma(t, t, g * NKS / G, (g + 1) * NKS / G, acc);
                        if ((lane & 3) == 0) {   // columns 0 (hi part) and 1 (lo part) of rows lane/4, lane/4 + 8
                            zp[u * 16 + (lane >> 2)] = (acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]);
                            zp[u * 16 + (lane >> 2) + 8] = (acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]);
                        }
                    }
                    __syncthreads();
                    if (tid < K) {
                        const int t = tid >> 4;
                        float z = 0.f;
                        for (int g = 0; g < G; ++g) z += zp[(t * G + g) * 16 + (tid & 15)];   // fixed order
                        z += spb[tid];
                        act = c + P * tid < a.hot_prefix || z > a.tau;
                    }
                } else {
                    // More tiles than slots: two groups of 8 warps take the tiles in turn (group g:
                    // tiles g, g + 2, ...), each warp of a group a 1/8 share of a tile's k steps, with
                    // a named barrier per group, so one group's synchronisation overlaps the other's
                    // products. A slot is refilled with the tile RT further on as soon as its tile's
                    // products are done (the mbarrier hands it to whichever group takes that tile),
                    // so up to RT - 2 tiles of copies stay in flight.
                    float *zt = sbias;   // the tiles' logits (sbias is written only after the list)
                    const int grp = warp >> 3, gw = warp & 7, gtid = tid & 255;
                    const int s0 = gw * NKS / 8, s1 = (gw + 1) * NKS / 8;
                    if (tid < RT) s_p2iss[tid] = tid < NR ? 1 : 0;   // uses of each slot issued in this layer
                    __syncthreads();
                    bool ok = true;
                    int j = grp, wrap = 0;   // slot of tile t, and t / RT (RT >= 2)
                    for (int t = grp; t < MT; t += 2) {
                        ok = mbar_wait(&s_p2bar[j], (uint32_t)(l * s_p2use[j] + wrap) & 1u);
                        ok = bar_and(1 + grp, 256, ok);   // the group decides together
                        if (!ok) break;
                        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        tile_mma(t, j, s0, s1, acc);
                        float *zb = zp + ((grp * 2 + ((t >> 1) & 1)) * 8) * 16;   // per group, double-buffered
                        if ((lane & 3) == 0) {
                            zb[gw * 16 + (lane >> 2)] = (acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1]);
                            zb[gw * 16 + (lane >> 2) + 8] = (acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3]);
                        }
                        bar_sync(1 + grp, 256);   // the slot's rows are read and the partials written
                        if (gtid < 16) {
                            float z = 0.f;
                            for (int w = 0; w < 8; ++w) z += zb[w * 16 + gtid];   // fixed order
                            zt[t * 16 + gtid] = z;
                        }
                        const int tn = t + RT;
                        if (tn < MT) {   // refill: one thread registers the bytes, 16 threads copy a row each
                            if (gtid == 32) {
                                s_p2iss[j] += 1;
                                mbar_arrive_expect_tx(&s_p2bar[j], tile_bytes(tn));
                            }
                            // two lanes of each of the group's 8 warps: a warp's bulk copies run one after
                            // another, so the 16 copies of a tile are spread over the warps
                            if (lane == 20 || lane == 21) {
                                const int q = gw * 2 + lane - 20;
                                copy_tile_rows(Lw.p2, tn, j, tn * 16 + q, tn * 16 + q + 1);
                            }
                        }
                        j += 2;
                        if (j >= RT) {
                            j -= RT;
                            ++wrap;
                        }
                    }
                    if (!__syncthreads_and(ok)) {
                        // a group gave up: wait (bounded) for every slot's last copies, then leave
                        if (tid == 0) {
                            set_status(a.status, ST_TIMEOUT);
                            for (int q = 0; q < RT; ++q)
                                if (s_p2iss[q] > 0) mbar_wait(&s_p2bar[q], (uint32_t)(l * s_p2use[q] + s_p2iss[q] - 1) & 1u);
                        }
                        return;
                    }
                    if (tid < K) {
                        const float z = zt[tid] + spb[tid];
                        act = c + P * tid < a.hot_prefix || z > a.tau;
                    }
                }
                if (tid < NI) s_p2par[tid] = -1;   // every staged copy has been waited for
            } else {
                rows_at(warp);
                issue_rows(lane);                                    // before hp is staged
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    constexpr int QH = VP / 4;
                    const int t = tid + u * STACK_NT;
                    if (t < r4) hp4[(t % QH) * nchr + t / QH] = hv[u];   // planar layout of the row dot products
                }
                if (!wait_staged(NR)) return;
                if (tid < NI) s_p2par[tid] = -1;
                for (int kbase = warp; kbase < K; kbase += SNW * 5) {
                    if (kbase != warp) {
                        rows_at(kbase);
                        issue_rows(lane);
                    }
                    float acc[5][1] = {{0.f}, {0.f}, {0.f}, {0.f}, {0.f}};
                    for (int cc = lane;;) {
                        rows_consume<PT, 5, 4, 1>(rc, cc, nchr, hp4, r, acc);
                        cc += 32 * 4;
                        if (cc >= nchr) break;
                        issue_rows(cc);
                    }
#pragma unroll
                    for (int q = 0; q < 5; ++q) {
                        const int k = kbase + SNW * q;
                        const int i = c + P * k;
                        const float z = warp_sum(acc[q][0]) + (k < K ? spb[k] : 0.f);
                        if (lane == 0 && k < K) sflag[k] = (i < a.hot_prefix || z > a.tau) ? 1 : 0;
                    }
                }
                __syncthreads();
                act = tid < K && sflag[tid];
            }
            // ascending list of the owned active neurons (thread k holds owned neuron k's flag)
            const uint32_t bal = __ballot_sync(0xffffffffu, act);
            if (lane == 0) wsum[warp] = __popc(bal);
            __syncthreads();
            int before = 0, nn = 0;
            for (int w = 0; w < SNW; ++w) {
                const int v = wsum[w];
                before += w < warp ? v : 0;
                nn += v;
            }
            if (act) {
                const int off = before + __popc(bal & ((1u << lane) - 1u));
                const int i = c + P * tid;
                if (!bias_bulk) sbias[off] = Lw.bg ? __ldg(Lw.bg + i) : 0.f;
                sneur[off] = i;
                if (a.idx_out) atomicOr(a.maskw + (size_t)l * W + (i >> 5), 1u << (i & 31));
            }
            if (tid == 0 && a.counts && nn) atomicAdd(a.counts + l, nn);
            __syncthreads();
            // Group balance, part 1 (a.balance = G > 1): within each group of G consecutive CTAs
            // every member publishes its list and an epoch (this launch and layer) with a release
            // store after the CTA barrier (a fence before it cost ~2 µs under the logits' copy
            // traffic; published after the first FFN copies, the flag round trips took microseconds
            // longer behind them). A member keeps the first K0 entries of its own
            // list, the first FFN batch, whose rows are requested at once; its share of the rest is
            // settled while they land (part 2, below).
            const int G = a.balance > 1 ? a.balance : 1;
            const int K0 = max(1, min(4, S / 2));   // the first cold batch (no hot slots with balance)
            if (G > 1) {
                const unsigned long long epoch = s_base + (unsigned long long)(l + 1);
                int32_t *gl = a.glist + (size_t)c * STACK_MAX_CHUNK;
                for (int m = tid; m < nn; m += STACK_NT) gl[m] = sneur[m];
                if (tid == 0) a.gcount[c] = nn;
                __syncthreads();   // the CTA's list stores come before the release below
                if (tid == 0) st_release_u64(a.gflag + c, epoch);   // release: the CTA's writes before the CTA barrier
                nn = min(nn, K0);
            }
            if (a.balance == 1) {
                // Every CTA publishes its list; after one more grid barrier each takes an equal share
                // (positions [c N / P, (c + 1) N / P)) of the lists concatenated in CTA order, so the
                // FFN's rows are spread evenly over the SMs whatever the per-CTA counts. The order
                // is fixed by the lists alone, so the result stays deterministic.
                int32_t *gl = a.glist + (size_t)c * STACK_MAX_CHUNK;
                for (int m = tid; m < nn; m += STACK_NT) gl[m] = sneur[m];
                if (tid == 0) a.gcount[c] = nn;
                if (!sync_grid(no_work)) return;
                int *pref = reinterpret_cast<int *>(spb);   // [P + 1]; the logits' biases are dead now
                if (warp == 0) {                           // exclusive prefix of the P counts
                    int run = 0;
                    for (int base = 0; base < P; base += 32) {
                        const int q = base + lane;
                        const int v = q < P ? __ldcg(a.gcount + q) : 0;
                        int x = v;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const int y = __shfl_up_sync(0xffffffffu, x, o);
                            if (lane >= o) x += y;
                        }
                        if (q < P) pref[q] = run + x - v;
                        run += __shfl_sync(0xffffffffu, x, 31);
                    }
                    if (lane == 0) pref[P] = run;
                }
                __syncthreads();
                const int N = pref[P];
                const int lo = (int)((long long)c * N / P);
                nn = (int)((long long)(c + 1) * N / P) - lo;
                for (int m = tid; m < nn; m += STACK_NT) {
                    const int q = lo + m;
                    int a0 = 0, a1 = P;   // pref[a0] <= q < pref[a1]
                    while (a1 - a0 > 1) {
                        const int mid = (a0 + a1) >> 1;
                        if (pref[mid] <= q) a0 = mid;
                        else a1 = mid;
                    }
                    const int i = __ldcg(a.glist + (size_t)a0 * STACK_MAX_CHUNK + (q - pref[a0]));
                    sneur[m] = i;
                    if (!bias_bulk) sbias[m] = Lw.bg ? __ldg(Lw.bg + i) : 0.f;
                }
                __syncthreads();
            }
            stamp(l, 3);
            if (nn == 0) stamp(l, 4);

            // list entries [0, nh) are hot (already in their slots), [nh, nn) cold
            const int HK = a.hot_k, SC = S - HK, hk = min(HK, K);
            int nh = 0;
            while (nh < nn && (sneur[nh] - c) / P < hk) ++nh;
            auto slot_of = [&](int m, uint32_t &par) -> int {
                if (m < nh) {
                    par = (uint32_t)l & 1u;
                    return (sneur[m] - c) / P;
                }
                const uint32_t sq = cseq + (uint32_t)(m - nh);
                par = (sq / (uint32_t)SC) & 1u;
                return HK + (int)(sq % (uint32_t)SC);
            };
            // the first cold neurons' copies: copy q goes to lane q / 16 of warp q % 16 (a warp
            // issues its copies one after another, so every warp takes a few)
            // The FFN's thread mapping: unit ci = tid + cc * STACK_NT (cc < CPT) of UW columns; int4:
            // one 32-bit word of a row (8 columns) per unit, so that all 16 warps take part and a
            // warp's loads of a row are 128 consecutive bytes; else one 16-byte chunk.
            // This thread's units of x_l are requested before the rows (behind a full copy queue
            // their loads would wait microseconds).
            constexpr bool I4 = WT == DT_INT4;
            constexpr int UW = I4 ? 8 : VW;
            const int nunit = d / UW;
            float4 xv[CPT][UW / 4];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                const int ci = tid + cc * STACK_NT;
#pragma unroll
                for (int e4 = 0; e4 < UW / 4; ++e4) {
                    xv[cc][e4] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ci < nunit) xv[cc][e4] = __ldcg(reinterpret_cast<const float4 *>(xl + (size_t)ci * UW) + e4);
                }
            }
            const int NPART = stage_parts<WT, KIND>(a);
            const int cq = lane * SNW + warp, cw = cq / NPART, cj = cq - cw * NPART;   // this thread's copy
            // Only the first batch's rows are requested now, the other free slots' rows once they
            // have landed: requested together with everything else (every CTA asks for most of its
            // rows at this point), the first rows land with the bulk of the layer's FFN bytes.
            // NF must equal the first cold batch's size (nbc below): that batch waits for all of its
            // slots before the held-back copies are issued.
            const int NF = nh == 0 ? max(1, min(4, SC / 2)) : SC;
            if (nh + cw < nn && cw < SC && cw < NF) {
                fence_proxy_async_smem();
                uint32_t par;
                stage_part<WT, KIND>(a, Lw, ring, mbar, slot_of(nh + cw, par), sneur[nh + cw], cj);
            }
            // The next layer's P2 rows that its logits will stream (not staged in the ring) into L2
            // while the FFN leaves the DRAM mostly idle (128-byte lines spread over the threads).
            if (a.pf_p2_ffn && l + 1 < a.L) {
                const int lines = (r * pb + 127) >> 7, kh = KS + (int)(((long long)(K - KS) * a.pf_p2_frac) >> 8);
                for (int j = tid; j < (kh - KS) * lines; j += STACK_NT) {
                    const int k = KS + j / lines;
                    prefetch_line_l2((const char *)s_p2next + (size_t)(c + (size_t)P * k) * r * pb + 128 * (j % lines));
                }
            }
            // this thread's columns of u, scaled, as fp32 pairs for the paired FMAs: int4 (i, i + 4)
            // of its word's 8 columns, the pairing of the decoded nibbles (i4_word_f32x2); else
            // (2j, 2j + 1) of its chunk
            float2 ur[I4 ? 1 : CPT][I4 ? 1 : VW / 2];
            float2 ux[I4 ? CPT : 1][4];
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                if constexpr (I4) {
                    ux[cc][0] = make_float2(xv[cc][0].x * inv, xv[cc][1].x * inv);
                    ux[cc][1] = make_float2(xv[cc][0].y * inv, xv[cc][1].y * inv);
                    ux[cc][2] = make_float2(xv[cc][0].z * inv, xv[cc][1].z * inv);
                    ux[cc][3] = make_float2(xv[cc][0].w * inv, xv[cc][1].w * inv);
                } else {
#pragma unroll
                    for (int e4 = 0; e4 < VW / 4; ++e4) {
                        ur[cc][2 * e4 + 0] = make_float2(xv[cc][e4].x * inv, xv[cc][e4].y * inv);
                        ur[cc][2 * e4 + 1] = make_float2(xv[cc][e4].z * inv, xv[cc][e4].w * inv);
                    }
                }
            }

            float2 yr[I4 ? 1 : CPT][I4 ? 1 : VW / 2];   // else: W_down sums as pairs (2j, 2j + 1)
            float2 yx[I4 ? CPT : 1][4];   // int4: W_down sums as pairs (i, i + 4) of the word's columns
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                if constexpr (I4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) yx[cc][j] = make_float2(0.f, 0.f);
                } else {
#pragma unroll
                    for (int j = 0; j < VW / 2; ++j) yr[cc][j] = make_float2(0.f, 0.f);
                }
            }

            if (G > 1) {
                // Group balance, part 2: wait for the other members' epochs. Member q keeps
                // L_q = min(n_q, K0) of its own entries; the rest of the group's lists (the pool,
                // in member order) is dealt so that member q ends with T / G (+1 for q < T mod G)
                // where it can: it takes pool positions [E_q, E_q + e_q), e_q = max(0, target_q - L_q),
                // cut at the pool's end. The slowest member has about the mean of the G counts
                // instead of its own. Deterministic: fixed by the lists alone.
                const int g0 = c & ~(G - 1), rk = c - g0;
                const unsigned long long epoch = s_base + (unsigned long long)(l + 1);
                bool okw = true;
                if (tid < G && tid != rk) okw = wait_flag_ge(a.gflag + g0 + tid, epoch);
                if (!__syncthreads_and(okw)) {
                    if (tid == 0) {   // wait (bounded) for the first batch's copies, then leave
                        set_status(a.status, ST_TIMEOUT);
                        for (int k = 0; k < nn && k < NF && k < SC; ++k) {
                            uint32_t par;
                            const int slot = slot_of(k, par);
                            mbar_wait(&mbar[slot], par);
                        }
                    }
                    return;
                }
                // pool prefix [G + 1], this member's range [2], the members' counts [G] (the logits'
                // biases are dead now)
                int *pp = reinterpret_cast<int *>(spb), *nq = pp + G + 3;
                if (tid == 0) {
                    int T = 0, run = 0;
                    for (int q = 0; q < G; ++q) {
                        nq[q] = __ldcg(a.gcount + g0 + q);
                        T += nq[q];
                    }
                    for (int q = 0; q < G; ++q) {
                        pp[q] = run;
                        run += nq[q] - min(nq[q], K0);
                    }
                    pp[G] = run;
                    int E = 0, myE = 0, mye = 0;
                    for (int q = 0; q < G; ++q) {
                        const int eq = max(0, T / G + (q < T % G ? 1 : 0) - min(nq[q], K0));
                        if (q == rk) {
                            myE = E;
                            mye = eq;
                        }
                        E += eq;
                    }
                    pp[G + 1] = myE;
                    pp[G + 2] = max(0, min(myE + mye, run) - myE);
                }
                __syncthreads();
                const int E0 = pp[G + 1], ne = pp[G + 2];
                for (int m = tid; m < ne; m += STACK_NT) {
                    const int q = E0 + m;
                    int a0 = 0;   // pp[a0] <= q < pp[a0 + 1]
                    while (a0 + 1 < G && pp[a0 + 1] <= q) ++a0;
                    const int i = __ldcg(a.glist + (size_t)(g0 + a0) * STACK_MAX_CHUNK + K0 + (q - pp[a0]));
                    sneur[nn + m] = i;
                    if (!bias_bulk) sbias[nn + m] = Lw.bg ? __ldg(Lw.bg + i) : 0.f;
                }
                __syncthreads();
                const int n0 = nn;
                nn += ne;
                if (cw >= n0 && cw < NF && cw < nn && cw < SC) {   // first-batch entries the own list left empty
                    fence_proxy_async_smem();
                    uint32_t par;
                    stage_part<WT, KIND>(a, Lw, ring, mbar, slot_of(cw, par), sneur[cw], cj);
                }
            }

            // Neurons are reduced a batch at a time, in list order (hot ones first): one CTA-wide
            // synchronisation per batch. Hot batches take up to NB resident neurons; a cold batch
            // waits only on copies issued at least one batch earlier, which needs 2 * nbc <= SC.
            // Cold list entry m0 + k sits in slot HK + cs + k (wrapping at SC, parity flipped on the
            // wrap), where (cs, cp) are the slot and parity of the batch's first entry.
            constexpr int NB = 4;
            constexpr int NV = KIND == KIND_GATED ? 2 * NB : NB;   // per-warp partial sums of a batch
            const int nbc = max(1, min(NB, SC / 2));
            uint32_t cs = cseq % (uint32_t)SC, cp = (cseq / (uint32_t)SC) & 1u;
            auto slot_at = [&](int m0, bool cold, int k, uint32_t &par) -> int {
                if (!cold) {
                    par = (uint32_t)l & 1u;
                    return (sneur[m0 + k] - c) / P;
                }
                uint32_t sk = cs + (uint32_t)k;
                par = cp;
                if (sk >= (uint32_t)SC) {
                    sk -= (uint32_t)SC;
                    par ^= 1u;
                }
                return HK + (int)sk;
            };
            int bi = 0;
            for (int m0 = 0; m0 < nn; ++bi) {
                const bool cold = m0 >= nh;
                const int mb = cold ? min(nbc, nn - m0) : min(NB, nh - m0);
                bool got = true;
                float v[NV];   // gated: gate and up partial of neuron k at 2k, 2k + 1; else gate at k
#pragma unroll
                for (int j = 0; j < NV; ++j) v[j] = 0.f;
                // the batch's slots land first; then every thread walks its columns of all the batch's
                // rows at once, one dependent chain per neuron and row, the chains interleaved (each
                // neuron's additions keep their order: the same bits as one neuron at a time)
                const unsigned char *sls[NB];
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    sls[k] = sls[0];   // an unused neuron reads the first neuron's (landed) slot; its sums are never used
                    if (k < mb) {
                        uint32_t par;
                        const int slot = slot_at(m0, cold, k, par);
                        sls[k] = ring + (size_t)slot * a.slot_bytes;
                        got = got && mbar_wait(&mbar[slot], par);
                    }
                }
                // the held-back first copies (also after a timed-out wait: the give-up path below
                // waits for every slot of the list's next SC entries)
                if (bi == 0 && nh + cw < nn && cw >= NF && cw < SC) {
                    fence_proxy_async_smem();
                    uint32_t par;
                    stage_part<WT, KIND>(a, Lw, ring, mbar, slot_of(nh + cw, par), sneur[nh + cw], cj);
                }
                if (got) {
                    constexpr int GI = KIND == KIND_GATED ? 2 : 1;
#pragma unroll
                    for (int cc = 0; cc < CPT; ++cc) {
                        const int ci = tid + cc * STACK_NT;
                        if (ci >= nunit) break;
                        if constexpr (I4) {
                            // the nibbles decoded by fp16 bit tricks (no integer-to-float conversions,
                            // which share the integer pipe with the shifts), two FMAs per instruction:
                            // neuron k's chain pairs columns (i, i + 4) of the word, then one scale
                            // (group ci / 16 of 128 columns) per word
#pragma unroll
                            for (int g = 0; g < GI; ++g) {   // gate rows, then up rows
                                uint32_t wv[NB];
#pragma unroll
                                for (int k = 0; k < NB; ++k) wv[k] = reinterpret_cast<const uint32_t *>(sls[k] + g * rowb)[ci];
#pragma unroll
                                for (int k = 0; k < NB; ++k) {
                                    float2 pv[4];
                                    i4_word_f32x2(wv[k], pv);
                                    float2 t2 = make_float2(pv[0].x * ux[cc][0].x, pv[0].y * ux[cc][0].y);
#pragma unroll
                                    for (int i = 1; i < 4; ++i) t2 = ffma2(pv[i], ux[cc][i], t2);
                                    const __half *ss = reinterpret_cast<const __half *>(sls[k] + ROWS * rowb);
                                    v[GI * k + g] = fmaf(__half2float(ss[g * (d / 128) + (ci >> 4)]), t2.x + t2.y, v[GI * k + g]);
                                }
                            }
                        } else {
#pragma unroll
                            for (int g = 0; g < GI; ++g) {   // gate rows, then up rows
                                float wf[NB][VW];
#pragma unroll
                                for (int k = 0; k < NB; ++k)
                                    unpack<WT>(reinterpret_cast<const uint4 *>(sls[k] + g * rowb)[ci], wf[k]);
#pragma unroll
                                for (int k = 0; k < NB; ++k) {   // paired chains (even, odd columns), added at the end
                                    float2 t2 = make_float2(wf[k][0] * ur[cc][0].x, wf[k][1] * ur[cc][0].y);
#pragma unroll
                                    for (int j = 1; j < VW / 2; ++j) t2 = ffma2(make_float2(wf[k][2 * j], wf[k][2 * j + 1]), ur[cc][j], t2);
                                    v[GI * k + g] += t2.x + t2.y;
                                }
                            }
                        }
                    }
                }
                {   // lane L ends with this warp's sum of value L / (32 / NV)
                    const float t = warp_transpose_sum<NV>(v, lane);
                    if ((lane & (32 / NV - 1)) == 0) red[bi & 1][warp][lane / (32 / NV)] = t;
                }
                if (!__syncthreads_and(got)) {
                    // give up: wait (bounded) for this CTA's copies still in flight, then leave
                    if (tid == 0) {
                        set_status(a.status, ST_TIMEOUT);
                        for (int k = 0; k < hk; ++k) mbar_wait(&mbar[k], (uint32_t)l & 1u);
                        for (int k = max(m0, nh); k < nn && k < max(m0, nh) + SC; ++k) {
                            uint32_t par;
                            const int slot = slot_of(k, par);
                            mbar_wait(&mbar[slot], par);
                        }
                    }
                    return;
                }
                if (bi == 0) stamp(l, 4);
                // the previous cold batch's slots are free: entry k + SC takes entry k's slot
                // (copy j of the batch's w-th refill goes to the thread that took copy j of cold entry w)
                if (cold && m0 - nbc >= nh && cw < nbc && m0 - nbc + cw + SC < nn) {
                    fence_proxy_async_smem();
                    int sk = (int)cs - nbc + cw;
                    if (sk < 0) sk += SC;
                    stage_part<WT, KIND>(a, Lw, ring, mbar, HK + sk, sneur[m0 - nbc + cw + SC], cj);
                }
                // The batch's sums, all its neurons at once (one shuffle chain instead of one per
                // neuron): lane (w, h) = (lane & 15, lane >> 4) holds warp w's partials of values h,
                // h + 2, ... (value v = GI k + g: gated g = 0 gate, g = 1 up; else v = k), each added
                // over the 16 warps in a fixed butterfly order, so that value v ends in lane
                // 16 (v & 1), register v / 2, with the same bits as one neuron at a time.
                constexpr int GV = KIND == KIND_GATED ? 2 : 1, NH = NV / 2;
                float sv[NH];
#pragma unroll
                for (int j = 0; j < NH; ++j) sv[j] = red[bi & 1][lane & 15][2 * j + (lane >> 4)];
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
                    for (int j = 0; j < NH; ++j) sv[j] += __shfl_xor_sync(0xffffffffu, sv[j], o);
                float hvb[NB];   // h of the batch's neurons (0 past the batch's end)
#pragma unroll
                for (int k = 0; k < NB; ++k) {
                    const int v = GV * k, mk = k < mb ? m0 + k : m0;
                    float g = __shfl_sync(0xffffffffu, sv[v >> 1], 16 * (v & 1));
                    g += bias_bulk ? reinterpret_cast<const float *>(sls[k] + bias_off)[sneur[mk] & 3] : sbias[mk];
                    float hv = fmaxf(g, 0.f);
                    if (KIND == KIND_GATED) hv *= __shfl_sync(0xffffffffu, sv[(v + 1) >> 1], 16 * ((v + 1) & 1));
                    hvb[k] = k < mb ? hv : 0.f;
                }
                // W_down: every output element takes the batch's neurons in list order (the same
                // bits as one neuron at a time); a full batch interleaves the neurons' rows.
                if (mb == NB) {
#pragma unroll
                    for (int cc = 0; cc < CPT; ++cc) {
                        const int ci = tid + cc * STACK_NT;
                        if (ci >= nunit) break;
                        if constexpr (I4) {
                            uint32_t w32[NB];
                            float hs[NB];
#pragma unroll
                            for (int k = 0; k < NB; ++k) {
                                w32[k] = reinterpret_cast<const uint32_t *>(sls[k] + (ROWS - 1) * rowb)[ci];
                                const __half *ss = reinterpret_cast<const __half *>(sls[k] + ROWS * rowb + (ROWS - 1) * sclb);
                                hs[k] = hvb[k] * __half2float(ss[ci >> 4]);
                            }
#pragma unroll
                            for (int k = 0; k < NB; ++k) {
                                const float2 hs2 = make_float2(hs[k], hs[k]);
                                float2 pv[4];
                                i4_word_f32x2(w32[k], pv);
#pragma unroll
                                for (int i = 0; i < 4; ++i) yx[cc][i] = ffma2(hs2, pv[i], yx[cc][i]);
                            }
                        } else {
                            uint4 w4[NB];
#pragma unroll
                            for (int k = 0; k < NB; ++k) w4[k] = reinterpret_cast<const uint4 *>(sls[k] + (ROWS - 1) * rowb)[ci];
#pragma unroll
                            for (int k = 0; k < NB; ++k) {
                                float wf[VW];
                                unpack<WT>(w4[k], wf);
#pragma unroll
                                for (int j = 0; j < VW / 2; ++j)
                                    yr[cc][j] = ffma2(make_float2(hvb[k], hvb[k]), make_float2(wf[2 * j], wf[2 * j + 1]), yr[cc][j]);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < NB; ++k) {
                        if (k >= mb) break;
                        const unsigned char *sl = sls[k];
#pragma unroll
                        for (int cc = 0; cc < CPT; ++cc) {
                            const int ci = tid + cc * STACK_NT;
                            if (ci >= nunit) break;
                            if constexpr (I4) {
                                const __half *ss = reinterpret_cast<const __half *>(sl + ROWS * rowb + (ROWS - 1) * sclb);
                                const float hs = hvb[k] * __half2float(ss[ci >> 4]);
                                const float2 hs2 = make_float2(hs, hs);
                                float2 pv[4];
                                i4_word_f32x2(reinterpret_cast<const uint32_t *>(sl + (ROWS - 1) * rowb)[ci], pv);
#pragma unroll
                                for (int i = 0; i < 4; ++i) yx[cc][i] = ffma2(hs2, pv[i], yx[cc][i]);
                            } else {
                                float wf[VW];
                                unpack<WT>(reinterpret_cast<const uint4 *>(sl + (ROWS - 1) * rowb)[ci], wf);
#pragma unroll
                                for (int j = 0; j < VW / 2; ++j)
                                    yr[cc][j] = ffma2(make_float2(hvb[k], hvb[k]), make_float2(wf[2 * j], wf[2 * j + 1]), yr[cc][j]);
                            }
                        }
                    }
                }
                if (cold) {
                    cs += (uint32_t)mb;
                    if (cs >= (uint32_t)SC) {
                        cs -= (uint32_t)SC;
                        cp ^= 1u;
                    }
                }
                m0 += mb;
            }
            cseq += (uint32_t)(nn - nh);
            float *pq = a.part + (size_t)c * d;
#pragma unroll
            for (int cc = 0; cc < CPT; ++cc) {
                const int ci = tid + cc * STACK_NT;
                if (ci >= nunit) break;
#pragma unroll
                for (int e4 = 0; e4 < UW / 4; ++e4) {
                    float4 y4;
                    if constexpr (I4) {   // the word's columns 0..3 are the pairs' x halves, 4..7 their y halves
                        y4 = e4 ? make_float4(yx[cc][0].y, yx[cc][1].y, yx[cc][2].y, yx[cc][3].y)
                                : make_float4(yx[cc][0].x, yx[cc][1].x, yx[cc][2].x, yx[cc][3].x);
                    } else {
                        y4 = make_float4(yr[cc][2 * e4].x, yr[cc][2 * e4].y, yr[cc][2 * e4 + 1].x, yr[cc][2 * e4 + 1].y);
                    }
                    reinterpret_cast<float4 *>(pq + (size_t)ci * UW)[e4] = y4;
                }
            }
            stamp(l, 5);
        }
        // Once every thread is done with the ring (the barrier's CTA sync), the next layer's hot
        // rows (a whole layer before their predictor runs) or its staged P2 rows are requested
        // while this CTA waits for the others.
        if (l + 1 < a.L) {
            expect_p2(l + 1);
            if (tid == 0 && a.hot_k > 0) s_pend = (l + 1) & 1;
        }
        if (!sync_grid([&] {
                if (l + 1 < a.L && a.pf_p1 == 1) prefetch_p1(a.layers[l + 1]);   // just in time
                if (l + 1 < a.L && a.hot_k > 0) issue_hot(a.layers[l + 1], l);
                if (l + 1 < a.L && KS > 0) stage_p2(s_p2next);
            }))
            return;
        stamp(l, 6);

        // ------------------------------------------------------------ D: fixed-order reduction + residual
        {
            // Up to four of this CTA's slices at a time, every partial load of them in flight together.
            // Thread (g, c4) adds partials g, g + 64, ... of float4 column c4; the 64 groups are then
            // added in a fixed tree (4 per warp by shuffles, 16 warps through shared memory).
            const int nsl = (d + STACK_SLICE - 1) / STACK_SLICE;
            const int c4 = tid & 7, g = tid >> 3;   // 8 float4 per slice, 64 groups of partials
            float4 *red4 = scr4;                   // [16 warps][4 slices][8 columns]
            for (int s0 = c; s0 < nsl; s0 += 4 * P) {
                float4 acc[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    const int col = (s0 + j * P) * STACK_SLICE + c4 * 4;
                    if (s0 + j * P < nsl && col < d) {
#pragma unroll 3
                        for (int q = g; q < P; q += STACK_NT / 8) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.part + (size_t)q * d + col));
                            acc[j].x += v.x; acc[j].y += v.y; acc[j].z += v.z; acc[j].w += v.w;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {   // lanes l, l ^ 8, l ^ 16, l ^ 24: the warp's 4 groups
#pragma unroll
                    for (int o = 8; o <= 16; o <<= 1) {
                        acc[j].x += __shfl_xor_sync(0xffffffffu, acc[j].x, o);
                        acc[j].y += __shfl_xor_sync(0xffffffffu, acc[j].y, o);
                        acc[j].z += __shfl_xor_sync(0xffffffffu, acc[j].z, o);
                        acc[j].w += __shfl_xor_sync(0xffffffffu, acc[j].w, o);
                    }
                    if (lane < 8) red4[(warp * 4 + j) * 8 + lane] = acc[j];
                }
                __syncthreads();
                if (tid < 32) {   // slice j = tid / 8, column c4
                    const int j = tid >> 3, s = s0 + j * P;
                    const int col = s * STACK_SLICE + c4 * 4;
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int w = 0; w < SNW; ++w) {   // fixed order
                        const float4 v = red4[(w * 4 + j) * 8 + c4];
                        y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
                    }
                    float ss = 0.f;
                    if (s < nsl && col < d) {
                        const float4 xv = __ldcg(reinterpret_cast<const float4 *>(xl + col));
                        y.x += xv.x; y.y += xv.y; y.z += xv.z; y.w += xv.w;
                        *reinterpret_cast<float4 *>(xn + col) = y;
                        if (a.x_layers) *reinterpret_cast<float4 *>(a.x_layers + (size_t)l * d + col) = y;
                        ss = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
                    }
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    if (c4 == 0 && s < nsl) a.sumsq[s] = ss;
                }
                __syncthreads();
            }
            // on request: the ascending active list of this layer, from its complete mask
            if (a.idx_out) {
                const int wa = (int)((long long)c * W / P), wz = (int)((long long)(c + 1) * W / P);
                int before = 0;
                for (int w = tid; w < wa; w += STACK_NT) before += __popc(__ldcg(a.maskw + (size_t)l * W + w));
                before = warp_sum_int(before);
                if (lane == 0) wsum[warp] = before;
                __syncthreads();
                if (tid == 0) {
                    int off = 0;
                    for (int w = 0; w < SNW; ++w) off += wsum[w];
                    for (int w = wa; w < wz; ++w) {
                        uint32_t m = __ldcg(a.maskw + (size_t)l * W + w);
                        while (m) {
                            a.idx_out[(size_t)l * f + off++] = w * 32 + __ffs(m) - 1;
                            m &= m - 1;
                        }
                    }
                }
                __syncthreads();
            }
            stamp(l, 7);
            if (l + 1 < a.L && !sync_grid(no_work)) return;
        }
    }
    // the last layer's hot copies of neurons that were not active have landed before the CTA leaves
    if (lane == 0)
        for (int k = warp; k < min(a.hot_k, K); k += SNW)
            if (!mbar_wait(&mbar[k], (uint32_t)(a.L - 1) & 1u)) set_status(a.status, ST_TIMEOUT);
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
    // units per thread of the FFN's mapping: 32-bit words (8 columns) for int4, else 16-byte chunks
    const int cpt = (a.d / (WT == DT_INT4 ? 8 : Vec<WT>::N) + STACK_NT - 1) / STACK_NT;
    auto pick = [&](auto k1, auto k2, auto k3) -> cudaError_t {
        return cpt <= 1 ? go(k1) : (cpt == 2 ? go(k2) : (cpt == 3 ? go(k3) : cudaErrorNotSupported));
    };
    const bool gated = kind == KIND_GATED;
    if constexpr (WT == DT_INT4) {   // words per thread 2 (d <= 8192), 3 (d <= 12288), 4 (d <= 16384)
        auto pick4 = [&](auto k2, auto k3, auto k4) -> cudaError_t {
            return cpt <= 2 ? go(k2) : (cpt == 3 ? go(k3) : (cpt == 4 ? go(k4) : cudaErrorNotSupported));
        };
        if (pdt == DT_F16)
            return gated ? pick4(k_decode_stack<WT, DT_F16, KIND_GATED, 2>, k_decode_stack<WT, DT_F16, KIND_GATED, 3>,
                                 k_decode_stack<WT, DT_F16, KIND_GATED, 4>)
                         : pick4(k_decode_stack<WT, DT_F16, KIND_RELU, 2>, k_decode_stack<WT, DT_F16, KIND_RELU, 3>,
                                 k_decode_stack<WT, DT_F16, KIND_RELU, 4>);
        if (pdt == DT_BF16)
            return gated ? pick4(k_decode_stack<WT, DT_BF16, KIND_GATED, 2>, k_decode_stack<WT, DT_BF16, KIND_GATED, 3>,
                                 k_decode_stack<WT, DT_BF16, KIND_GATED, 4>)
                         : pick4(k_decode_stack<WT, DT_BF16, KIND_RELU, 2>, k_decode_stack<WT, DT_BF16, KIND_RELU, 3>,
                                 k_decode_stack<WT, DT_BF16, KIND_RELU, 4>);
    } else {
        if (pdt == WT)
            return gated ? pick(k_decode_stack<WT, WT, KIND_GATED, 1>, k_decode_stack<WT, WT, KIND_GATED, 2>,
                                k_decode_stack<WT, WT, KIND_GATED, 3>)
                         : pick(k_decode_stack<WT, WT, KIND_RELU, 1>, k_decode_stack<WT, WT, KIND_RELU, 2>,
                                k_decode_stack<WT, WT, KIND_RELU, 3>);
    }
    return cudaErrorNotSupported;
}

}  // namespace pi
