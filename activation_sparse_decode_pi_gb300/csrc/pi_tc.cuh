// pi_tc.cuh -- the batch >= 16 path of the sparse FFN on the 5th-generation tensor cores.
//
// "PowerInfer" summary page, Methodology: neuron-aware sparse operators touch only the
// rows of the neurons the predictor marked. With 16 or more sequences decoded together
// the gathered rows meet enough activation columns to make each one a real contraction:
//
//   TC_PRED_HIDDEN  hp  = ReLU(U . P1T^T)             rows of P1T,  K = d
//   TC_LOGITS       z   = hp . P2T^T + b_p; mask; idx rows of P2T,  K = r
//   TC_GATED        h   = ReLU(U . Wg^T + bg) * (U . Wu^T)  rows Wg/Wu[idx], K = d
//   TC_RELU         h   = ReLU(U . W1^T + b1)               rows W1[idx],    K = d
//   TC_DOWN         y   = H . WdT[idx]  (+ residual)        columns of d, K = active neurons
//
// Every product is D[128 x NB] = A[128 x K] * X[NB x K]^T with fp32 accumulation in
// tensor memory: A is 128 gathered weight rows (K-major) or, for TC_DOWN, a 128-column
// slice of 64 gathered W_down^T rows per step (MN-major); X is the activation tile,
// batch rows padded to NB with zeros. The activations are fp32 on the path; they enter
// the tensor core as the weights' 16-bit type split into hi + lo, two products per step,
// so the result keeps ~24 bits of the activation, not 8 or 11.
//
// Work split (stream-K): the T = tiles x k-blocks iterations are cut into one equal
// contiguous range per CTA. A tile finished inside one CTA is written out directly; a
// tile shared by several CTAs leaves fp32 partials, and the CTA whose share completes
// the tile's k-block count adds them in CTA order, so the result does not depend on
// timing (only on the grid size).
//
// Roles: warps 0-3 drain the accumulators (TMEM lane quarter = warp), warps 4-11 copy
// the operands into a shared-memory ring with cp.async (16 bytes a thread, swizzled
// into the 128-byte canonical layouts), warp 12 owns TMEM and one of its threads issues
// the MMAs. Accumulators are double-buffered so the drain overlaps the next tile.
// Every wait is bounded (200 ms): on expiry the kernel records PI_ERR_TIMEOUT, stops,
// waits for its own copies and products, frees its TMEM and returns.
#pragma once

#include <type_traits>

#include "pi_internal.h"
#include "pi_umma.cuh"

namespace pi {

constexpr int TC_PROD = 384;                       // producer threads (warps 4..11)
constexpr int TC_MMA_WARP = 4 + TC_PROD / 32;      // warp 12: TMEM owner and MMA issuer
constexpr int TC_THREADS = 32 * (TC_MMA_WARP + 1);

__host__ __device__ constexpr uint32_t tc_tmem_cols(uint32_t need)
{
    return need <= 32 ? 32u : need <= 64 ? 64u : need <= 128 ? 128u : need <= 256 ? 256u : 512u;
}

// bytes of one pipeline step: weight blocks, then activation hi and lo blocks
__host__ __device__ constexpr uint32_t tc_stage_bytes(int mode, int nb, int w)
{
    return mode == TC_DOWN ? (uint32_t)w * 16384u + 2u * (uint32_t)nb * 128u
                           : (mode == TC_GATED ? 2u : 1u) * (uint32_t)w * 16384u + 2u * (uint32_t)w * nb * 128u;
}

// first iteration of CTA c's stream-K range
__device__ __forceinline__ long long tc_begin(int c, long long T, int P) { return (long long)c * T / P; }
// CTA whose range holds iteration `it`
__device__ __forceinline__ int tc_owner(long long it, long long T, int P)
{
    return (int)(((it + 1) * P + T - 1) / T - 1);
}

// Ticket on a tile counter: release this CTA's partial (written before the caller's
// CTA-level barrier), and acquire everyone else's when the returned value completes the tile.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// W: 64-wide K blocks per pipeline step (row modes), or 128-column W_down^T slices per tile (TC_DOWN).
//
// Shared memory of one step: the weight blocks (16 KB each), then per K block the activation
// tile as 2*NB rows, hi rows first, lo rows after: one MMA with N = 2*NB multiplies a weight
// block by both halves, and the drain adds accumulator columns b and NB + b.
template <int WT, int MODE, int NB, int W>
__global__ void __launch_bounds__(TC_THREADS, 1) k_tc(const TcArgs a)
{
    constexpr bool DOWN = MODE == TC_DOWN;
    constexpr int NMAT = MODE == TC_GATED ? 2 : 1;
    constexpr int NACC = DOWN ? W : NMAT;                  // accumulators per tile
    constexpr int KW = DOWN ? 1 : W;                       // 64-wide K blocks per step
    constexpr uint32_t BLK = 16384u;                       // one 128 x 64 (or 64 x 128) weight block
    constexpr uint32_t XB = (uint32_t)NB * 128u;           // one NB x 64 activation half
    constexpr uint32_t A_BYTES = (uint32_t)(DOWN ? W : NMAT * KW) * BLK;
    constexpr uint32_t STAGE = tc_stage_bytes(MODE, NB, W);
    constexpr uint32_t ACOLS = 2u * NB;                    // TMEM columns of one accumulator (hi | lo)
    constexpr uint32_t ACC = (uint32_t)NACC * ACOLS;       // TMEM columns of one buffer
    constexpr int NBUF = 2 * ACC <= 512 ? 2 : 1;           // accumulator buffers (drain overlaps the next tile)
    constexpr uint32_t TCOLS = tc_tmem_cols(NBUF * ACC);
    constexpr uint32_t PCOLS = (uint32_t)(NACC * NB);      // fp32 columns of one partial
    constexpr uint32_t IDESC = f16_idesc(WT == DT_BF16 ? 1 : 0, DOWN ? 1 : 0, 0, 128, 2 * NB);
    constexpr int CH = 1024 / TC_PROD + (1024 % TC_PROD ? 1 : 0);   // weight chunks per thread and block
    static_assert(NB % 16 == 0 && NB >= 16 && NB <= 128, "batch tile");
    static_assert(ACC <= 512, "accumulators exceed tensor memory");
    static_assert(A_BYTES + 2u * KW * XB == STAGE, "stage layout");

    extern __shared__ uint8_t dsm[];
    __shared__ uint64_t full[TC_MAX_STAGES], empty[TC_MAX_STAGES], accf[2], acce[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int s_abort;    // any role gave up: the others stop early
    __shared__ volatile int s_dabort;   // written by drain threads only, read after a drain barrier
    __shared__ int s_last, s_wsum[TC_THREADS / 32];
    __shared__ int s_compact;           // this CTA completed the last logits tile: it lists the active rows

    const uint32_t sbase = (smem_u32(dsm) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], TC_PROD);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&accf[s], 1);
            mbar_init(&acce[s], 4);
        }
        mbar_init(&fin, 1);
        s_abort = 0;
        s_dabort = 0;
        s_compact = 0;
        fence_mbar_init();
    }
    if (warp == TC_MMA_WARP) tmem_alloc(&tmem_base, TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    pdl_launch_dependents();
    // Weight rows that do not depend on the previous kernel (the predictor's: no list, no
    // count) are requested for the ring's first steps before waiting for that kernel, so their
    // latency overlaps its tail; the activation tiles follow after the wait.
    constexpr bool PRE_OK = MODE == TC_PRED_HIDDEN || MODE == TC_LOGITS;
    const bool pre = PRE_OK && a.count == nullptr && a.idx == nullptr;
    uint32_t npre = 0;
    if constexpr (PRE_OK) {
        if (pre && warp >= 4 && warp < TC_MMA_WARP) {
            const int p = threadIdx.x - 128;
            const int tiles0 = (a.n_static + 127) / 128, KB0 = a.K / (64 * KW);
            const long long T0 = (long long)tiles0 * KB0;
            const long long b0 = T0 ? tc_begin(blockIdx.x, T0, gridDim.x) : 0;
            const long long e0 = T0 ? tc_begin(blockIdx.x + 1, T0, gridDim.x) : 0;
            for (long long it = b0; it < e0 && npre < (uint32_t)S; ++it, ++npre) {
                const int t = (int)(it / KB0), kb = (int)(it - (long long)t * KB0);
                const uint32_t st = sbase + npre * STAGE;
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int c = p + TC_PROD * i;
                    const int j = t * 128 + (c >> 3);
                    if (c >= 1024) continue;
                    const bool ok = j < a.n_static;
                    const uint16_t *src = a.w0 + (size_t)(ok ? a.row0 + j : 0) * a.K + (c & 7) * 8;
#pragma unroll
                    for (int w = 0; w < KW; ++w)
                        cp_async16(st + w * BLK + sw128_off(c >> 3, c & 7), src + (kb * KW + w) * 64, ok ? 16u : 0u);
                }
            }
        }
    }
    pdl_wait();

    // ---- problem size and this CTA's stream-K range
    int n = a.n_static;
    if (a.count) {
        n = __ldcg(a.count);
        if (n < 0 || n > a.f) {
            if (threadIdx.x == 0) set_status(a.status, ST_DEVICE_CHECK);
            n = n < 0 ? 0 : a.f;
        }
    }
    const int tiles = DOWN ? a.d / (128 * W) : (n + 127) / 128;
    const int KB = DOWN ? (n + 63) / 64 : a.K / (64 * KW);   // pipeline steps per tile
    const long long T = (long long)tiles * KB;
    const int P = gridDim.x, cta = blockIdx.x;
    const long long it0 = T ? tc_begin(cta, T, P) : 0, it1 = T ? tc_begin(cta + 1, T, P) : 0;

    if (DOWN && n == 0) {   // no active neuron: y = 0
        for (int e = cta * TC_THREADS + threadIdx.x; e < a.B * a.d; e += P * TC_THREADS)
            a.out[e] = a.xin ? __ldcg(a.xin + e) : 0.f;
    }

    if (warp >= 4 && warp < TC_MMA_WARP) {
        // ================================================================ producers
        const int p = threadIdx.x - 128;
        const uint16_t *const W0 = a.w0;
        uint32_t q = 0;
        bool bad = false;
        // the step's slot is complete for the MMA when every producer's copies into it have
        // landed: each thread's arrival is triggered by its own copies' completion
        auto step_done = [&]() { cp_async_arrive_noinc(&full[q % S]); };
        // activation tile of K block kb: NB hi rows then NB lo rows, 8 chunks of 16 bytes a row
        auto load_x = [&](uint32_t xs, int kb) {
            for (int c = p; c < 2 * NB * 8; c += TC_PROD) {
                const int xr = c >> 3, xc = c & 7;
                const uint16_t *src = (xr < NB ? a.xhi : a.xlo) + (size_t)(xr % NB) * a.ldx + kb * 64 + xc * 8;
                cp_async16(xs + sw128_off(xr, xc), src, 16u);
            }
        };
        if constexpr (!DOWN) {
            // 128 gathered rows x (KW x 64) columns per step; chunk c = row * 8 + 16-byte piece
            const uint16_t *rp[NMAT][CH];
            for (long long it = it0; it < it1 && !s_abort;) {
                const int t = (int)(it / KB), kb0 = (int)(it - (long long)t * KB);
                const int kb1 = (int)min((long long)KB, kb0 + (it1 - it));
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int c = p + TC_PROD * i;
                    const int j = t * 128 + (c >> 3);
                    int id = -1;
                    if (c < 1024 && j < n) {
                        id = a.idx ? __ldcg(a.idx + j) : a.row0 + j;
                        if (id < 0 || id >= a.f) {
                            bad = true;
                            id = -1;
                        }
                    }
                    rp[0][i] = id >= 0 ? W0 + (size_t)id * a.K + (c & 7) * 8 : nullptr;
                    if constexpr (NMAT == 2) rp[1][i] = id >= 0 ? a.w1 + (size_t)id * a.K + (c & 7) * 8 : nullptr;
                }
                for (int kb = kb0; kb < kb1; ++kb, ++q) {
                    const int slot = (int)(q % (uint32_t)S);
                    if (q >= (uint32_t)S && !mbar_wait(&empty[slot], ((q / S) - 1) & 1)) {
                        set_status(a.status, ST_TIMEOUT);
                        s_abort = 1;
                        break;
                    }
                    const uint32_t st = sbase + (uint32_t)slot * STAGE;
                    const bool need_a = q >= npre;   // the first npre steps' rows were requested before the wait
#pragma unroll
                    for (int w = 0; w < KW; ++w) {
                        const int k0 = (kb * KW + w) * 64;
#pragma unroll
                        for (int m = 0; m < NMAT; ++m)
#pragma unroll
                            for (int i = 0; i < CH; ++i) {
                                const int c = p + TC_PROD * i;
                                if (c < 1024 && need_a) {
                                    const uint16_t *src = rp[m][i];
                                    cp_async16(st + (m * KW + w) * BLK + sw128_off(c >> 3, c & 7), src ? src + k0 : W0,
                                               src ? 16u : 0u);
                                }
                            }
                        load_x(st + A_BYTES + 2 * w * XB, kb * KW + w);
                    }
                    step_done();
                }
                it += kb1 - kb0;
            }
        } else {
            // W_down^T: 64 neuron rows x (W x 128) columns per step; chunk c = row * 16 + 16-byte piece.
            // Neuron ids of the next ID_AHEAD steps live in registers, so the list reads overlap the
            // copies instead of stalling each step; -2 marks the zero rows past the list's end.
            constexpr int ID_AHEAD = 4;
            int ids[ID_AHEAD][CH];
            auto load_ids = [&](long long it, int (&dst)[CH]) {
                const int kb = it < it1 ? (int)(it % KB) : 0;
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int c = p + TC_PROD * i;
                    const int j = kb * 64 + (c >> 4);
                    dst[i] = (it < it1 && c < 1024 && j < n) ? __ldcg(a.idx + j) : -2;
                }
            };
#pragma unroll
            for (int u = 0; u < ID_AHEAD; ++u) load_ids(it0 + u, ids[u]);
            for (long long its = it0; its < it1 && !s_abort; its += ID_AHEAD)
#pragma unroll
            for (int u = 0; u < ID_AHEAD; ++u) {
                const long long it = its + u;
                if (it >= it1 || s_abort) break;
                const int t = (int)(it / KB), kb = (int)(it - (long long)t * KB);
                const int slot = (int)(q % (uint32_t)S);
                if (q >= (uint32_t)S && !mbar_wait(&empty[slot], ((q / S) - 1) & 1)) {
                    set_status(a.status, ST_TIMEOUT);
                    s_abort = 1;
                    break;
                }
                const uint32_t st = sbase + (uint32_t)slot * STAGE;
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int c = p + TC_PROD * i;
                    if (c >= 1024) continue;
                    int id = ids[u][i];
                    if (id >= a.f || id < -2 || id == -1) {
                        bad = true;
                        id = -2;
                    }
                    const uint16_t *src = id >= 0 ? W0 + (size_t)id * a.d + (size_t)t * 128 * W + (c & 15) * 8 : nullptr;
                    const uint32_t dst = st + (uint32_t)((c & 15) >> 3) * 8192u + sw128_off(c >> 4, c & 7);
#pragma unroll
                    for (int w = 0; w < W; ++w) cp_async16(dst + w * BLK, src ? src + w * 128 : W0, src ? 16u : 0u);
                }
                load_x(st + A_BYTES, kb);
                load_ids(it + ID_AHEAD, ids[u]);   // consumed ID_AHEAD steps later
                step_done();
                ++q;
            }
        }
        cp_async_wait_all();
        if (bad) set_status(a.status, ST_DEVICE_CHECK);
    } else if (warp == TC_MMA_WARP) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            uint32_t q = 0, si = 0;
            for (long long it = it0; it < it1 && !s_abort; ++si) {
                const int t = (int)(it / KB), kb0 = (int)(it - (long long)t * KB);
                const int kb1 = (int)min((long long)KB, kb0 + (it1 - it));
                const uint32_t ab = si % NBUF;
                if (si >= (uint32_t)NBUF && !mbar_wait(&acce[ab], ((si / NBUF) - 1) & 1)) {
                    set_status(a.status, ST_TIMEOUT);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + ab * ACC;
                for (int kb = kb0; kb < kb1; ++kb, ++q) {
                    const int slot = (int)(q % (uint32_t)S);
                    if (!mbar_wait(&full[slot], (q / S) & 1)) {
                        set_status(a.status, ST_TIMEOUT);
                        s_abort = 1;
                        break;
                    }
                    fence_proxy_async_smem();   // the producers' copies, seen through the barrier, to the tensor core
                    tc_fence_after();
                    const uint32_t st = sbase + (uint32_t)slot * STAGE;
                    const uint64_t a0 = sw128_desc(st, DOWN ? 8192u : 16u, 1024u);
                    const uint64_t x0 = sw128_desc(st + A_BYTES, 16u, 1024u);
#pragma unroll
                    for (int w = 0; w < KW; ++w)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            // descriptor start addresses advance in 16-byte units
                            const uint64_t bd = x0 + ((2 * w * XB + j * 32) >> 4);
                            const bool acc = kb > kb0 || w > 0 || j > 0;
#pragma unroll
                            for (int m = 0; m < NACC; ++m) {
                                const uint64_t ad = DOWN ? a0 + ((m * BLK + j * 2048) >> 4)
                                                         : a0 + (((m * KW + w) * BLK + j * 32) >> 4);
                                umma_f16(d0 + m * ACOLS, ad, bd, IDESC, acc);
                            }
                        }
                    umma_commit(&empty[slot]);
                }
                if (s_abort) break;
                umma_commit(&accf[ab]);
                it += kb1 - kb0;
            }
            umma_commit(&fin);
            if (!mbar_wait(&fin, 0)) set_status(a.status, ST_TIMEOUT);
        }
    } else {
        // ================================================================ drain (warps 0-3)
        const int m = 32 * warp + lane;
        const int nwords = (a.f + 31) / 32;
        uint32_t si = 0;
        for (long long it = it0; it < it1; ++si) {
            const int t = (int)(it / KB), kb0 = (int)(it - (long long)t * KB);
            const int kb1 = (int)min((long long)KB, kb0 + (it1 - it));
            it += kb1 - kb0;
            const uint32_t ab = si % NBUF;
            // all four drain warps take the same decision, so none is left at a named barrier
            if (!mbar_wait(&accf[ab], (si / NBUF) & 1)) s_dabort = 1;
            named_sync(1, 128);
            if (s_dabort) {
                if (threadIdx.x == 0) set_status(a.status, ST_TIMEOUT);
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * warp) << 16) + ab * ACC;
            // 16 columns of accumulator mm: hi-part products plus lo-part products
            auto acc16 = [&](int mm, int c, float (&v)[16]) {
                float lo[16];
                tmem_ld16(tb + mm * ACOLS + c, v);
                tmem_ld16(tb + mm * ACOLS + NB + c, lo);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += lo[i];
            };
            const bool whole = kb0 == 0 && kb1 == KB;
            if (!whole) {
                const int slot = it0 >= (long long)t * KB ? 0 : 1;
                float *mypart = a.part + (size_t)(cta * 2 + slot) * PCOLS * 128;
#pragma unroll 1
                for (int mm = 0; mm < NACC; ++mm)
#pragma unroll 1
                    for (int c = 0; c < NB; c += 16) {
                        float v[16];
                        acc16(mm, c, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) mypart[(mm * NB + c + i) * 128 + m] = v[i];
                    }
            }
            // the tile's final values, 16 batch columns at a time, from TMEM or from the partials
            auto chunk = [&](int c, float (&v)[NACC][16]) {
                if (whole) {
#pragma unroll
                    for (int mm = 0; mm < NACC; ++mm) acc16(mm, c, v[mm]);
                    return;
                }
#pragma unroll
                for (int mm = 0; mm < NACC; ++mm)
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[mm][i] = 0.f;
                const long long tb0 = (long long)t * KB;
                const int c0 = tc_owner(tb0, T, P), c1 = tc_owner(tb0 + KB - 1, T, P);
                // contributors in CTA order; each group's loads are issued together
                constexpr int G = NACC == 1 ? 2 : 1;
                for (int cg = c0; cg <= c1; cg += G) {
                    float u[G][NACC][16];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int cc = cg + g;
                        const long long b0 = cc <= c1 ? tc_begin(cc, T, P) : 0;
                        const bool use = cc <= c1 && tc_begin(cc + 1, T, P) != b0;   // skip empty ranges
                        const float *pp = a.part + (size_t)(cc * 2 + (b0 >= tb0 ? 0 : 1)) * PCOLS * 128;
#pragma unroll
                        for (int mm = 0; mm < NACC; ++mm)
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                u[g][mm][i] = use ? __ldcg(pp + (mm * NB + c + i) * 128 + m) : 0.f;
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int mm = 0; mm < NACC; ++mm)
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[mm][i] += u[g][mm][i];
                }
            };
            bool last = whole;
            if (!whole) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acce[ab]);
                named_sync(1, 128);
                if (threadIdx.x == 0) {
                    const int add = kb1 - kb0;
                    s_last = (int)atom_add_acq_rel(a.tile_cnt + t, (uint32_t)add) + add == KB;
                }
                named_sync(1, 128);
                last = s_last != 0;
            }
            if (last) {
                int id = -1;
                if constexpr (!DOWN) {
                    const int j = t * 128 + m;
                    if (j < n) {
                        id = a.idx ? __ldcg(a.idx + j) : a.row0 + j;
                        if (id < 0 || id >= a.f) id = -1;
                    }
                }
                const float bias = (id >= 0 && a.bias) ? __ldg(a.bias + id) : 0.f;
                bool act = false;
#pragma unroll 1
                for (int c = 0; c < NB; c += 16) {
                    float v[NACC][16];
                    chunk(c, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int b = c + i;
                        if constexpr (DOWN) {
                            if (b < a.B) {
#pragma unroll
                                for (int mm = 0; mm < NACC; ++mm) {
                                    const size_t o = (size_t)b * a.d + (size_t)t * 128 * W + mm * 128 + m;
                                    a.out[o] = (a.xin ? __ldcg(a.xin + o) : 0.f) + v[mm][i];
                                }
                            }
                        } else if constexpr (MODE == TC_LOGITS) {
                            act |= id >= 0 && b < a.B && (id < a.hot || v[0][i] + bias > a.tau);
                        } else {
                            const int j = t * 128 + m;
                            float hv = 0.f;
                            if (b < a.B && id >= 0) {
                                if constexpr (MODE == TC_PRED_HIDDEN) hv = fmaxf(v[0][i], 0.f);
                                else if constexpr (MODE == TC_RELU) hv = fmaxf(v[0][i] + bias, 0.f);
                                else hv = fmaxf(v[0][i] + bias, 0.f) * v[NMAT - 1][i];
                            }
                            if (j < a.ldo) {
                                uint16_t hi, lo;
                                split16<WT>(hv, hi, lo);
                                a.ohi[(size_t)b * a.ldo + j] = hi;
                                a.olo[(size_t)b * a.ldo + j] = lo;
                            }
                        }
                    }
                }
                if (whole) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acce[ab]);
                } else if (threadIdx.x == 0) {
                    a.tile_cnt[t] = 0u;
                }
                if constexpr (MODE == TC_LOGITS) {
                    const uint32_t word = __ballot_sync(0xffffffffu, act);
                    const int wi = (a.row0 + t * 128 + 32 * warp) >> 5;
                    if (lane == 0 && wi < nwords) a.maskw[wi] = word;
                    named_sync(1, 128);   // the four warps' mask words before the releasing ticket
                    if (threadIdx.x == 0 && atom_add_acq_rel(a.done_cnt, 1u) == (unsigned)tiles - 1) s_compact = 1;
                }
            }
        }
    }

    // ---- the CTA that completed the last logits tile lists the active rows, with every warp
    if constexpr (MODE == TC_LOGITS) {
        __syncthreads();
        if (s_compact) {
            compact_words<TC_THREADS / 32>(a.maskw, (a.f + 31) / 32, a.row0 / 32, a.idx_out, a.count_out, s_wsum,
                                           [] { __syncthreads(); });
            if (threadIdx.x == 0) *a.done_cnt = 0u;
        }
    }

    // ---- teardown: all copies and products of this CTA are complete
    tc_fence_before();
    __syncthreads();
    if (warp == TC_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
    }
}

// x [B x d] fp32 -> hi, lo [NB x ld] in the weights' 16-bit type; rows B..NB-1 zero.
// rms: scale row b by 1/sqrt(mean(x_b^2) + eps) first (the stack's pre-norm).
template <int WT>
__global__ void __launch_bounds__(256) k_tc_split(const float *__restrict__ x, int d, int B, int ld, int rms, float eps,
                                                  uint16_t *__restrict__ hi, uint16_t *__restrict__ lo)
{
    __shared__ float ws[8];
    const int b = blockIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    uint2 *h2 = reinterpret_cast<uint2 *>(hi + (size_t)b * ld), *l2 = reinterpret_cast<uint2 *>(lo + (size_t)b * ld);
    if (b >= B) {
        for (int i = threadIdx.x; i < d / 4; i += blockDim.x) h2[i] = l2[i] = make_uint2(0u, 0u);
        return;
    }
    const float4 *x4 = reinterpret_cast<const float4 *>(x + (size_t)b * d);
    float inv = 1.f;
    if (rms) {
        float t = 0.f;
        for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
            const float4 v = __ldcg(x4 + i);
            t = fmaf(v.x, v.x, t);
            t = fmaf(v.y, v.y, t);
            t = fmaf(v.z, v.z, t);
            t = fmaf(v.w, v.w, t);
        }
        t = warp_sum(t);
        if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = t;
        __syncthreads();
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += ws[w];
        inv = 1.0f / sqrtf(s / (float)d + eps);
    }
    for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
        const float4 v = __ldcg(x4 + i);
        const float e[4] = {v.x * inv, v.y * inv, v.z * inv, v.w * inv};
        uint16_t hh[4], ll[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) split16<WT>(e[k], hh[k], ll[k]);
        h2[i] = make_uint2(hh[0] | ((uint32_t)hh[1] << 16), hh[2] | ((uint32_t)hh[3] << 16));
        l2[i] = make_uint2(ll[0] | ((uint32_t)ll[1] << 16), ll[2] | ((uint32_t)ll[3] << 16));
    }
}

template <int WT, int MODE>
cudaError_t launch_tc_mode(int nb, int w, const TcArgs &a, int grid, size_t smem, cudaStream_t s, bool pdl)
{
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = ensure_smem(kern, smem);
        if (e != cudaSuccess) return e;
        Launch L;
        L.grid = dim3(grid);
        L.block = dim3(TC_THREADS);
        L.smem = smem;
        L.stream = s;
        L.pdl = pdl;
        L.nsm = grid;
        return launch_ex(L, kern, a);
    };
    auto by_w = [&](auto nbc) -> cudaError_t {
        constexpr int NB = decltype(nbc)::value;
        if (w == 1) return go(k_tc<WT, MODE, NB, 1>);
        if (w == 2) return go(k_tc<WT, MODE, NB, 2>);
        return cudaErrorInvalidValue;
    };
    switch (nb) {
    case 16: return by_w(std::integral_constant<int, 16>());
    case 32: return by_w(std::integral_constant<int, 32>());
    case 64: return by_w(std::integral_constant<int, 64>());
    case 128: return by_w(std::integral_constant<int, 128>());
    }
    return cudaErrorInvalidValue;
}

template <int WT>
cudaError_t launch_tc_split_wt(const float *x, int d, int B, int nb, int ld, int rms, float eps, uint16_t *hi,
                               uint16_t *lo, cudaStream_t s, bool pdl)
{
    Launch L;
    L.grid = dim3(nb);
    L.block = dim3(256);
    L.smem = 0;
    L.stream = s;
    L.pdl = pdl;
    L.nsm = nb;
    return launch_ex(L, k_tc_split<WT>, x, d, B, ld, rms, eps, hi, lo);
}

}  // namespace pi
