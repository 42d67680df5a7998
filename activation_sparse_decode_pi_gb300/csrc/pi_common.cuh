// pi_common.cuh -- device helpers shared by the sm_103a kernels of libpi_ffn.so.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_internal.h"

namespace pi {

// element types and FFN kinds (numbering of include/pi_ffn.h)
constexpr int DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2, DT_INT4 = 3;
constexpr int KIND_GATED = 0, KIND_RELU = 1;

// status codes written by kernels (pi_status_t values)
constexpr uint32_t ST_DEVICE_CHECK = 6;
constexpr uint32_t ST_TIMEOUT = 5;

// Elements of a given type in one 16-byte chunk.
template <int DT> struct Vec;
template <> struct Vec<DT_F32>  { static constexpr int N = 4; };
template <> struct Vec<DT_BF16> { static constexpr int N = 8; };
template <> struct Vec<DT_F16>  { static constexpr int N = 8; };
template <> struct Vec<DT_INT4> { static constexpr int N = 32; };

// 16-byte load of weights that are streamed once per decode step: read-only
// path, not kept in L1.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_scale(const __half *p)
{
    unsigned short b;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(b) : "l"(p));
    return __half2float(__ushort_as_half(b));
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait until the previous kernel's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Last-CTA ticket: one acquire-release atomic instead of fence + atomic + fence. The release
// publishes this CTA's stores (made before the caller's CTA barrier); the CTA that draws the last
// ticket acquires everyone else's (its other threads after the next CTA barrier).
__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t code)
{
    if (status) atomicCAS(status, 0u, code);
}

// Widen one 16-byte chunk of a 16/32-bit type to fp32.
template <int DT>
__device__ __forceinline__ void unpack(const uint4 &w, float (&o)[Vec<DT>::N]);

template <>
__device__ __forceinline__ void unpack<DT_F32>(const uint4 &w, float (&o)[4])
{
    o[0] = __uint_as_float(w.x);
    o[1] = __uint_as_float(w.y);
    o[2] = __uint_as_float(w.z);
    o[3] = __uint_as_float(w.w);
}

template <>
__device__ __forceinline__ void unpack<DT_BF16>(const uint4 &w, float (&o)[8])
{
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(a[i] << 16);
        o[2 * i + 1] = __uint_as_float(a[i] & 0xffff0000u);
    }
}

template <>
__device__ __forceinline__ void unpack<DT_F16>(const uint4 &w, float (&o)[8])
{
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&a[i]);
        float2 f = __half22float2(h);
        o[2 * i] = f.x;
        o[2 * i + 1] = f.y;
    }
}

// Signed 4-bit value k (0..7) of a 32-bit word: bits [4k+3 : 4k], two's complement.
__device__ __forceinline__ float nib(uint32_t w, int k)
{
    return (float)((int32_t)(w << (28 - 4 * k)) >> 28);
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c)   // (a & b) ^ c
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ __half2 u32_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }

// The eight signed 4-bit values of w (value e in bits [4e + 3 : 4e]) as exact fp32 pairs:
// p[i] = (v_i, v_{i+4}), i < 4. Each 16-bit half is built as the fp16 number 1024 + (v + 8) by
// masking a nibble into the mantissa of 1024 (flipping the nibble's top bit turns two's
// complement into offset binary); subtracting 1032 leaves v exactly. A nibble in bits 4..7 of a
// half lands as 16 (v + 8) and is scaled back by 1/16 in the same exact fused step. Integer to
// float conversions are avoided: they share the integer pipe with the shifts and masks.
__device__ __forceinline__ void i4_word_f32x2(uint32_t w, float2 (&p)[4])
{
    const uint32_t w8 = w >> 8;
    const __half2 k1032 = u32_h2(0x64086408u);   // 1032
    const __half2 k16th = u32_h2(0x2C002C00u);   // 1 / 16
    const __half2 km72 = u32_h2(0xD480D480u);    // -72 = -(1024 / 16 + 8)
    p[0] = __half22float2(__hsub2(u32_h2(lop3_and_xor(w, 0x000F000Fu, 0x64086408u)), k1032));
    p[1] = __half22float2(__hfma2(u32_h2(lop3_and_xor(w, 0x00F000F0u, 0x64806480u)), k16th, km72));
    p[2] = __half22float2(__hsub2(u32_h2(lop3_and_xor(w8, 0x000F000Fu, 0x64086408u)), k1032));
    p[3] = __half22float2(__hfma2(u32_h2(lop3_and_xor(w8, 0x00F000F0u, 0x64806480u)), k16th, km72));
}

// (a.x b.x + c.x, a.y b.y + c.y): two fp32 FMAs in one instruction, each rounded as fmaf.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

template <>
__device__ __forceinline__ void unpack<DT_INT4>(const uint4 &w, float (&o)[32])
{
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) o[8 * i + k] = nib(a[i], k);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Ascending list of the set bits of maskw[0..nwords) (bit b of word w = neuron 32 w + b;
// the first `full` words are taken as all ones without being read) into idx, and their
// number into *count, by NWARPS warps; `sync` is a barrier over exactly those warps, wsum
// NWARPS ints of shared memory. Warp g takes a contiguous block of words and reads it in
// slabs of 32 * CW words, all loads of a slab in flight at once (one round trip to L2 per
// slab); each word's set bits go to consecutive entries in one coalesced store.
template <int NWARPS, typename Sync>
__device__ __forceinline__ void compact_words(const uint32_t *__restrict__ maskw, int nwords, int full,
                                              int32_t *__restrict__ idx, int32_t *__restrict__ count, int *wsum,
                                              Sync sync)
{
    constexpr int CW = 8;   // words per lane per slab
    const int warp = (threadIdx.x >> 5) % NWARPS, lane = threadIdx.x & 31;
    const int wpw = (nwords + NWARPS - 1) / NWARPS;
    const int wb = min(nwords, warp * wpw), we = min(nwords, wb + wpw);
    auto slab = [&](int b, uint32_t (&w)[CW]) {   // lane's words b + lane + 32 k
#pragma unroll
        for (int k = 0; k < CW; ++k) {
            const int i = b + lane + 32 * k;
            w[k] = i < we ? (i < full ? 0xffffffffu : __ldcg(maskw + i)) : 0u;
        }
    };
    int cnt = 0;
    for (int b = wb; b < we; b += 32 * CW) {
        uint32_t w[CW];
        slab(b, w);
#pragma unroll
        for (int k = 0; k < CW; ++k) cnt += __popc(w[k]);
    }
    cnt = warp_sum_int(cnt);
    if (lane == 0) wsum[warp] = cnt;
    sync();
    int off = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
        off += w < warp ? wsum[w] : 0;
        total += wsum[w];
    }
    const uint32_t below = (1u << lane) - 1u;
    for (int b = wb; b < we; b += 32 * CW) {
        uint32_t w[CW];
        slab(b, w);
#pragma unroll
        for (int k = 0; k < CW; ++k) {
            const int nk = min(32, we - (b + 32 * k));
            for (int q = 0; q < nk; ++q) {
                const uint32_t m = __shfl_sync(0xffffffffu, w[k], q);
                if ((m >> lane) & 1u) idx[off + __popc(m & below)] = (b + 32 * k + q) * 32 + lane;
                off += __popc(m);
            }
        }
    }
    if (threadIdx.x % (32 * NWARPS) == 0) *count = total;
    sync();
}

}  // namespace pi
