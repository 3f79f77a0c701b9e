// sv_kernel.cuh -- persistent verification kernel for sm_103a.
//
// One launch runs one verification round for B sequences (the rule of the
// nextadmin.net lesson "Speculative Decoding", § Core algorithm steps 4-6, and
// of aiengineeringfromscratch.com lesson 25, § The exact rule / § Greedy case;
// q = target, p = draft).
//
// Work is split into tasks, scheduled left to right by position:
//   stats task    one chunk of one row at position i: the online maximum and
//                 sum of 2^((x - m) * log2(e) / T) (greedy: maximum and its
//                 lowest index).  All position-0 tasks of every sequence come
//                 first, then position 1, ...; a task whose sequence already
//                 stopped before position i is skipped without reading its
//                 rows (the rule discards everything after the first rejection).
//   decision      the worker that finishes the last chunk of (sequence,
//                 position) merges the chunk partials in float64, draws u_i
//                 (Philox) and decides accept_i = u_i < min(1, q_i(d_i)/p_i(d_i)).
//                 Decisions are published in a per-sequence bit word; the first
//                 non-accepted decided position j, with all earlier ones
//                 accepted, ends the sequence.
//   residual task one chunk of rows j (target and draft) of an ended
//                 sequence: r(x) = max(0, q_j(x) - p_j(x)) (r = q_{K+1} for a
//                 bonus), summed per 256-token segment.  The worker finishing the
//                 last one locates the token by inverse CDF: a float64 scan over
//                 segment masses, then a scan inside one segment.  No
//                 probability is stored.
//
// Every warp is an independent worker: it pops tasks from global counters,
// streams its tasks' rows through its own ring of shared-memory stages with
// cp.async.bulk (completion on one mbarrier per stage), reduces them, and
// publishes, decides or locates itself.  Warps share nothing but the CTA's
// shared-memory carve-up, so a slow warp never holds the others back; sixteen
// workers per SM hide each other's memory and synchronisation latency.
// Every wait is bounded by Params::spin_limit; a wait that runs out sets
// SPEC_ERR_TIMEOUT and the worker winds down after draining its own copies.
// The last CTA to finish resets the workspace control words for the next call.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "sv_params.h"

namespace sv {

constexpr int NWARP = 16;                    // workers per CTA
constexpr int NTHREADS = NWARP * 32;
constexpr int RS = 3;                        // ring stages per worker
constexpr int SB = 4096;                     // bytes per stage
constexpr int SEG = 256;                     // tokens per segment
constexpr uint32_t DRAIN_LIMIT = 1u << 24;   // polls while waiting for our own bulk copies
// Floor of the bound on waits for a CTA's own barriers (its copies, its
// hand-offs between warps): the spin limit lowers only the waits on other
// CTAs, so a small limit exercises those and never leaves copies in flight.
constexpr uint32_t OWN_WAIT_MIN = 1u << 20;
#define F_INF __int_as_float(0x7f800000)

enum Kind { K_NONE = 0, K_STAT_T = 1, K_STAT_D = 2, K_RES = 3 };

// What one ring stage holds.
struct Meta {
    int kind, b, pos;
    int kf;           // stats: first unit of the run this stage belongs to; residual: task index
    int ku;           // stats: this stage's unit
    int e0, n, last, direct;
    const void *g0;   // row element e0 (target row, or draft row for K_STAT_D)
    const void *g1;   // residual: draft row element e0
    float4 rc;        // residual: Mt, Lt2, dLhi, dLlo of the sequence's last position
};


// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}
// Programmatic dependent launch: a kernel launched with it may start while
// the one before it in the stream is finishing; pdl_wait() blocks until that
// kernel has completed and its writes are visible (a no-op otherwise), and
// pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of parity `parity`.  Returns false when `limit`
// polls ran out or (if `abort` is given) the CTA is winding down.
__device__ __forceinline__ bool mbar_wait(unsigned long long *bar, uint32_t parity, uint32_t limit,
                                          const volatile int *abort)
{
    for (uint32_t it = 0;; ++it) {
        if (mbar_test(bar, parity))
            return true;
        if (it >= limit || (abort && *abort))
            return false;
        if (it > 16)
            __nanosleep(128);
    }
}
// Warp-uniform bounded wait: lane 0 polls, then every lane observes the
// completed phase itself (one test, which cannot fail once lane 0 has seen
// it, since the phase cannot move on before this warp arrives elsewhere).
__device__ __forceinline__ bool warp_wait(unsigned long long *bar, uint32_t parity, uint32_t limit,
                                          const volatile int *abort, int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = mbar_wait(bar, parity, limit, abort);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok)
        (void)mbar_test(bar, parity);
    __syncwarp();
    return ok;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         unsigned long long *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}
__device__ __forceinline__ float ex2a(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
// Two floats in one 64-bit register, for the packed f32x2 instructions.
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ f2 pku(uint32_t lo, uint32_t hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void upk(f2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2 ex2x2(f2 v)
{
    float a, b;
    upk(v, a, b);
    return pk(ex2a(a), ex2a(b));
}
// Elementwise NaN-propagating max of two bfloat16 pairs.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <class T> __device__ __forceinline__ T ld_vol(const T *p) { return *(const volatile T *)p; }
__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
template <class T> __device__ __forceinline__ void st_vol(T *p, T v) { *(volatile T *)p = v; }

// ------------------------------------------------------------------ warp helpers
__device__ __forceinline__ float warp_max_nan(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_sumf(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_maxi(int v)
{
    return __reduce_max_sync(0xffffffffu, v);
}
__device__ __forceinline__ int warp_or(int v)
{
    return __reduce_or_sync(0xffffffffu, v);
}
__device__ __forceinline__ double warp_incl_scan(double v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += t;
    }
    return v;
}
// (value, index) argmax merge: larger value wins, lower index on ties.
__device__ __forceinline__ void argmax_merge(float &v, int &i, float v2, int i2)
{
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

// ------------------------------------------------------------------ numerics
// A float pair (hi + lo) carries partial sums across threads, warps and chunks
// without the float64 pipe (which GB300 runs at a small fraction of float32).
struct DF {
    float hi, lo;
};
__device__ __forceinline__ DF two_sum(float a, float b)
{
    const float s = a + b, bb = s - a;
    return DF{s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ DF df_add(DF a, DF b)
{
    const DF s = two_sum(a.hi, b.hi);
    const float lo = s.lo + (a.lo + b.lo);
    const float hi = s.hi + lo;
    return DF{hi, lo - (hi - s.hi)};
}
// x * 2^d for d <= 0: the integer part of d scales the exponent exactly, the
// fraction goes through one ex2.approx; the product is kept exact as a pair.
__device__ __forceinline__ DF df_scale_pow2(DF x, float d)
{
    if (!(d > -120.0f))
        return DF{0.0f, 0.0f};
    const float n = floorf(d);
    const float f = ex2a(d - n);                                   // [1, 2)
    const float e2 = __int_as_float(((int)n + 127) << 23);         // exact 2^n
    const float p = x.hi * f;
    const float perr = fmaf(x.hi, f, -p);
    return df_add(DF{p * e2, 0.0f}, DF{perr * e2, x.lo * f * e2});
}
__device__ __forceinline__ DF warp_sum_df(DF v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = df_add(v, DF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)});
    return v;
}

// 1 - 2^delta for delta < 0.  Near 0 it is -expm1(delta ln 2) from its Taylor
// series (ten terms; truncation below 1e-9 relative on [-ln 2, 0]), which
// avoids the cancellation of 1 - ex2(delta).
__device__ __forceinline__ float one_minus_pow2(float delta)
{
    if (delta <= -1.0f)
        return 1.0f - ex2a(delta);
    const float t = delta * 0.69314718055994531f;
    float e = 1.0f / 3628800.0f;
    e = fmaf(e, t, 1.0f / 362880.0f);
    e = fmaf(e, t, 1.0f / 40320.0f);
    e = fmaf(e, t, 1.0f / 5040.0f);
    e = fmaf(e, t, 1.0f / 720.0f);
    e = fmaf(e, t, 1.0f / 120.0f);
    e = fmaf(e, t, 1.0f / 24.0f);
    e = fmaf(e, t, 1.0f / 6.0f);
    e = fmaf(e, t, 0.5f);
    e = fmaf(e, t, 1.0f);
    return -(t * e);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): round constants and key
// increments from the paper's definition.
__device__ __forceinline__ uint4 philox10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                          uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}
__device__ __forceinline__ double uniform24(uint32_t w)
{
    return ((double)(w >> 8) + 0.5) * (1.0 / 16777216.0);
}
// The same uniform (2n + 1) 2^-25, n = w >> 8, in float32 arithmetic.  It has
// 25 significant bits, one more than a float holds, so it is never rounded to
// a float; instead:
//  - u24_below(w, a): whether it is below a in [0, 1], decided exactly:
//    2n + 1 < a 2^25 holds for the integer 2n + 1 iff it is below ceil(a 2^25)
//    (a 2^25 is an exact scaling, and its ceiling an exact conversion);
//  - u24_scale(w, F): its product with the float pair F, as a float pair, from
//    the exact parts n 2^-24 and 2^-25 (the rounding of the pair alone).
__device__ __forceinline__ bool u24_below(uint32_t w, float a)
{
    return (w >> 8) * 2u + 1u < __float2uint_ru(a * 33554432.0f);
}
__device__ __forceinline__ DF u24_scale(uint32_t w, DF F)
{
    const float vh = (float)(w >> 8) * (1.0f / 16777216.0f);
    const float th = vh * F.hi;
    return df_add(DF{th, fmaf(vh, F.hi, -th)}, DF{fmaf(vh, F.lo, F.hi * (1.0f / 33554432.0f)), 0.0f});
}

// ------------------------------------------------------------------ element types
struct F32 {
    static constexpr int ES = 4;
    static constexpr int VE = 4;
    __device__ static __forceinline__ void unpack(const uint4 &v, float *o)
    {
        o[0] = __uint_as_float(v.x);
        o[1] = __uint_as_float(v.y);
        o[2] = __uint_as_float(v.z);
        o[3] = __uint_as_float(v.w);
    }
    __device__ static __forceinline__ float load(const void *base, size_t i)
    {
        return __ldg(static_cast<const float *>(base) + i);
    }
    __device__ static __forceinline__ float load_cg(const void *base, size_t i)
    {
        return __ldcg(static_cast<const float *>(base) + i);
    }
    __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
    // element pairs (2i, 2i+1) of one 16-byte vector
    __device__ static __forceinline__ f2 pair(const uint4 &v, int i)
    {
        return i == 0 ? pku(v.x, v.y) : pku(v.z, v.w);
    }
    // NaN-propagating max of the elements of four vectors
    __device__ static __forceinline__ float quad_max(const uint4 *v)
    {
        float m[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m[2 * k] = fmax_nan(__uint_as_float(v[k].x), __uint_as_float(v[k].y));
            m[2 * k + 1] = fmax_nan(__uint_as_float(v[k].z), __uint_as_float(v[k].w));
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i)
                m[i] = fmax_nan(m[i], m[i + w]);
        return m[0];
    }
    __device__ static __forceinline__ float vec_max(const uint4 &v)
    {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
};
struct BF16 {
    static constexpr int ES = 2;
    static constexpr int VE = 8;
    __device__ static __forceinline__ void unpack(const uint4 &v, float *o)
    {
        o[0] = __uint_as_float(v.x << 16);
        o[1] = __uint_as_float(v.x & 0xffff0000u);
        o[2] = __uint_as_float(v.y << 16);
        o[3] = __uint_as_float(v.y & 0xffff0000u);
        o[4] = __uint_as_float(v.z << 16);
        o[5] = __uint_as_float(v.z & 0xffff0000u);
        o[6] = __uint_as_float(v.w << 16);
        o[7] = __uint_as_float(v.w & 0xffff0000u);
    }
    __device__ static __forceinline__ float load(const void *base, size_t i)
    {
        const unsigned short h = __ldg(static_cast<const unsigned short *>(base) + i);
        return __uint_as_float((uint32_t)h << 16);
    }
    __device__ static __forceinline__ float load_cg(const void *base, size_t i)
    {
        const unsigned short h = __ldcg(static_cast<const unsigned short *>(base) + i);
        return __uint_as_float((uint32_t)h << 16);
    }
    __device__ static __forceinline__ uint4 neg_inf() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }
    __device__ static __forceinline__ f2 pair(const uint4 &v, int i)
    {
        const uint32_t w = i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
        return pku(w << 16, w & 0xffff0000u);
    }
    __device__ static __forceinline__ float word_max(uint32_t w)
    {
        return fmax_nan(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static __forceinline__ float quad_max(const uint4 *v)
    {
        uint32_t m[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m[2 * k] = bmax2(v[k].x, v[k].y);
            m[2 * k + 1] = bmax2(v[k].z, v[k].w);
        }
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i)
                m[i] = bmax2(m[i], m[i + w]);
        return word_max(m[0]);
    }
    __device__ static __forceinline__ float vec_max(const uint4 &v)
    {
        return word_max(bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)));
    }
};

// ------------------------------------------------------------------ small shared steps
__device__ __forceinline__ void set_status(const Params &P, int code)
{
    atomicCAS(&P.ctl[CTL_STATUS], 0u, (uint32_t)code);
}
__device__ __forceinline__ void write_error(const Params &P, int b, int code)
{
    for (int i = 0; i <= P.K; ++i)
        P.out_tokens[(size_t)b * (P.K + 1) + i] = -1;
    P.out_len[b] = -code;
    if (P.aux_R)
        P.aux_R[b] = __int_as_float(0x7fc00000);
    set_status(P, code);
}
// First position j not accepted; the sequence has ended once j is decided.
__device__ __forceinline__ bool resolved(unsigned long long st, int &j)
{
    const uint32_t D = (uint32_t)st, A = (uint32_t)(st >> 32);
    j = __ffs(~A) - 1;
    return (D >> j) & 1u;
}

// =================================================================== stage math
struct Acc {
    float m;     // running max (raw logits) / greedy best value
    float s;     // running sum of 2^((x - m) c)
    int idx;     // greedy best index
    int flag;    // bit 0: NaN / +inf seen; bit 1: bad shortlist entry
};

// Four 16-byte vectors of a stats stage for this lane: vector v = lane + 32*(4h + k).
template <class E>
__device__ __forceinline__ void load_quad(const Meta &m, const uint8_t *st, int lane, int h, uint4 *v)
{
    constexpr int VE = E::VE;
    if (!m.direct) {
        const uint4 *sv = reinterpret_cast<const uint4 *>(st);
        const int nvec = m.n / VE;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = lane + 32 * (4 * h + k);
            v[k] = i < nvec ? sv[i] : E::neg_inf();
        }
    } else {
        // unaligned rows: element loads, -inf past the end (same bit layout as a vector)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (E::ES == 4) {
                    const int i = (lane + 32 * (4 * h + k)) * 4 + q;
                    w[q] = i < m.n ? __float_as_uint(E::load(m.g0, i)) : 0xff800000u;
                } else {
                    const int i = (lane + 32 * (4 * h + k)) * 8 + 2 * q;
                    const uint32_t lo = i < m.n ? (__float_as_uint(E::load(m.g0, i)) >> 16) : 0xff80u;
                    const uint32_t hi = i + 1 < m.n ? (__float_as_uint(E::load(m.g0, i + 1)) >> 16) : 0xff80u;
                    w[q] = lo | (hi << 16);
                }
            }
            v[k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Online max / sum of 2^((x - m) c) over the elements of four vectors:
// packed bf16x2 max tree, f32x2 arithmetic, tree sums.
template <class E>
__device__ __forceinline__ void online_update(const uint4 *v, float c, Acc &a)
{
    constexpr int NP = 2 * E::VE;   // element pairs in four vectors
    const float mn = fmax_nan(a.m, E::quad_max(v));
    const float ref = (mn == -F_INF) ? 0.0f : mn;
    if (mn != a.m)
        a.s *= ex2a((a.m - ref) * c);
    const f2 nref = pk(-ref, -ref), cc = pk(c, c);
    f2 e[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p)
        e[p] = ex2x2(mul2(add2(E::pair(v[p / (NP / 4)], p % (NP / 4)), nref), cc));
#pragma unroll
    for (int w = NP / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            e[i] = add2(e[i], e[i + w]);
    float lo, hi;
    upk(e[0], lo, hi);
    a.s += lo + hi;
    a.m = mn;
}

// Running (max, lowest index): a vector's elements are examined one by one
// only when its maximum beats the lane's best so far (rare after the start).
template <class E>
__device__ __forceinline__ void greedy_update(const uint4 *v, const Meta &m, int lane, int h, Acc &a)
{
    constexpr int VE = E::VE;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float vm = E::vec_max(v[k]);
        if (vm != vm) {
            a.flag |= 1;
        } else if (vm > a.m) {
            float x[VE];
            E::unpack(v[k], x);
            const int base = m.e0 + (lane + 32 * (4 * h + k)) * VE;
#pragma unroll
            for (int e = VE - 1; e >= 0; --e)
                if (x[e] == vm)
                    a.idx = base + e;
            a.m = vm;
        }
    }
}

// Shortlist: check entries [e0, e0+n) of sequence b's index row (ascending,
// unique, inside [0, V)); at position 0 also record, for each 256-token
// segment t, the first entry whose token is >= 256 t.
static __device__ void shortlist_scan(const Params &P, const Meta &m, int lane, bool record, int &flag)
{
    const int32_t *idx = P.shortlist + (size_t)m.b * P.S;
    int32_t *lb = P.sl_lb + (size_t)m.b * (P.nseg + 1);
    for (int s = m.e0 + lane; s < m.e0 + m.n; s += 32) {
        const int cur = __ldg(idx + s);
        const int prev = s > 0 ? __ldg(idx + s - 1) : -1;
        if (cur < 0 || cur >= P.V || cur <= prev) {
            flag |= 2;
            continue;
        }
        if (!record)
            continue;
        // segments t with prev < 256 t <= cur start at entry s
        const int t_lo = prev < 0 ? 0 : prev / SEG + 1;
        const int t_hi = cur / SEG;
        for (int t = t_lo; t <= t_hi; ++t)
            lb[t] = s;
        if (s == P.S - 1)
            for (int t = t_hi + 1; t <= P.nseg; ++t)
                lb[t] = P.S;
    }
}

// Residual coefficients for (b, j) and the per-element residual.
struct ResCoef {
    float Mt, Lt2, dLhi, dLlo, c;
};
__device__ __forceinline__ ResCoef load_coef(const Params &P, int b, int j)
{
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(P.dec + (size_t)b * (P.K + 1) + j));
    return ResCoef{v.x, v.y, v.z, v.w, P.c};
}
// r(x) and q(x) for 8 tokens given as 4 target pairs XT and 4 draft pairs XD
// (draft logits, or probabilities when PROBS); `bonus` samples q itself.
//   q = 2^((xt - Mt) c - log2 St)
//   delta = log2(p / q) = (xd - xt) c - dL, and r = q (1 - 2^delta) for delta < 0,
// where 1 - 2^delta comes from -expm1(delta ln 2) as a degree-8 Taylor
// polynomial on (-1, 0) (no cancellation near 0; truncation below 1.5e-7
// relative) and from 1 - ex2(delta) below -1.  Tokens with xt = -inf give 0.
template <bool PROBS>
__device__ __forceinline__ void res8(const f2 *XT, const f2 *XD, const ResCoef &k, bool bonus, f2 *R, f2 *Q)
{
    const f2 nMt = pk(-k.Mt, -k.Mt), cc = pk(k.c, k.c), nLt = pk(-k.Lt2, -k.Lt2);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const f2 q = ex2x2(fma2(add2(XT[p], nMt), cc, nLt));
        Q[p] = q;
        if (bonus) {
            R[p] = q;
        } else if (PROBS) {
            float q0, q1, p0, p1;
            upk(q, q0, q1);
            upk(XD[p], p0, p1);
            R[p] = pk(fmaxf(q0 - p0, 0.0f), fmaxf(q1 - p1, 0.0f));
        } else {
            const f2 dd = fma2(XT[p], pk(-1.0f, -1.0f), XD[p]);                             // xd - xt
            const f2 dl = add2(fma2(dd, cc, pk(-k.dLhi, -k.dLhi)), pk(-k.dLlo, -k.dLlo));   // delta
            float d0, d1;
            upk(dl, d0, d1);
            d0 = fminf(d0, 0.0f);   // also maps NaN (both logits -inf) to 0
            d1 = fminf(d1, 0.0f);
            const f2 t = mul2(pk(fmaxf(d0, -1.0f), fmaxf(d1, -1.0f)), pk(0.69314718055994531f, 0.69314718055994531f));
            f2 P = pk(-1.0f / 40320.0f, -1.0f / 40320.0f);
            P = fma2(P, t, pk(-1.0f / 5040.0f, -1.0f / 5040.0f));
            P = fma2(P, t, pk(-1.0f / 720.0f, -1.0f / 720.0f));
            P = fma2(P, t, pk(-1.0f / 120.0f, -1.0f / 120.0f));
            P = fma2(P, t, pk(-1.0f / 24.0f, -1.0f / 24.0f));
            P = fma2(P, t, pk(-1.0f / 6.0f, -1.0f / 6.0f));
            P = fma2(P, t, pk(-0.5f, -0.5f));
            P = fma2(P, t, pk(-1.0f, -1.0f));
            float o0, o1;
            upk(mul2(t, P), o0, o1);              // 1 - 2^delta on [-1, 0]
            if (d0 <= -1.0f)
                o0 = 1.0f - ex2a(d0);
            if (d1 <= -1.0f)
                o1 = 1.0f - ex2a(d1);
            R[p] = mul2(q, pk(o0, o1));
        }
    }
}

// Target pairs XT and draft pairs XD of the 8 tokens [x0 + 8 lane, +8) of a
// 256-token segment: from the stage (bulk copies) or global memory; with a
// shortlist, the segment's entries are first scattered into a per-warp buffer
// (absent tokens read as -inf logits / zero probabilities, i.e. p = 0).
// Tokens past the row end read as -inf targets (so r = q = 0).
template <class E, int MODE, bool PROBS>
__device__ __forceinline__ void seg_inputs(const Params &P, int b, int j, int x0, int cnt, int lane,
                                           const uint8_t *st_t, const void *g_t, const uint8_t *st_d,
                                           const void *g_d, bool direct, float *pscr, f2 *XT, f2 *XD, int &flag)
{
    if (!direct && cnt == 8) {
        const uint4 *sv = reinterpret_cast<const uint4 *>(st_t + (size_t)lane * 8 * E::ES);
        if (E::VE == 8) {
            const uint4 v = sv[0];
#pragma unroll
            for (int p = 0; p < 4; ++p)
                XT[p] = E::pair(v, p);
        } else {
            const uint4 v0 = sv[0], v1 = sv[1];
            XT[0] = E::pair(v0, 0);
            XT[1] = E::pair(v0, 1);
            XT[2] = E::pair(v1, 0);
            XT[3] = E::pair(v1, 1);
        }
    } else {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            x[e] = e < cnt ? E::load(g_t, (size_t)lane * 8 + e) : -F_INF;
#pragma unroll
        for (int p = 0; p < 4; ++p)
            XT[p] = pk(x[2 * p], x[2 * p + 1]);
    }
    if (j == P.K) {   // bonus: q only
#pragma unroll
        for (int p = 0; p < 4; ++p)
            XD[p] = 0ull;
        return;
    }
    float xd[8];
    if (MODE == MODE_SHORT) {
        const float absent = PROBS ? 0.0f : -F_INF;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            pscr[lane * 8 + e] = absent;
        __syncwarp();
        const int seg = x0 / SEG;
        const int32_t *lbp = P.sl_lb + (size_t)b * (P.nseg + 1);
        const int lo = __ldcg(lbp + seg), hi = __ldcg(lbp + seg + 1);
        const int32_t *idx = P.shortlist + (size_t)b * P.S;
        const size_t drow = ((size_t)b * P.K + j) * (size_t)P.S;
        for (int s = lo + lane; s < hi; s += 32) {
            const int pos = __ldg(idx + s) - x0;
            const float v = PROBS ? F32::load(P.draft, drow + s) : E::load(P.draft, drow + s);
            if (PROBS && !(v >= 0.0f && v != F_INF))
                flag |= 1;
            if (pos >= 0 && pos < SEG)
                pscr[pos] = v;
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < 8; ++e)
            xd[e] = pscr[lane * 8 + e];
        __syncwarp();
    } else {
        using D = typename std::conditional<PROBS, F32, E>::type;
        if (!direct && cnt == 8) {
            const uint4 *sv = reinterpret_cast<const uint4 *>(st_d + (size_t)lane * 8 * D::ES);
            if (D::VE == 8) {
                D::unpack(sv[0], xd);
            } else {
                D::unpack(sv[0], xd);
                D::unpack(sv[1], xd + 4);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                xd[e] = e < cnt ? D::load(g_d, (size_t)lane * 8 + e) : 0.0f;
        }
        if (PROBS)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                flag |= e < cnt && !(xd[e] >= 0.0f && xd[e] != F_INF);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
        XD[p] = pk(xd[2 * p], xd[2 * p + 1]);
}

// Sum of the 8 values of 4 pairs: (v0 + v4) + (v2 + v6) + ... as a fixed tree.
__device__ __forceinline__ float sum8(const f2 *V)
{
    const f2 s = add2(add2(V[0], V[2]), add2(V[1], V[3]));
    float lo, hi;
    upk(s, lo, hi);
    return lo + hi;
}

// =================================================================== decisions
static __device__ void emit_tokens(const Params &P, int b, int j, int last_token)
{
    int32_t *out = P.out_tokens + (size_t)b * (P.K + 1);
    for (int i = 0; i < j; ++i)
        out[i] = __ldg(P.tokens + (size_t)b * P.K + i);
    out[j] = last_token;
    for (int i = j + 1; i <= P.K; ++i)
        out[i] = -1;
    P.out_len[b] = j;
}

// Warp-cooperative lower bound of `key` in the ascending row idx[0..S).
static __device__ int warp_lower_bound(const int32_t *idx, int S, int key, int lane)
{
    int lo = 0, hi = S;
    while (hi - lo > 32) {
        const int step = (hi - lo + 31) / 32;
        const int p = lo + lane * step;
        const bool less = p < hi && __ldg(idx + p) < key;
        const int c = __popc(__ballot_sync(0xffffffffu, less));
        const int nlo = c > 0 ? lo + (c - 1) * step + 1 : lo;
        const int nhi = (c < 32 && lo + c * step < hi) ? lo + c * step : hi;
        lo = nlo;
        hi = nhi;
    }
    const int p = lo + lane;
    const bool less = p < hi && __ldg(idx + p) < key;
    return lo + __popc(__ballot_sync(0xffffffffu, less));
}

// Ended at position j: greedy writes its outputs; otherwise the sequence is
// published for its residual tasks (also when it ended with an error, so that
// the tickets of its slot are consumed).
template <int MODE>
__device__ void resolve(const Params &P, int b, int j)
{
    const int code = ld_vol(&P.errcode[(size_t)b * (P.K + 1) + j]);
    if (code) {
        write_error(P, b, code);
        st_vol(&P.terminal[b], -1);
    } else {
        st_vol(&P.terminal[b], j);
        if (MODE == MODE_GREEDY) {
            emit_tokens(P, b, j, ld_vol(&P.gtok[(size_t)b * (P.K + 1) + j]));
            if (P.aux_R)
                P.aux_R[b] = __int_as_float(0x7fc00000);
        }
    }
    if (MODE == MODE_GREEDY || code) {
        __threadfence();
        st_vol(&P.fin[b], 1);
    }
    if (MODE != MODE_GREEDY) {
        const uint32_t slot = atomicAdd(&P.ctl[CTL_RES_COUNT], 1u);
        ResRec *rec = P.res_rec + slot;
        rec->j = code ? -1 : j;
        if (!code) {
            const float4 dc = __ldcg(reinterpret_cast<const float4 *>(P.dec + (size_t)b * (P.K + 1) + j));
            *reinterpret_cast<float4 *>(rec->rc) = dc;
        }
        __threadfence();
        st_vol(&rec->b1, b + 1);
    }
}

template <class E, int MODE, bool PROBS>
__device__ void decide(const Params &P, int b, int pos, int lane)
{
    const int K = P.K;
    const size_t bp = (size_t)b * (K + 1) + pos;
    const Partial *pp = P.part + bp * P.npt;
    const int nt = P.nct;
    const int nd = (pos < K && MODE != MODE_GREEDY && !PROBS) ? P.ncd : 0;
    int code = 0;
    bool accept = false;
    const int d = pos < K ? __ldg(P.tokens + (size_t)b * K + pos) : -1;
    const bool tok_ok = pos == K || (d >= 0 && d < P.V);

    if (MODE == MODE_GREEDY) {
        float bv = -F_INF;
        int bi = 0x7fffffff, fl = 0;
        for (int k = lane; k < nt; k += 32) {
            fl |= ld_vol(&pp[k].flag);
            argmax_merge(bv, bi, ld_vol(&pp[k].m), __float_as_int(ld_vol(&pp[k].s_hi)));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
            argmax_merge(bv, bi, v2, i2);
        }
        fl = warp_or(fl);
        if (lane == 0) {
            if (!tok_ok)
                code = ST_TOKEN;
            else if (fl || !(bv > -F_INF) || bi == 0x7fffffff)
                code = ST_NONFINITE;
            P.gtok[bp] = bi;
            accept = !code && pos < K && bi == d;
        }
    } else {
        float Mt = -F_INF, Md = -F_INF;
        int ft = 0, fd = 0;
        for (int k = lane; k < nt; k += 32) {
            Mt = fmax_nan(Mt, ld_vol(&pp[k].m));
            ft |= ld_vol(&pp[k].flag);
        }
        for (int k = lane; k < nd; k += 32) {
            Md = fmax_nan(Md, ld_vol(&pp[nt + k].m));
            fd |= ld_vol(&pp[nt + k].flag);
        }
        Mt = warp_max_nan(Mt);
        Md = warp_max_nan(Md);
        ft = warp_or(ft);
        fd = warp_or(fd);
        double St = 0.0, Sd = 0.0;
        for (int k = lane; k < nt; k += 32) {
            const float mk = ld_vol(&pp[k].m);
            if (mk > -F_INF)
                St += ((double)ld_vol(&pp[k].s_hi) + (double)ld_vol(&pp[k].s_lo)) *
                      exp2(((double)mk - (double)Mt) * P.cd);
        }
        for (int k = lane; k < nd; k += 32) {
            const float mk = ld_vol(&pp[nt + k].m);
            if (mk > -F_INF)
                Sd += ((double)ld_vol(&pp[nt + k].s_hi) + (double)ld_vol(&pp[nt + k].s_lo)) *
                      exp2(((double)mk - (double)Md) * P.cd);
        }
        St = warp_sum(St);
        Sd = warp_sum(Sd);
        const bool sl_bad = MODE == MODE_SHORT && (fd & 2);
        const bool t_ok = !(ft & 1) && Mt > -F_INF && St > 0.0;
        const bool d_ok = PROBS || (!(fd & 1) && Md > -F_INF && Sd > 0.0);
        // the drafted token's shortlist entry (warp-cooperative search)
        int s_at = -1;
        if (MODE == MODE_SHORT && pos < K && tok_ok && !sl_bad) {
            const int32_t *idx = P.shortlist + (size_t)b * P.S;
            const int lb = warp_lower_bound(idx, P.S, d, lane);
            if (lb < P.S && __ldg(idx + lb) == d)
                s_at = lb;
        }
        if (lane == 0) {
            const double lSt = log2(St), lSd = log2(Sd);
            if (MODE == MODE_SHORT && pos == 0 && sl_bad)
                code = ST_SHORTLIST;
            else if (!tok_ok)
                code = ST_TOKEN;
            else if (!t_ok)
                code = ST_NONFINITE;
            else if (pos < K && !d_ok)
                code = ST_NONFINITE;
            double qd = __longlong_as_double(0x7ff8000000000000ll), pd = qd;
            bool qp_ok = false;
            if (pos < K && tok_ok && t_ok && d_ok && !sl_bad) {
                const float zt = E::load(P.target, bp * (size_t)P.V + d);
                qd = exp2(((double)zt - (double)Mt) * P.cd - lSt);
                const size_t drow = ((size_t)b * K + pos) * (size_t)P.Vd;
                bool p_ok = true;
                if (MODE == MODE_STOCH) {
                    if (PROBS) {
                        const float pv = F32::load(P.draft, drow + d);
                        p_ok = pv >= 0.0f && pv != F_INF;
                        pd = pv;
                    } else {
                        const float zd = E::load(P.draft, drow + d);
                        pd = exp2(((double)zd - (double)Md) * P.cd - lSd);
                    }
                } else {
                    if (s_at < 0) {
                        pd = 0.0;
                    } else if (PROBS) {
                        const float pv = F32::load(P.draft, drow + s_at);
                        p_ok = pv >= 0.0f && pv != F_INF;
                        pd = pv;
                    } else {
                        const float zd = E::load(P.draft, drow + s_at);
                        pd = exp2(((double)zd - (double)Md) * P.cd - lSd);
                    }
                }
                if (!p_ok && !code)
                    code = ST_NONFINITE;
                qp_ok = p_ok;
                if (!code) {
                    const uint4 w = philox10((uint32_t)pos, (uint32_t)b, 0u, 0u, P.key0, P.key1);
                    const double u = uniform24(w.x);
                    accept = pd > 0.0 ? (u < fmin(1.0, qd / pd)) : true;
                }
            }
            Dec dc;
            dc.Mt = Mt;
            dc.Lt2 = (float)lSt;
            const double dL = (PROBS || pos == K) ? 0.0 : ((double)Md - (double)Mt) * P.cd + lSd - lSt;
            dc.dLhi = (float)dL;
            dc.dLlo = (float)(dL - (double)dc.dLhi);
            P.dec[bp] = dc;
            if (P.full) {
                const float nanf_ = __int_as_float(0x7fc00000);
                if (P.aux_lse) {
                    P.aux_lse[(size_t)b * (2 * K + 1) + pos] = t_ok ? (float)((double)Mt * P.invT + log(St)) : nanf_;
                    if (pos < K)
                        P.aux_lse[(size_t)b * (2 * K + 1) + K + 1 + pos] =
                            (!PROBS && d_ok && !sl_bad) ? (float)((double)Md * P.invT + log(Sd)) : nanf_;
                }
                if (pos < K) {
                    if (P.aux_q)
                        P.aux_q[(size_t)b * K + pos] = qp_ok ? (float)qd : nanf_;
                    if (P.aux_p)
                        P.aux_p[(size_t)b * K + pos] = qp_ok ? (float)pd : nanf_;
                }
            }
        }
    }
    // publish the decision
    int j = -1;
    if (lane == 0) {
        P.errcode[bp] = code;
        __threadfence();
        const unsigned long long bits = (1ull << pos) | (accept ? (1ull << (32 + pos)) : 0ull);
        const unsigned long long old = atomicOr(&P.state[b], bits);
        int j_old, j_new;
        const bool was = resolved(old, j_old);
        const bool now = resolved(old | bits, j_new);
        if (now && !was)
            j = j_new;
    }
    j = __shfl_sync(0xffffffffu, j, 0);
    if (j >= 0 && lane == 0) {
        __threadfence();
        resolve<MODE>(P, b, j);
    }
}

// Inverse-CDF sample of the ended sequence b (ended at j) from its segment
// masses: float64 scan over segments, then a scan inside one segment.
template <class E, int MODE, bool PROBS>
__device__ void locate(const Params &P, float *pscr, int b, int j, int lane)
{
    const int nseg = P.nseg;
    const SegMass *sg = P.seg + (size_t)b * nseg;
    const int per = (nseg + 31) / 32;
    const int s0 = min(nseg, lane * per), s1 = min(nseg, s0 + per);
    double lr = 0.0, lq = 0.0;
    for (int s = s0; s < s1; ++s) {
        lr += (double)ld_vol(&sg[s].r);
        lq += (double)ld_vol(&sg[s].q);
    }
    double incl = warp_incl_scan(lr, lane);
    double R = __shfl_sync(0xffffffffu, incl, 31);
    const bool use_q = !(R > 0.0);
    double lsum = lr;
    if (use_q) {
        incl = warp_incl_scan(lq, lane);
        R = __shfl_sync(0xffffffffu, incl, 31);
        lsum = lq;
    }
    const int bad = ld_vol(&P.errres[b]);
    if (bad) {
        if (lane == 0) {
            write_error(P, b, ST_NONFINITE);
            __threadfence();
            st_vol(&P.fin[b], 1);
        }
        return;
    }
    const uint4 w = philox10((uint32_t)j, (uint32_t)b, 0u, 0u, P.key0, P.key1);
    const double v = uniform24(w.y);
    const double thr = v * R;
    const unsigned ball = __ballot_sync(0xffffffffu, incl > thr);
    int seg_star = -1;
    double pre = 0.0;
    if (ball) {
        const int L = __ffs(ball) - 1;
        if (lane == L) {
            double cum = incl - lsum;
            for (int s = s0; s < s1; ++s) {
                const double mass = use_q ? (double)ld_vol(&sg[s].q) : (double)ld_vol(&sg[s].r);
                if (cum + mass > thr) {
                    seg_star = s;
                    pre = cum;
                    break;
                }
                cum += mass;
            }
            if (seg_star < 0) {   // rounding: the last segment of this lane with mass
                seg_star = s1 - 1;
                pre = cum;
            }
        }
        seg_star = __shfl_sync(0xffffffffu, seg_star, L);
        pre = __shfl_sync(0xffffffffu, pre, L);
    }
    int x = -1;
    if (seg_star >= 0) {
        // rescan the segment with the same per-token arithmetic as the residual tasks
        const int x0 = seg_star * SEG;
        const int cnt = max(0, min(8, P.V - x0 - lane * 8));
        const ResCoef kc = load_coef(P, b, j);
        const char *row_t = static_cast<const char *>(P.target) + ((size_t)b * (P.K + 1) + j) * (size_t)P.V * P.es_t;
        const bool has_d = (MODE == MODE_STOCH) && j < P.K;
        const char *row_d = has_d ? static_cast<const char *>(P.draft) + ((size_t)b * P.K + j) * (size_t)P.Vd * P.es_d
                                  : nullptr;
        f2 XT[4], XD[4], R[4], Q[4];
        int flag = 0;
        seg_inputs<E, MODE, PROBS>(P, b, j, x0, cnt, lane, nullptr, row_t + (size_t)x0 * P.es_t, nullptr,
                                   has_d ? row_d + (size_t)x0 * P.es_d : nullptr, true, pscr, XT, XD, flag);
        res8<PROBS>(XT, XD, kc, j == P.K, R, Q);
        const f2 *W = use_q ? Q : R;
        float qv[8];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            upk(W[p], qv[2 * p], qv[2 * p + 1]);
        const float rsum = sum8(W);
        int lastpos = -1;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (qv[e] > 0.0f)
                lastpos = x0 + lane * 8 + e;
        lastpos = warp_maxi(lastpos);
        const double lane_excl = warp_incl_scan((double)rsum, lane) - (double)rsum;
        const double t2 = thr - pre;
        const unsigned b2 = __ballot_sync(0xffffffffu, lane_excl + (double)rsum > t2 && rsum > 0.0f);
        if (b2) {
            const int L2 = __ffs(b2) - 1;
            if (lane == L2) {
                double cum = lane_excl;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    cum += (double)qv[e];
                    if (x < 0 && qv[e] > 0.0f && cum > t2)
                        x = x0 + lane * 8 + e;
                }
                if (x < 0)
                    for (int e = 7; e >= 0; --e)
                        if (x < 0 && qv[e] > 0.0f)
                            x = x0 + lane * 8 + e;
            }
            x = __shfl_sync(0xffffffffu, x, L2);
        }
        if (x < 0)   // rounding left no crossing: the segment's last token with mass
            x = lastpos;
    }
    if (x < 0) {
        // no segment found (rounding): the largest token with positive mass
        int cand = -1;
        for (int s = s0; s < s1; ++s)
            if ((use_q ? ld_vol(&sg[s].q) : ld_vol(&sg[s].r)) > 0.0f)
                cand = s;
        cand = warp_maxi(cand);
        if (cand >= 0) {
            const int x0 = cand * SEG;
            const int cnt = max(0, min(8, P.V - x0 - lane * 8));
            const ResCoef kc = load_coef(P, b, j);
            const char *row_t = static_cast<const char *>(P.target) + ((size_t)b * (P.K + 1) + j) * (size_t)P.V * P.es_t;
            const bool has_d = (MODE == MODE_STOCH) && j < P.K;
            const char *row_d = has_d ? static_cast<const char *>(P.draft) + ((size_t)b * P.K + j) * (size_t)P.Vd * P.es_d
                                      : nullptr;
            f2 XT[4], XD[4], R[4], Q[4];
            int flag = 0;
            seg_inputs<E, MODE, PROBS>(P, b, j, x0, cnt, lane, nullptr, row_t + (size_t)x0 * P.es_t, nullptr,
                                       has_d ? row_d + (size_t)x0 * P.es_d : nullptr, true, pscr, XT, XD, flag);
            res8<PROBS>(XT, XD, kc, j == P.K, R, Q);
            float v8[8];
#pragma unroll
            for (int p = 0; p < 4; ++p)
                upk(use_q ? Q[p] : R[p], v8[2 * p], v8[2 * p + 1]);
            int lp = -1;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (v8[e] > 0.0f)
                    lp = x0 + lane * 8 + e;
            x = warp_maxi(lp);
        }
        if (x < 0)
            x = P.V - 1;
    }
    if (lane == 0) {
        emit_tokens(P, b, j, x);
        if (P.aux_R)
            P.aux_R[b] = (float)R;
        __threadfence();
        st_vol(&P.fin[b], 1);
    }
}

// =================================================================== worker
// Stats work comes in units of one stage (one 4 KB chunk of one row), ordered
// (position, sequence, chunk), target chunks before draft chunks.  A worker's
// first batch of units is fixed by its index; later batches come from a global
// counter, up to 8 units per atomic, fewer as the work runs out.  Consecutive
// units of one row in a batch form a run, reduced into one partial.

// What lane 0 streams next: one stats unit, or the stages of one residual task.
struct Cursor {
    int kind, b, pos, kf, ku, e, e_end, se, es0, es1;
    bool bulk, run_last;
    const char *row0, *row1;
    float4 rc;
};

// Lane 0's work queue.
struct Queue {
    uint32_t u, ue;                // current batch [u, ue)
    int upos, ub, uk;              // decoded form of unit u (stepped, not divided, within a batch)
    uint32_t pc, pG;               // counter value and size of the next batch (atomic in flight)
    int run_pos, run_b, run_t, run_kf;   // the current run
    bool in_run, run_dead;
    uint32_t ticket, tnext;        // residual ticket; counter value for the next one
    int pf_b1, pf_j;               // the ticket's slot record, loaded one batch boundary ahead
    float4 pf_rc;
    bool stats_left;
};

// Lane 0: load the ticket's slot record (flag first, with acquire).
__device__ __forceinline__ void prefetch_slot(const Params &P, Queue &q)
{
    if (q.ticket < P.n_res) {
        const ResRec *rec = P.res_rec + q.ticket / (uint32_t)P.ncr;
        q.pf_b1 = ld_acquire(&rec->b1);
        q.pf_j = __ldcg(&rec->j);
        q.pf_rc = __ldcg(reinterpret_cast<const float4 *>(rec->rc));
    }
}

__device__ __forceinline__ void decode_unit(const Params &P, uint32_t t, int &pos, int &b, int &k)
{
    const uint32_t per_pos = (uint32_t)P.B * (uint32_t)P.npt;
    if (t < (uint32_t)P.K * per_pos) {
        pos = (int)(t / per_pos);
        const uint32_t rr = t % per_pos;
        b = (int)(rr / (uint32_t)P.npt);
        k = (int)(rr % (uint32_t)P.npt);
    } else {
        const uint32_t rr = t - (uint32_t)P.K * per_pos;
        pos = P.K;
        b = (int)(rr / (uint32_t)P.nct);
        k = (int)(rr % (uint32_t)P.nct);
    }
}

// Units to ask for next: a third of a per-worker share of what is left, 1..32.
__device__ __forceinline__ uint32_t guided(const Params &P, uint32_t seen)
{
    const uint32_t left = P.n_stats > seen ? P.n_stats - seen : 0u;
    return max(1u, min(16u, left / (3u * P.workers)));
}

// The unit after (pos, b, k) in the static order.
__device__ __forceinline__ void step_unit(const Params &P, int &pos, int &b, int &k)
{
    if (++k == (pos < P.K ? P.npt : P.nct)) {
        k = 0;
        if (++b == P.B) {
            b = 0;
            ++pos;
        }
    }
}

// Lane 0: move to the next batch and ask the counter for the one after it.
__device__ __forceinline__ void next_batch(const Params &P, Queue &q)
{
    q.u = P.first_units + q.pc;
    q.ue = min(q.u + q.pG, P.n_stats);
    if (q.u < q.ue)
        decode_unit(P, q.u, q.upos, q.ub, q.uk);
    q.pG = guided(P, q.u);
    q.pc = atomicAdd(&P.ctl[CTL_STATS_NEXT], q.pG);
}

__device__ __forceinline__ void set_unit_cursor(const Params &P, Cursor &c, int b, int pos, int k, int kf,
                                                bool run_last)
{
    const bool is_t = k < P.nct;
    const int kk = is_t ? k : k - P.nct;
    c.kind = is_t ? K_STAT_T : K_STAT_D;
    c.b = b;
    c.pos = pos;
    c.kf = kf;
    c.ku = k;
    c.es0 = is_t ? P.es_t : P.es_d;
    c.es1 = 0;
    c.se = is_t ? P.se_t : P.se_d;
    const int n_row = is_t ? P.V : P.Vd;
    c.bulk = is_t ? P.bulk_t : P.bulk_d;
    c.row0 = is_t ? static_cast<const char *>(P.target) + ((size_t)b * (P.K + 1) + pos) * (size_t)P.V * P.es_t
                  : static_cast<const char *>(P.draft) + ((size_t)b * P.K + pos) * (size_t)P.Vd * P.es_d;
    c.row1 = nullptr;
    c.e = kk * c.se;
    c.e_end = min(n_row, c.e + c.se);
    c.run_last = run_last;
}

template <int MODE>
__device__ void set_res_cursor(const Params &P, Cursor &c, int b, int j, int k, float4 rc)
{
    const bool has_d = (MODE == MODE_STOCH) && j < P.K;
    c.kind = K_RES;
    c.b = b;
    c.pos = j;
    c.kf = k;
    c.ku = k;
    c.es0 = P.es_t;
    c.es1 = has_d ? P.es_d : 0;
    c.se = P.rse;
    c.bulk = P.bulk_t && (!has_d || P.bulk_d);
    c.row0 = static_cast<const char *>(P.target) + ((size_t)b * (P.K + 1) + j) * (size_t)P.V * P.es_t;
    c.row1 = has_d ? static_cast<const char *>(P.draft) + ((size_t)b * P.K + j) * (size_t)P.Vd * P.es_d : nullptr;
    c.rc = rc;
    c.e = k * P.rspt * P.rse;
    c.e_end = min(P.V, c.e + P.rspt * P.rse);
    c.run_last = true;
}

// Lane 0: the next unit or residual task for this worker, or false when none
// is available now.  Residual work is looked for between batches (and while
// idle), from a load issued one batch earlier.
template <int MODE>
__device__ bool pop_task(const Params &P, Queue &q, Cursor &c)
{
    for (;;) {
        if (q.u >= q.ue) {
            // 1. residual work for our ticket, once its sequence has ended (first,
            //    so that the rows it re-reads are still in L2)
            if (q.ticket < P.n_res && q.pf_b1 > 0) {
                const int b = q.pf_b1 - 1, j = q.pf_j, kres = (int)(q.ticket % (uint32_t)P.ncr);
                const float4 rc = q.pf_rc;
                q.ticket = P.workers + q.tnext;
                q.tnext = atomicAdd(&P.ctl[CTL_RES_TICKET], 1u);
                q.pf_b1 = 0;
                if (j < 0)
                    continue;   // the sequence ended with an error: nothing to sample
                set_res_cursor<MODE>(P, c, b, j, kres, rc);
                return true;
            }
            prefetch_slot(P, q);   // used at the next boundary
            // 2. the next batch of stats units
            if (!q.stats_left)
                return false;
            next_batch(P, q);
            q.in_run = false;
            if (q.u >= P.n_stats) {
                q.stats_left = false;
                return false;
            }
        }
        // the next stats unit, left to right by position
        ++q.u;
        const int pos = q.upos, b = q.ub, k = q.uk;
        step_unit(P, q.upos, q.ub, q.uk);
        const int is_t = k < P.nct;
        if (!q.in_run || pos != q.run_pos || b != q.run_b || is_t != q.run_t) {
            // a new run: skipped whole when its sequence ended before this position
            q.in_run = true;
            q.run_pos = pos;
            q.run_b = b;
            q.run_t = is_t;
            q.run_kf = k;
            q.run_dead = false;
            if (!P.full && pos > 0) {
                int j;
                q.run_dead = resolved(ld_vol(&P.state[b]), j) && j < pos;
            }
        }
        if (q.run_dead)
            continue;
        const bool run_last =
            q.u >= q.ue || !(q.upos == pos && q.ub == b && (q.uk < P.nct) == is_t);
        set_unit_cursor(P, c, b, pos, k, q.run_kf, run_last);
        return true;
    }
}

// Lane 0: issue the cursor's next stage into ring slot s.
__device__ __forceinline__ void issue_stage(const Params &P, Meta &m, unsigned long long *bar, uint8_t *ring, int s,
                                            Cursor &c, bool &tx)
{
    const int n = min(c.se, c.e_end - c.e);
    m.kind = c.kind;
    m.b = c.b;
    m.pos = c.pos;
    m.kf = c.kf;
    m.ku = c.ku;
    m.e0 = c.e;
    m.n = n;
    m.last = (c.e + c.se >= c.e_end) && c.run_last;
    m.direct = !c.bulk;
    m.g0 = c.row0 + (size_t)c.e * c.es0;
    m.g1 = c.row1 ? c.row1 + (size_t)c.e * c.es1 : nullptr;
    m.rc = c.rc;
    if (c.bulk) {
        const uint32_t b0 = (uint32_t)(n * c.es0), b1 = c.row1 ? (uint32_t)(n * c.es1) : 0u;
        uint8_t *dst = ring + (size_t)s * SB;
        // The slot's previous contents were read by this warp's lanes, whose
        // values are all consumed before the warp gets here: no reader is
        // left for the copy to overwrite.
        mbar_arrive_tx(bar, b0 + b1);
        bulk_g2s(dst, m.g0, b0, bar);
        if (b1)
            bulk_g2s(dst + P.rd_off, m.g1, b1, bar);
        tx = true;
    } else {
        mbar_arrive(bar);
        tx = false;
    }
    c.e += c.se;
    if (c.e >= c.e_end)
        c.kind = K_NONE;
}

// Residual stage: one 256-token segment at a time, the warp's lanes 8 tokens each.
template <class E, int MODE, bool PROBS>
__device__ __forceinline__ int residual_stage(const Params &P, const Meta &m, const uint8_t *st, float *pscr,
                                              int lane)
{
    int flag = 0;
    const ResCoef kc{m.rc.x, m.rc.y, m.rc.z, m.rc.w, P.c};
    for (int eb = 0; eb < m.n; eb += SEG) {
        const int x0 = m.e0 + eb;
        const int cnt = max(0, min(8, m.n - eb - lane * 8));
        const void *g_t = static_cast<const char *>(m.g0) + (size_t)eb * P.es_t;
        const void *g_d = m.g1 ? static_cast<const char *>(m.g1) + (size_t)eb * P.es_d : nullptr;
        f2 XT[4], XD[4], R[4], Q[4];
        seg_inputs<E, MODE, PROBS>(P, m.b, m.pos, x0, cnt, lane, st + (size_t)eb * P.es_t, g_t,
                                   st + P.rd_off + (size_t)eb * P.es_d, g_d, m.direct != 0, pscr, XT, XD, flag);
        res8<PROBS>(XT, XD, kc, m.pos == P.K, R, Q);
        const float rsum = warp_sumf(sum8(R));
        const float qsum = warp_sumf(sum8(Q));
        if (lane == 0)
            P.seg[(size_t)m.b * P.nseg + x0 / SEG] = SegMass{rsum, qsum};
    }
    return warp_or(flag);
}

// Finished runs and residual tasks wait in a per-warp list (entry i held by
// lane i) and are published together: their results are written, one fence,
// then their counters are bumped in parallel.  The worker whose bump completes
// a position decides it; the one completing a sequence's residual locates.
constexpr int PEND = 1;

struct Pend {
    int kind, b, pos, kf, cnt;
    Partial out;
};

// The finished run's (or residual task's) result, on every lane.
template <int MODE>
__device__ __forceinline__ Partial run_result(const Params &P, const Meta &m, const Acc &a, int rflag)
{
    Partial out{0.0f, 0, 0.0f, 0.0f};
    if (m.kind == K_RES) {
        out.flag = warp_or(rflag);
    } else if (MODE == MODE_GREEDY) {
        float v = a.m;
        int i = a.idx;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
            argmax_merge(v, i, v2, i2);
        }
        out.m = v;
        out.flag = warp_or(a.flag | (a.m == F_INF));
        out.s_hi = __int_as_float(i);
    } else {
        const float wm = warp_max_nan(a.m);
        DF contrib{0.0f, 0.0f};
        if (a.m > -F_INF && a.s > 0.0f)
            contrib = df_scale_pow2(DF{a.s, 0.0f}, (a.m - wm) * P.c);
        const DF ws = warp_sum_df(contrib);
        out.m = wm;
        out.flag = warp_or(a.flag | (a.m != a.m) | (a.m == F_INF));
        out.s_hi = ws.hi;
        out.s_lo = ws.lo;
    }
    return out;
}

template <class E, int MODE, bool PROBS>
__device__ void publish(const Params &P, const Pend *pend, int &npend, float *pscr, int lane)
{
    Pend pe{};
    if (lane < npend)
        pe = pend[lane];
    const Partial neutral{-F_INF, 0, MODE == MODE_GREEDY ? __int_as_float(0x7fffffff) : 0.0f, 0.0f};
    if (lane < npend) {
        if (pe.kind == K_RES) {
            if (pe.out.flag)
                st_vol(&P.errres[pe.b], 1);
        } else {
            P.part[((size_t)pe.b * (P.K + 1) + pe.pos) * P.npt + pe.kf] = pe.out;
        }
    }
    // neutral partials for the other units of each run
    for (int e = 0; e < npend; ++e) {
        const int kind = __shfl_sync(0xffffffffu, pe.kind, e), cnt = __shfl_sync(0xffffffffu, pe.cnt, e);
        if (kind == K_RES || cnt <= 1)
            continue;
        const int b = __shfl_sync(0xffffffffu, pe.b, e), pos = __shfl_sync(0xffffffffu, pe.pos, e);
        const int kf = __shfl_sync(0xffffffffu, pe.kf, e);
        Partial *pp = P.part + ((size_t)b * (P.K + 1) + pos) * P.npt + kf;
        for (int i = 1 + lane; i < cnt; i += 32)
            pp[i] = neutral;
    }
    __threadfence();
    bool last = false;
    if (lane < npend) {
        if (pe.kind == K_RES) {
            last = atomicAdd(&P.res_cnt[pe.b], 1u) == (uint32_t)P.ncr - 1u;
        } else {
            const size_t bp = (size_t)pe.b * (P.K + 1) + pe.pos;
            const uint32_t nparts = pe.pos < P.K ? (uint32_t)P.npt : (uint32_t)P.nct;
            last = atomicAdd(&P.pair_cnt[bp], (uint32_t)pe.cnt) + (uint32_t)pe.cnt == nparts;
        }
    }
    unsigned lastmask = __ballot_sync(0xffffffffu, last);
    if (lastmask)
        __threadfence();
    while (lastmask) {
        const int i = __ffs(lastmask) - 1;
        lastmask &= lastmask - 1;
        const int kind = __shfl_sync(0xffffffffu, pe.kind, i);
        const int b = __shfl_sync(0xffffffffu, pe.b, i);
        const int pos = __shfl_sync(0xffffffffu, pe.pos, i);
        if (kind == K_RES)
            locate<E, MODE, PROBS>(P, pscr, b, pos, lane);
        else
            decide<E, MODE, PROBS>(P, b, pos, lane);
    }
    npend = 0;
}

// Per-warp shared memory: the ring's barriers and stage descriptions, lane 0's
// queue and cursor, the pending results and the shortlist scatter buffer.
struct WorkerShared {
    unsigned long long full[RS];
    Meta meta[RS];
    Queue q;
    Cursor c;
    Pend pend[PEND];
    float pscr[SEG];
};

struct Shared {
    WorkerShared w[NWARP];
    int last_cta;
};

constexpr size_t SMEM_BYTES = (size_t)NWARP * RS * SB + sizeof(Shared);

template <class E, int MODE, bool PROBS>
__device__ void worker(const Params &P, WorkerShared &ws, uint8_t *ring, int wid, int lane)
{
    Queue &q = ws.q;
    Cursor &c = ws.c;
    uint32_t txmask = 0;   // lane 0: ring slots whose current stage is a bulk copy
    if (lane == 0) {
        c.kind = K_NONE;
        // the first residual ticket and the first batch of units follow from the
        // worker's index; the counters hand out what comes after them
        q.ticket = (uint32_t)wid;
        q.tnext = P.n_res ? atomicAdd(&P.ctl[CTL_RES_TICKET], 1u) : 0u;
        q.pf_b1 = 0;
        q.u = (uint32_t)wid * P.g0;
        q.ue = min(q.u + P.g0, P.n_stats);
        if (q.u < q.ue)
            decode_unit(P, q.u, q.upos, q.ub, q.uk);
        q.pG = guided(P, P.first_units);
        q.pc = atomicAdd(&P.ctl[CTL_STATS_NEXT], q.pG);
        q.in_run = false;
        q.stats_left = true;
    }
    uint32_t issued = 0, consumed = 0, idle = 0;
    // A residual task may come between two units of one stats run: the run's
    // accumulator and the residual task's flag are kept apart.
    Acc a{-F_INF, 0.0f, 0x7fffffff, 0};
    int rflag = 0;
    int npend = 0;
    bool ok = true;
    for (;;) {
        // top up the ring
        int finished = 0;
        if (lane == 0 && issued - consumed < (uint32_t)RS) {
            Queue ql = q;     // register copies for the top-up; the compute phase
            Cursor cl = c;    // below does not keep them live
            while (issued - consumed < (uint32_t)RS) {
                if (cl.kind == K_NONE && !pop_task<MODE>(P, ql, cl))
                    break;
                const int s = (int)(issued % RS);
                bool tx;
                issue_stage(P, ws.meta[s], &ws.full[s], ring, s, cl, tx);
                txmask = tx ? (txmask | (1u << s)) : (txmask & ~(1u << s));
                ++issued;
            }
            finished = (issued == consumed) && !ql.stats_left && ql.ticket >= P.n_res;
            q = ql;
            c = cl;
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        finished = __shfl_sync(0xffffffffu, finished, 0);
        if (issued == consumed) {
            if (npend) {   // never idle or leave with results unpublished
                publish<E, MODE, PROBS>(P, ws.pend, npend, ws.pscr, lane);
                continue;
            }
            if (finished)
                break;
            // nothing in flight: wait for our residual slot to be published
            int give_up = 0;
            if (lane == 0) {
                give_up = ++idle > P.spin_limit || ld_vol(&P.ctl[CTL_STATUS]) == (uint32_t)ST_TIMEOUT;
                if (!give_up) {
                    __nanosleep(256);
                    Queue ql = q;
                    prefetch_slot(P, ql);
                    q = ql;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) {
                ok = false;
                break;
            }
            continue;
        }
        idle = 0;
        const int s = (int)(consumed % RS);
        if (!warp_wait(&ws.full[s], (consumed / RS) & 1u, max(P.spin_limit, OWN_WAIT_MIN), nullptr, lane)) {
            ok = false;
            break;
        }
        const Meta m = ws.meta[s];
        const uint8_t *st = ring + (size_t)s * SB;
        if (m.kind == K_RES) {
            rflag |= residual_stage<E, MODE, PROBS>(P, m, st, ws.pscr, lane);
        } else if (m.kind == K_STAT_T || !PROBS) {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint4 v[4];
                load_quad<E>(m, st, lane, h, v);
                if (MODE == MODE_GREEDY)
                    greedy_update<E>(v, m, lane, h, a);
                else
                    online_update<E>(v, P.c, a);
            }
            if (MODE == MODE_SHORT && m.kind == K_STAT_D && (m.pos == 0 || P.full))
                shortlist_scan(P, m, lane, m.pos == 0, a.flag);
        }
        __syncwarp();
        ++consumed;
        if (m.last) {
            const Partial out = run_result<MODE>(P, m, a, rflag);
            if (lane == 0)
                ws.pend[npend] = Pend{m.kind, m.b, m.pos, m.kf, m.ku - m.kf + 1, out};
            __syncwarp();
            ++npend;
            if (m.kind == K_RES)
                rflag = 0;
            else
                a = Acc{-F_INF, 0.0f, 0x7fffffff, 0};
            if (npend == PEND)
                publish<E, MODE, PROBS>(P, ws.pend, npend, ws.pscr, lane);
        }
    }
    if (!ok) {
        // Winding down: report, then wait for our own copies still in flight.
        set_status(P, ST_TIMEOUT);
        if (lane == 0)
            for (uint32_t n = consumed; n < issued; ++n)
                if (txmask & (1u << (n % RS)))
                    mbar_wait(&ws.full[n % RS], (n / RS) & 1u, DRAIN_LIMIT, nullptr);
    }
    __syncwarp();
}

// =================================================================== kernel
template <class E, int MODE, bool PROBS>
__global__ void __launch_bounds__(NTHREADS, 1) verify_kernel(const __grid_constant__ Params P)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw + (size_t)NWARP * RS * SB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WorkerShared &ws = sh.w[warp];
    uint8_t *ring = smem_raw + (size_t)warp * RS * SB;
    if (lane == 0)
        for (int s = 0; s < RS; ++s)
            mbar_init(&ws.full[s], 1);
    if (threadIdx.x == 0)
        sh.last_cta = 0;
    __syncwarp();
    if (lane == 0)
        asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    worker<E, MODE, PROBS>(P, ws, ring, blockIdx.x * NWARP + warp, lane);
    __syncthreads();

    // The last CTA out finalises: sequences left unfinished by a timeout get
    // an error, the status is reported, and the control words are zeroed.
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&P.ctl[CTL_EXIT], 1u);
        sh.last_cta = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!sh.last_cta)
        return;
    __threadfence();
    for (int b = threadIdx.x; b < P.B; b += NTHREADS)
        if (ld_vol(&P.fin[b]) == 0)
            write_error(P, b, ST_TIMEOUT);
    __syncthreads();
    if (threadIdx.x == 0 && P.aux_status)
        P.aux_status[0] = (int32_t)ld_vol(&P.ctl[CTL_STATUS]);
    __syncthreads();
    // [ctl, errcode) is the region a call must find zeroed
    const uint32_t words = (uint32_t)((reinterpret_cast<const char *>(P.errcode) -
                                       reinterpret_cast<const char *>(P.ctl)) / 4);
    for (uint32_t i = threadIdx.x; i < words; i += NTHREADS)
        P.ctl[i] = 0u;
}

}  // namespace sv
