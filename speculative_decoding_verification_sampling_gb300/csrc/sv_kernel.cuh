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
//                 lowest index).  All positions-0 tasks of every sequence come
//                 first, then position 1, ...; a task whose sequence already
//                 stopped before position i is skipped without reading its
//                 rows (the rule discards everything after the first rejection).
//   decision      the last stats task of (sequence, position) merges the
//                 chunk partials in float64, draws u_i (Philox) and decides
//                 accept_i = u_i < min(1, q_i(d_i) / p_i(d_i)).  Decisions are
//                 published in a per-sequence bit word; the first non-accepted
//                 decided position j with all earlier ones accepted ends the
//                 sequence.
//   residual task one chunk of rows j (target and draft) of an ended
//                 sequence: r(x) = max(0, q_j(x) - p_j(x)) (r = q_{K+1} for a
//                 bonus), summed per 256-token segment.  The last one locates
//                 the token by inverse CDF: a float64 scan over segment masses,
//                 then a scan inside one segment.  No probability is stored.
//
// Each CTA has three roles:
//   warp 8  (producer)  pops tasks and streams their rows into a ring of
//                       shared-memory stages with cp.async.bulk, completion on
//                       mbarriers;
//   warps 0-7 (consumers) process stages and hand per-task warp results over;
//   warp 9  (finisher)  publishes partials, decides, resolves and locates.
// Every wait is bounded by Params::spin_limit; a wait that runs out sets
// SPEC_ERR_TIMEOUT and the CTA winds down, draining its own bulk copies.
// The last CTA to finish resets the workspace control words for the next call.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "sv_params.h"

namespace sv {

constexpr int NCW = 8;                       // consumer warps
constexpr int W_PROD = NCW;                  // producer warp
constexpr int W_FIN = NCW + 1;               // finisher warp
constexpr int NTHREADS = (NCW + 2) * 32;
constexpr int STAGE_BYTES = 16384;
constexpr int NST = 6;                       // ring stages
constexpr int NH = 8;                        // hand-off slots
constexpr int RSE = 2048;                    // elements per residual stage
constexpr int RD_OFF = 8192;                 // byte offset of the draft part of a residual stage
constexpr int SEG = 256;                     // tokens per segment
constexpr uint32_t DRAIN_LIMIT = 1u << 24;   // polls while waiting for our own bulk copies
#define F_INF __int_as_float(0x7f800000)

enum Kind { K_EXIT = 0, K_STAT_T = 1, K_STAT_D = 2, K_RES = 3 };

struct Meta {
    int kind, b, pos, k, e0, n, last, direct;
    const void *g0;   // row element e0 (target row, or draft row for K_STAT_D)
    const void *g1;   // residual: draft row element e0
};

struct Hand {
    int kind, b, pos, k;
    float wm[NCW];
    int wf[NCW];
    int wi[NCW];
    float ws_hi[NCW];
    float ws_lo[NCW];
};

struct Shared {
    unsigned long long full[NST], empty[NST], hfull[NH], hempty[NH];
    Meta meta[NST];
    Hand hand[NH];
    float pscr[NCW + 1][SEG];
    volatile int abort;
    int last_cta;
};

constexpr size_t SMEM_BYTES = (size_t)NST * STAGE_BYTES + sizeof(Shared);

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}
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
};

// ------------------------------------------------------------------ small shared steps
__device__ __forceinline__ void set_status(const Params &P, int code)
{
    atomicCAS(&P.ctl[CTL_STATUS], 0u, (uint32_t)code);
}
__device__ __forceinline__ void abort_cta(const Params &P, Shared &sh)
{
    set_status(P, ST_TIMEOUT);
    sh.abort = 1;
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
__device__ __forceinline__ bool seq_dead(const Params &P, int b, int pos)
{
    int j;
    return resolved(ld_vol(&P.state[b]), j) && j < pos;
}

// =================================================================== producer
struct Ring {
    uint32_t slot = 0, ph = 0, txmask = 0, phmask = 0;
};

__device__ __forceinline__ bool ring_acquire(const Params &P, Shared &sh, Ring &r)
{
    return mbar_wait(&sh.empty[r.slot], r.ph ^ 1u, P.spin_limit, &sh.abort);
}
__device__ __forceinline__ void ring_advance(Ring &r)
{
    if (++r.slot == NST) {
        r.slot = 0;
        r.ph ^= 1u;
    }
}
// Publish the stage in r.slot: bulk copies of `bytes0` from g0 (and `bytes1`
// from g1 at RD_OFF), or a plain arrival when the consumers read global memory.
__device__ __forceinline__ void ring_publish(Shared &sh, uint8_t *ring, Ring &r, bool bulk,
                                             const void *g0, uint32_t bytes0, const void *g1,
                                             uint32_t bytes1)
{
    unsigned long long *bar = &sh.full[r.slot];
    if (bulk) {
        mbar_arrive_tx(bar, bytes0 + bytes1);
        uint8_t *dst = ring + (size_t)r.slot * STAGE_BYTES;
        bulk_g2s(dst, g0, bytes0, bar);
        if (bytes1)
            bulk_g2s(dst + RD_OFF, g1, bytes1, bar);
        r.txmask |= 1u << r.slot;
        r.phmask = (r.phmask & ~(1u << r.slot)) | (r.ph << r.slot);
    } else {
        mbar_arrive(bar);
    }
}

template <class E, int MODE, bool PROBS>
__device__ bool issue_stats(const Params &P, Shared &sh, uint8_t *ring, Ring &r, int b, int pos, int k)
{
    const bool is_t = k < P.nct;
    const int kk = is_t ? k : k - P.nct;
    const int es = is_t ? P.es_t : P.es_d, se = is_t ? P.se_t : P.se_d;
    const int spt = is_t ? P.spt_t : P.spt_d, n_row = is_t ? P.V : P.Vd;
    const bool bulk = is_t ? P.bulk_t : P.bulk_d;
    const char *row = is_t ? static_cast<const char *>(P.target) +
                                 ((size_t)b * (P.K + 1) + pos) * (size_t)P.V * es
                           : static_cast<const char *>(P.draft) +
                                 ((size_t)b * P.K + pos) * (size_t)P.Vd * es;
    const int e_begin = kk * spt * se;
    const int e_end = min(n_row, e_begin + spt * se);
    for (int e0 = e_begin; e0 < e_end; e0 += se) {
        const int n = min(se, e_end - e0);
        if (!ring_acquire(P, sh, r))
            return false;
        Meta &m = sh.meta[r.slot];
        m.kind = is_t ? K_STAT_T : K_STAT_D;
        m.b = b;
        m.pos = pos;
        m.k = k;
        m.e0 = e0;
        m.n = n;
        m.last = (e0 + se >= e_end);
        m.direct = !bulk;
        m.g0 = row + (size_t)e0 * es;
        m.g1 = nullptr;
        ring_publish(sh, ring, r, bulk, m.g0, (uint32_t)(n * es), nullptr, 0);
        ring_advance(r);
    }
    return true;
}

template <class E, int MODE, bool PROBS>
__device__ bool issue_residual(const Params &P, Shared &sh, uint8_t *ring, Ring &r, int b, int j, int k)
{
    const bool has_d = (MODE == MODE_STOCH) && j < P.K;
    const char *row_t = static_cast<const char *>(P.target) + ((size_t)b * (P.K + 1) + j) * (size_t)P.V * P.es_t;
    const char *row_d = has_d ? static_cast<const char *>(P.draft) + ((size_t)b * P.K + j) * (size_t)P.Vd * P.es_d
                              : nullptr;
    const bool bulk = P.bulk_t && (!has_d || P.bulk_d);
    const int e_begin = k * P.rspt * RSE;
    const int e_end = min(P.V, e_begin + P.rspt * RSE);
    for (int e0 = e_begin; e0 < e_end; e0 += RSE) {
        const int n = min(RSE, e_end - e0);
        if (!ring_acquire(P, sh, r))
            return false;
        Meta &m = sh.meta[r.slot];
        m.kind = K_RES;
        m.b = b;
        m.pos = j;
        m.k = k;
        m.e0 = e0;
        m.n = n;
        m.last = (e0 + RSE >= e_end);
        m.direct = !bulk;
        m.g0 = row_t + (size_t)e0 * P.es_t;
        m.g1 = has_d ? row_d + (size_t)e0 * P.es_d : nullptr;
        ring_publish(sh, ring, r, bulk, m.g0, (uint32_t)(n * P.es_t), m.g1,
                     has_d ? (uint32_t)(n * P.es_d) : 0u);
        ring_advance(r);
    }
    return true;
}

template <class E, int MODE, bool PROBS>
__device__ void producer(const Params &P, Shared &sh, uint8_t *ring)
{
    Ring r;
    uint32_t ticket = P.n_res ? atomicAdd(&P.ctl[CTL_RES_TICKET], 1u) : 0xffffffffu;
    // The next stats task id is always fetched one task ahead, so the atomic's
    // round trip overlaps the issue of the current task.
    uint32_t t_next = atomicAdd(&P.ctl[CTL_STATS_NEXT], 1u);
    bool stats_left = true, ok = true;
    uint32_t idle = 0;
    const uint32_t per_pos = (uint32_t)P.B * (uint32_t)P.npt;
    while (ok) {
        if (sh.abort) {
            ok = false;
            break;
        }
        const uint32_t t = t_next;
        const bool have_t = stats_left && t < P.n_stats;
        int pos = 0, b = 0, k = 0;
        if (have_t) {
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
        // Both loads go out back to back; one round trip covers them.
        const bool want_res = ticket < P.n_res;
        const int b1 = want_res ? ld_acquire(&P.res_seq[ticket / (uint32_t)P.ncr]) : 0;
        const bool check_dead = have_t && pos > 0 && !P.full;
        const unsigned long long st = check_dead ? ld_vol(&P.state[b]) : 0ull;

        // 1. residual work for our ticket, once its sequence has ended (first,
        //    so that the rows it re-reads are still in L2)
        if (b1 > 0) {
            const int rb = b1 - 1, kres = (int)(ticket % (uint32_t)P.ncr);
            ticket = atomicAdd(&P.ctl[CTL_RES_TICKET], 1u);
            const int j = ld_vol(&P.terminal[rb]);
            if (j >= 0)
                ok = issue_residual<E, MODE, PROBS>(P, sh, ring, r, rb, j, kres);
            idle = 0;
            continue;
        }
        // 2. the next stats task, left to right by position; skipped when its
        //    sequence already ended before this position
        if (have_t) {
            t_next = atomicAdd(&P.ctl[CTL_STATS_NEXT], 1u);
            int j;
            if (check_dead && resolved(st, j) && j < pos)
                continue;
            ok = issue_stats<E, MODE, PROBS>(P, sh, ring, r, b, pos, k);
            idle = 0;
            continue;
        }
        stats_left = false;
        if (!want_res)
            break;
        if (ld_vol(&P.ctl[CTL_STATUS]) == (uint32_t)ST_TIMEOUT || ++idle > P.spin_limit) {
            ok = false;
            break;
        }
        __nanosleep(256);
    }
    if (ok && ring_acquire(P, sh, r)) {
        sh.meta[r.slot].kind = K_EXIT;
        mbar_arrive(&sh.full[r.slot]);
        return;
    }
    // Winding down: make the other warps leave, then wait for our own copies.
    abort_cta(P, sh);
    for (int s = 0; s < NST; ++s)
        if (r.txmask & (1u << s))
            mbar_wait(&sh.full[s], (r.phmask >> s) & 1u, DRAIN_LIMIT, nullptr);
}

// =================================================================== consumers
struct Acc {
    float m;     // running max (raw logits) / greedy best value
    float s;     // running sum relative to m
    int idx;     // greedy best index
    int flag;
};

template <class E>
__device__ __forceinline__ void load_stage(const Meta &m, const uint8_t *st, int ctid, float *x)
{
    constexpr int VE = E::VE;
    if (!m.direct) {
        const uint4 *sv = reinterpret_cast<const uint4 *>(st);
        const int nvec = m.n / VE;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = ctid + 256 * k;
            const uint4 w = v < nvec ? sv[v] : E::neg_inf();
            E::unpack(w, x + k * VE);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                const int i = (ctid + 256 * k) * VE + e;
                x[k * VE + e] = i < m.n ? E::load(m.g0, i) : -F_INF;
            }
    }
}

// Online max / sum of 2^((x - m) c) over the 4*VE elements of this thread.
template <int NE>
__device__ __forceinline__ void online_update(const float *x, float c, Acc &a)
{
    float lm = x[0];
#pragma unroll
    for (int i = 1; i < NE; ++i)
        lm = fmax_nan(lm, x[i]);
    const float mn = fmax_nan(a.m, lm);
    const float ref = (mn == -F_INF) ? 0.0f : mn;
    if (mn != a.m)
        a.s *= ex2a((a.m - ref) * c);
    float t[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i)
        t[i] = ex2a((x[i] - ref) * c);
#pragma unroll
    for (int w = NE / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] += t[i + w];
    a.s += t[0];
    a.m = mn;
}

template <class E>
__device__ __forceinline__ void greedy_update(const float *x, const Meta &m, int ctid, Acc &a)
{
    constexpr int VE = E::VE;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            const float v = x[k * VE + e];
            a.flag |= (v != v);
            if (v > a.m) {
                a.m = v;
                a.idx = m.e0 + (ctid + 256 * k) * VE + e;
            }
        }
}

// Shortlist: check entries [e0, e0+n) of sequence b's index row (ascending,
// unique, inside [0, V)); at position 0 also record, for each 256-token
// segment t, the first entry whose token is >= 256 t.
static __device__ void shortlist_scan(const Params &P, const Meta &m, int ctid, bool record, int &flag)
{
    const int32_t *idx = P.shortlist + (size_t)m.b * P.S;
    int32_t *lb = P.sl_lb + (size_t)m.b * (P.nseg + 1);
    for (int s = m.e0 + ctid; s < m.e0 + m.n; s += 256) {
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
// r(x) for one token: target logit xt, draft value xd (logit, or probability
// when PROBS); q receives q(x).  `bonus` samples q itself.
template <bool PROBS>
__device__ __forceinline__ float res_elem(float xt, float xd, const ResCoef &k, bool bonus, float &q)
{
    if (xt == -F_INF) {
        q = 0.0f;
        return 0.0f;
    }
    q = ex2a((xt - k.Mt) * k.c - k.Lt2);
    if (bonus)
        return q;
    if (PROBS) {
        const float d = q - xd;
        return d > 0.0f ? d : 0.0f;
    }
    const float delta = ((xd - xt) * k.c - k.dLhi) - k.dLlo;   // log2(p(x) / q(x))
    return delta < 0.0f ? q * one_minus_pow2(delta) : 0.0f;
}

// Draft values of the 8 tokens [x0 + 8 lane, +8) of a 256-token segment.
// Full vocabulary: from the stage (bulk) or global memory.  Shortlist: scatter
// the segment's entries into a per-warp buffer first (absent tokens read as
// -inf logits / zero probabilities, i.e. p = 0).
template <class E, int MODE, bool PROBS>
__device__ __forceinline__ void draft_values(const Params &P, int b, int j, int x0, int lane, int cnt,
                                             const uint8_t *st_d, const void *g_d, bool direct,
                                             float *pscr, float *xd, int &flag)
{
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
        if (!direct) {
            float tmp[8];
            const uint4 *sv = reinterpret_cast<const uint4 *>(st_d + (size_t)lane * 8 * D::ES);
            if (D::VE == 8) {
                D::unpack(sv[0], tmp);
            } else {
                D::unpack(sv[0], tmp);
                D::unpack(sv[1], tmp + 4);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                xd[e] = tmp[e];
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
}

// r and q for the 8 tokens starting at x0 + 8*lane of one segment, the
// lane's sums (in token order) and the last token with r > 0.
template <class E, int MODE, bool PROBS>
__device__ __forceinline__ void residual_lane(const Params &P, int b, int j, int x0, int cnt, int lane,
                                              const uint8_t *st_t, const void *g_t, const uint8_t *st_d,
                                              const void *g_d, bool direct, float *pscr,
                                              const ResCoef &kc, float *r, float &rsum, float &qsum,
                                              int &last, int &flag)
{
    const bool bonus = (j == P.K);
    float xt[8], xd[8];
    if (!direct && cnt == 8) {
        const uint4 *sv = reinterpret_cast<const uint4 *>(st_t + (size_t)lane * 8 * E::ES);
        if (E::VE == 8) {
            E::unpack(sv[0], xt);
        } else {
            E::unpack(sv[0], xt);
            E::unpack(sv[1], xt + 4);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            xt[e] = e < cnt ? E::load(g_t, (size_t)lane * 8 + e) : -F_INF;
    }
    if (!bonus) {
        draft_values<E, MODE, PROBS>(P, b, j, x0, lane, cnt, st_d, g_d, direct || cnt != 8, pscr, xd, flag);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            xd[e] = 0.0f;
    }
    rsum = 0.0f;
    qsum = 0.0f;
    last = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        float q = 0.0f;
        r[e] = 0.0f;
        if (e < cnt)
            r[e] = res_elem<PROBS>(xt[e], xd[e], kc, bonus, q);
        rsum += r[e];
        qsum += q;
        if (r[e] > 0.0f)
            last = x0 + lane * 8 + e;
    }
}

// Hand the warp's task result to the finisher.
__device__ __forceinline__ bool hand_over(const Params &P, Shared &sh, int cw, int lane, uint32_t &hs,
                                          uint32_t &hph, int kind, const Meta &m, float wm, DF ws,
                                          int wf, int wi)
{
    if (!warp_wait(&sh.hempty[hs], hph ^ 1u, P.spin_limit, &sh.abort, lane))
        return false;
    if (lane == 0) {
        Hand &h = sh.hand[hs];
        if (cw == 0) {
            h.kind = kind;
            h.b = m.b;
            h.pos = m.pos;
            h.k = m.k;
        }
        h.wm[cw] = wm;
        h.ws_hi[cw] = ws.hi;
        h.ws_lo[cw] = ws.lo;
        h.wf[cw] = wf;
        h.wi[cw] = wi;
        mbar_arrive(&sh.hfull[hs]);
    }
    __syncwarp();
    if (++hs == NH) {
        hs = 0;
        hph ^= 1u;
    }
    return true;
}

template <class E, int MODE, bool PROBS>
__device__ void consumer(const Params &P, Shared &sh, const uint8_t *ring, int cw, int lane)
{
    constexpr int NE = 4 * E::VE;
    const int ctid = cw * 32 + lane;
    uint32_t slot = 0, ph = 0, hs = 0, hph = 0;
    Acc a{-F_INF, 0.0f, 0x7fffffff, 0};
    for (;;) {
        if (!warp_wait(&sh.full[slot], ph, P.spin_limit, &sh.abort, lane)) {
            abort_cta(P, sh);
            return;
        }
        const Meta m = sh.meta[slot];
        const uint8_t *st = ring + (size_t)slot * STAGE_BYTES;
        if (m.kind == K_EXIT) {
            hand_over(P, sh, cw, lane, hs, hph, K_EXIT, m, 0.0f, DF{0.0f, 0.0f}, 0, 0);
            return;
        }
        if (m.kind == K_RES) {
            // one 256-token segment per warp
            int flag = 0;
            const int eb = cw * SEG;
            if (eb < m.n) {
                const int x0 = m.e0 + eb;
                const int cnt = max(0, min(8, m.n - eb - lane * 8));
                const ResCoef kc = load_coef(P, m.b, m.pos);
                float r[8], rsum, qsum;
                int last;
                const void *g_t = static_cast<const char *>(m.g0) + (size_t)eb * P.es_t;
                const void *g_d = m.g1 ? static_cast<const char *>(m.g1) + (size_t)eb * P.es_d : nullptr;
                residual_lane<E, MODE, PROBS>(P, m.b, m.pos, x0, cnt, lane, st + (size_t)eb * P.es_t, g_t,
                                              st + RD_OFF + (size_t)eb * P.es_d, g_d, m.direct != 0,
                                              sh.pscr[cw], kc, r, rsum, qsum, last, flag);
                rsum = warp_sumf(rsum);
                qsum = warp_sumf(qsum);
                last = warp_maxi(last);
                flag = warp_or(flag);
                if (lane == 0) {
                    const size_t si = (size_t)m.b * P.nseg + x0 / SEG;
                    P.seg[si] = SegMass{rsum, qsum};
                    P.seglast[si] = last;
                }
            }
            a.flag |= flag;
        } else {
            float x[NE];
            if (m.kind == K_STAT_D && PROBS) {
                // draft probabilities have no stats pass
            } else if (m.kind == K_STAT_D) {
                load_stage<E>(m, st, ctid, x);
                online_update<NE>(x, P.c, a);
            } else {
                load_stage<E>(m, st, ctid, x);
                if (MODE == MODE_GREEDY)
                    greedy_update<E>(x, m, ctid, a);
                else
                    online_update<NE>(x, P.c, a);
            }
            if (MODE == MODE_SHORT && m.kind == K_STAT_D && (m.pos == 0 || P.full))
                shortlist_scan(P, m, ctid, m.pos == 0, a.flag);
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sh.empty[slot]);
        if (m.last) {
            bool hok;
            if (m.kind == K_RES) {
                hok = hand_over(P, sh, cw, lane, hs, hph, K_RES, m, 0.0f, DF{0.0f, 0.0f}, warp_or(a.flag), 0);
            } else if (MODE == MODE_GREEDY) {
                float v = a.m;
                int i = a.idx;
#pragma unroll
                for (int o = 16; o; o >>= 1) {
                    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
                    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
                    argmax_merge(v, i, v2, i2);
                }
                const int fl = warp_or(a.flag | (a.m == F_INF));
                hok = hand_over(P, sh, cw, lane, hs, hph, m.kind, m, v, DF{0.0f, 0.0f}, fl, i);
            } else {
                const float wm = warp_max_nan(a.m);
                const int fl = warp_or(a.flag | (a.m != a.m) | (a.m == F_INF));
                DF contrib{0.0f, 0.0f};
                if (a.m > -F_INF && a.s > 0.0f)
                    contrib = df_scale_pow2(DF{a.s, 0.0f}, (a.m - wm) * P.c);
                const DF ws = warp_sum_df(contrib);
                hok = hand_over(P, sh, cw, lane, hs, hph, m.kind, m, wm, ws, fl, 0);
            }
            if (!hok) {
                abort_cta(P, sh);
                return;
            }
            a = Acc{-F_INF, 0.0f, 0x7fffffff, 0};
        }
        if (++slot == NST) {
            slot = 0;
            ph ^= 1u;
        }
    }
}

// =================================================================== finisher
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
        __threadfence();
        const uint32_t slot = atomicAdd(&P.ctl[CTL_RES_COUNT], 1u);
        st_vol(&P.res_seq[slot], b + 1);
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
__device__ void locate(const Params &P, Shared &sh, int b, int j, int lane)
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
        float r[8], rsum, qsum;
        int last, flag = 0;
        residual_lane<E, MODE, PROBS>(P, b, j, x0, cnt, lane, nullptr, row_t + (size_t)x0 * P.es_t, nullptr,
                                      has_d ? row_d + (size_t)x0 * P.es_d : nullptr, true, sh.pscr[NCW], kc, r,
                                      rsum, qsum, last, flag);
        float qv[8];
        if (use_q) {
            // sample q itself: recompute q per token
            rsum = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float q = 0.0f;
                if (e < cnt) {
                    const float xt = E::load(row_t + (size_t)x0 * P.es_t, (size_t)lane * 8 + e);
                    res_elem<PROBS>(xt, 0.0f, kc, true, q);
                }
                qv[e] = q;
                rsum += q;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                qv[e] = r[e];
        }
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
            cand = max(cand, ld_vol(&P.seglast[(size_t)b * nseg + s]));
        x = warp_maxi(cand);
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

// Merge the 8 warp results of a stats hand-off into one chunk partial.
template <int MODE>
__device__ __forceinline__ Partial merge_hand(const Params &P, const Hand &h, int lane)
{
    Partial out;
    if (MODE == MODE_GREEDY) {
        float v = lane < NCW ? h.wm[lane] : -F_INF;
        int i = lane < NCW ? h.wi[lane] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
            argmax_merge(v, i, v2, i2);
        }
        out.m = v;
        out.s_hi = __int_as_float(i);
        out.s_lo = 0.0f;
    } else {
        const float wm = lane < NCW ? h.wm[lane] : -F_INF;
        const float M = warp_max_nan(wm);
        DF c{0.0f, 0.0f};
        if (lane < NCW && wm > -F_INF)
            c = df_scale_pow2(DF{h.ws_hi[lane], h.ws_lo[lane]}, (wm - M) * P.c);
        const DF t = warp_sum_df(c);
        out.m = M;
        out.s_hi = t.hi;
        out.s_lo = t.lo;
    }
    out.flag = warp_or(lane < NCW ? h.wf[lane] : 0);
    return out;
}

// The finisher takes every hand-off that is ready (up to NH), merges them,
// writes all their results, fences once, and bumps all their counters in
// parallel (one lane per hand-off); the hand-offs whose counter completes a
// position (or a sequence's residual) then decide (or locate).
template <class E, int MODE, bool PROBS>
__device__ void finisher(const Params &P, Shared &sh, int lane)
{
    uint32_t hs = 0, hph = 0;
    for (;;) {
        if (!warp_wait(&sh.hfull[hs], hph, P.spin_limit, &sh.abort, lane)) {
            abort_cta(P, sh);
            return;
        }
        int n = 1;
        if (lane == 0) {
            uint32_t s = hs, p = hph;
            while (n < NH) {
                if (++s == NH) {
                    s = 0;
                    p ^= 1u;
                }
                if (!mbar_test(&sh.hfull[s], p))
                    break;
                ++n;
            }
        }
        n = __shfl_sync(0xffffffffu, n, 0);
        int my_kind = -1, my_b = 0, my_pos = 0, my_k = 0;
        Partial my_out{0.0f, 0, 0.0f, 0.0f};
        bool exit_seen = false;
        int m = 0;
        for (int i = 0; i < n; ++i) {
            if (i > 0)
                (void)mbar_test(&sh.hfull[hs], hph);   // this lane's own acquire of the completed phase
            __syncwarp();
            const Hand &h = sh.hand[hs];
            const int kind = h.kind;
            if (kind == K_EXIT) {
                exit_seen = true;
                break;
            }
            Partial out{0.0f, 0, 0.0f, 0.0f};
            if (kind == K_RES) {
                out.flag = warp_or(lane < NCW ? h.wf[lane] : 0);
            } else {
                out = merge_hand<MODE>(P, h, lane);
            }
            if (lane == i) {
                my_kind = kind;
                my_b = h.b;
                my_pos = h.pos;
                my_k = h.k;
                my_out = out;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sh.hempty[hs]);
            ++m;
            if (++hs == NH) {
                hs = 0;
                hph ^= 1u;
            }
        }
        // publish: one lane per hand-off writes, one fence, then the counters
        const size_t bp = (size_t)my_b * (P.K + 1) + my_pos;
        if (lane < m) {
            if (my_kind == K_RES) {
                if (my_out.flag)
                    st_vol(&P.errres[my_b], 1);
            } else {
                P.part[bp * P.npt + my_k] = my_out;
            }
        }
        __threadfence();
        bool last = false;
        if (lane < m) {
            if (my_kind == K_RES) {
                last = atomicAdd(&P.res_cnt[my_b], 1u) == (uint32_t)P.ncr - 1u;
            } else {
                const int nparts = my_pos < P.K ? P.npt : P.nct;
                last = atomicAdd(&P.pair_cnt[bp], 1u) == (uint32_t)nparts - 1u;
            }
        }
        unsigned lastmask = __ballot_sync(0xffffffffu, last);
        if (lastmask)
            __threadfence();
        while (lastmask) {
            const int i = __ffs(lastmask) - 1;
            lastmask &= lastmask - 1;
            const int kind = __shfl_sync(0xffffffffu, my_kind, i);
            const int b = __shfl_sync(0xffffffffu, my_b, i);
            const int pos = __shfl_sync(0xffffffffu, my_pos, i);
            if (kind == K_RES)
                locate<E, MODE, PROBS>(P, sh, b, pos, lane);
            else
                decide<E, MODE, PROBS>(P, b, pos, lane);
        }
        if (exit_seen)
            return;
    }
}

// =================================================================== kernel
template <class E, int MODE, bool PROBS>
__global__ void __launch_bounds__(NTHREADS, 2) verify_kernel(const __grid_constant__ Params P)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *ring = smem_raw;
    Shared &sh = *reinterpret_cast<Shared *>(smem_raw + (size_t)NST * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], NCW);
        }
        for (int h = 0; h < NH; ++h) {
            mbar_init(&sh.hfull[h], NCW);
            mbar_init(&sh.hempty[h], 1);
        }
        sh.abort = 0;
        sh.last_cta = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (warp < NCW)
        consumer<E, MODE, PROBS>(P, sh, ring, warp, lane);
    else if (warp == W_PROD) {
        if (lane == 0)
            producer<E, MODE, PROBS>(P, sh, ring);
    } else {
        finisher<E, MODE, PROBS>(P, sh, lane);
    }
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
