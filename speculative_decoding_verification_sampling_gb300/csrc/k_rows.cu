// k_rows.cu -- row-parallel verification: statistics, residual masses, draw.
//
// The rule is that of the other kernels (nextadmin.net lesson "Speculative
// Decoding", § Core algorithm steps 4-6; aiengineeringfromscratch.com lesson
// 25, § The exact rule and § Greedy case; q = target, p = draft).  Here the
// work is cut by rows instead of by sequences, so that every SM streams
// independent rows at full bandwidth:
//   1. Row statistics: each logit row is streamed once into its reference
//      and sum, keeping the logit at the drafted token.
//      The second row of a position to finish decides it; a rejection (or an
//      error) sets the position's bit in the sequence's mask.  Rows of a
//      sequence with a bit below their position skip their reads, so only the
//      rows the left-to-right rule examines are streamed (up to the rows
//      started before the decision they wait on is known).
//      - vr_stream (stochastic calls with draft logits and aligned rows): one
//        persistent launch; rows are claimed position-major from a counter
//        and copied in 16 KB stages by cp.async.bulk into a shared-memory
//        ring, reduced by consumer warps; an epilogue thread decides.
//      - vr_stats (shortlisted drafts, unaligned rows): one launch for
//        positions 0-1 and one for the rest, one CTA per part of a row,
//        16-byte loads with four in flight per thread.
//   2. vr_residual: eight CTAs per sequence.  The mask gives the position j
//      where the sequence ends; each CTA streams its eighth of row pair j into
//      residual masses r' = q' (1 - 2^delta)_+ and target masses q' per
//      256-token segment, in token order.
//   3. vr_sample: one CTA per sequence.  It scans the segment masses for the
//      one crossing v * R, reads that segment again and locates the token
//      (inverse CDF in ascending token order); it writes the outputs and
//      re-zeroes the sequence's control words.
// Small calls whose rows all fit shared memory run on vr_resident and
// vr_sample; greedy verification has its own kernels (k_greedy_rows.cu).
#include "sv_cluster.cuh"
#include "sv_launch.h"

#include <algorithm>
#include <cstdlib>

namespace sv {
namespace {

constexpr int VR_NCH = 8;      // vr_residual CTAs per sequence
constexpr int VRT = 256;       // threads of a vr_residual CTA
constexpr int VST = 128;       // threads of a vr_sample CTA
constexpr int VSEG = 256;      // tokens per residual segment (one per lane-unit of a warp)

// Tokens [x0, x0 + 8) of a row as four float pairs (-inf at or past V).
template <class E>
struct Unit {
    uint4 a, b;   // raw 16-byte loads (b only for float32)
};
template <class E>
__device__ __forceinline__ Unit<E> fetch_unit(const uint8_t *row, int x0, int V, bool vec)
{
    Unit<E> u{};
    if (vec && x0 + 8 <= V) {
        const uint4 *p = reinterpret_cast<const uint4 *>(row + (size_t)x0 * E::ES);
        u.a = __ldg(p);
        if constexpr (E::ES == 4)
            u.b = __ldg(p + 1);
        return u;
    }
    uint32_t w[8];
    if constexpr (E::ES == 2) {
        const uint16_t *h = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = x0 + 2 * k < V ? (uint32_t)__ldg(h + x0 + 2 * k) : 0xff80u;
            const uint32_t hi = x0 + 2 * k + 1 < V ? (uint32_t)__ldg(h + x0 + 2 * k + 1) : 0xff80u;
            w[k] = lo | (hi << 16);
        }
        u.a = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        const uint32_t *f = reinterpret_cast<const uint32_t *>(row);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            w[k] = x0 + k < V ? __ldg(f + x0 + k) : 0xff800000u;
        u.a = make_uint4(w[0], w[1], w[2], w[3]);
        u.b = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return u;
}
template <class E>
__device__ __forceinline__ void unit_pairs(const Unit<E> &u, f2 *X)
{
    if constexpr (E::ES == 2) {
#pragma unroll
        for (int p = 0; p < 4; ++p)
            X[p] = E::pair(u.a, p);
    } else {
        X[0] = E::pair(u.a, 0);
        X[1] = E::pair(u.a, 1);
        X[2] = E::pair(u.b, 0);
        X[3] = E::pair(u.b, 1);
    }
}

__device__ __forceinline__ VrStat ld_vrstat(const VrStat *p)
{
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    return VrStat{a.x, a.y, a.z, __float_as_int(a.w), b.x, 0, 0, 0};
}
__device__ __forceinline__ uint32_t vr_atom_add(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Decide position i of sequence b from the statistics of its target row t and
// draft row d (the drafted token dt).  Returns 0 and sets accept, or a status
// code.  Checks in the oracle's order: token, target row, draft row.
__device__ __forceinline__ int vr_decide(const RowsParams &P, int b, int i, int dt, const VrStat &t,
                                         const VrStat &d, bool &accept)
{
    accept = false;
    if (i < P.K && (d.flags & VR_SLBAD))
        return ST_SHORTLIST;   // the position's shortlist, before its token
    if (i < P.K && !(dt >= 0 && dt < P.V))
        return ST_TOKEN;
    if ((t.flags & VR_BAD) || !(t.m > -F_INF) || !(t.s_hi > 0.0f))
        return ST_NONFINITE;
    if (i == P.K)
        return 0;
    if (P.probs) {
        // the given p_i(d_i): finite and >= 0; 0 accepts; else
        // log2(q(d) / p(d)) = zt c - Mt - log2 St - log2 p(d)
        const float pd = __ldg(static_cast<const float *>(P.draft) + ((size_t)b * P.K + i) * (size_t)P.V + dt);
        if (!(pd >= 0.0f) || pd == F_INF)
            return ST_NONFINITE;
        if (pd == 0.0f) {
            accept = true;
            return 0;
        }
        int et;
        float ft;
        log2_split(DF{t.s_hi, t.s_lo}, et, ft);
        const float X = t.zd * P.c - (t.m + ((float)et + ft)) - lg2a(pd);
        const uint4 w = philox10((uint32_t)i, (uint32_t)b, 0u, 0u, P.key0, P.key1);
        accept = X >= 0.0f || u24_below(w.x, ex2a(X));
        return 0;
    }
    if ((d.flags & VR_BAD) || !(d.m > -F_INF) || !(d.s_hi > 0.0f))
        return ST_NONFINITE;
    int et, ed;
    float ft, fd;
    log2_split(DF{t.s_hi, t.s_lo}, et, ft);
    log2_split(DF{d.s_hi, d.s_lo}, ed, fd);
    const float zt = t.zd, zd = d.zd;
    // p(d) == 0 (or below the float64 range) accepts
    const float lp = zd * P.c - d.m - ((float)ed + fd);
    if (zd == -F_INF || lp < -1074.5f) {
        accept = true;
        return 0;
    }
    // log2(q(d) / p(d)) = (zt - zd) c - (Mt - Md) - (log2 St - log2 Sd)
    const float X = (zt - zd) * P.c - ((t.m - d.m) + ((float)(et - ed) + (ft - fd)));
    const uint4 w = philox10((uint32_t)i, (uint32_t)b, 0u, 0u, P.key0, P.key1);
    accept = X >= 0.0f || u24_below(w.x, ex2a(X));
    return 0;
}

// Where sequence b ends, from the decisions of the row kernels: the first
// position decided against (its status in errc; 0 for a plain rejection), or
// K when all K drafts were accepted (errc[K] if the bonus row is in error).
// Every position before it was computed and accepted: none of its rows could
// skip, and the second of its rows to finish decided it.
__device__ __forceinline__ int vr_end(const RowsParams &P, int b, int &j)
{
    const uint32_t m = __ldcg(P.rej + b);
    j = m ? __ffs(m) - 1 : P.K;
    return (m >> j) & 1u ? __ldcg(P.errc + (size_t)b * (P.K + 1) + j) : 0;
}

__device__ __forceinline__ unsigned long long vr_atom_or64(unsigned long long *p, unsigned long long v)
{
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t ld_acq(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_acq_s32(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_rel_s32(int *p, int v)
{
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Whether a sequence's word (decided positions low, ending positions high)
// says it has ended: the first ending position j and every position up to it
// decided.
__device__ __forceinline__ bool vr_ended(unsigned long long w)
{
    const uint32_t E = (uint32_t)(w >> 32), D = (uint32_t)w;
    if (!E)
        return false;
    const int j = __ffs(E) - 1;
    const uint32_t need = j == 31 ? 0xffffffffu : (2u << j) - 1u;
    return (D & need) == need;
}
__device__ __noinline__ void vr_post_end(const RowsParams &P, int b, unsigned long long w);

// The statistics of a row from its n parts' records (pp[0..n)): the largest
// reference, the sums rescaled to it (exact powers of two) and added as a
// float pair, the flags, the drafted token's logit from the part holding it.
__device__ __forceinline__ VrStat merge_parts(const VrStat *pp, int n)
{
    constexpr int MU = 4;   // records loaded at once (a few registers: the kernel keeps 3 CTAs per SM)
    float M = -F_INF, zd = 0.0f;
    DF S{0.0f, 0.0f};
    int fl = 0;
    for (int h0 = 0; h0 < n; h0 += MU) {
        float4 a[MU];
        float z[MU];
#pragma unroll
        for (int k = 0; k < MU; ++k)
            if (h0 + k < n) {
                a[k] = __ldcg(reinterpret_cast<const float4 *>(pp + h0 + k));
                z[k] = __ldcg(&pp[h0 + k].zd);
            }
#pragma unroll
        for (int k = 0; k < MU; ++k)
            if (h0 + k < n) {
                const int f = __float_as_int(a[k].w);
                fl |= f;
                if (f & VR_HASD)
                    zd = z[k];
                const float mk = a[k].x;
                if (mk > -F_INF) {
                    if (mk > M) {
                        S = M > -F_INF ? df_scale_pow2(S, M - mk) : DF{0.0f, 0.0f};
                        M = mk;
                    }
                    S = df_add(S, df_scale_pow2(DF{a[k].y, a[k].z}, mk - M));
                }
            }
    }
    return VrStat{M, S.hi, S.lo, fl, zd, 0, 0, 0};
}

// The epilogue of vr_stream: part `part` of the target (kind 0) or draft
// (kind 1) row of position i of sequence b has statistics st.  One counter per
// position counts the parts of both rows; the last part to finish merges
// every part (one round of loads), records the two rows and decides the
// position.  A rejection or an error sets the position's bit in rej, and the
// per-sequence word of decided and ending positions finds the sequence's end
// (vr_commit's way).
// A part's statistics st of row ridx (sequence b, position i; kind 1: the
// draft row), from one CTA: the last part of the row to finish merges the
// parts in part order and writes the row's statistics; the second row of a
// position to finish decides it (position K: the only row), and a rejection
// or an error sets the position's bit in rej.
__device__ __noinline__ void vr_commit(const RowsParams &P, size_t ridx, int b, int i, int kind, int part, int dt,
                                       VrStat st, bool slrow)
{
    const int K = P.K;
    const bool pairs = i < K;
    if (P.parts > 1) {
        // the last part of the row to finish merges the parts, in part order
        VrStat *pp = P.vpart + ridx * VR_SMAX;
        pp[part] = st;
        if (vr_atom_add(P.rowcnt + ridx, 1u) != (uint32_t)(P.parts - 1))
            return;
        // the parts' records, four loads in flight at a time
        VrStat m = merge_parts(pp, P.parts);
        if (slrow && !(m.flags & VR_HASD))
            m.zd = -F_INF;   // the drafted token is not on the list: p(d) = 0
        st = m;
    }
    P.stat[ridx] = st;
    // the second row of a position to finish decides it (position K: the only
    // row); a rejection or an error sets the position's bit
    VrStat t = st, d{};
    if (pairs) {
        if (vr_atom_add(P.pair + (size_t)b * (K + 1) + i, 1u) != 1u)
            return;
        const VrStat o = ld_vrstat(P.stat + (size_t)b * (2 * K + 1) + (kind ? i : K + 1 + i));
        t = kind ? o : st;
        d = kind ? st : o;
    }
    bool acc = false;
    const int code = vr_decide(P, b, i, dt, t, d, acc);
    const bool ends = code || (!acc && i < K);
    if (ends) {
        P.errc[(size_t)b * (K + 1) + i] = code;
        atomicOr(P.rej + b, 1u << i);
    }
    if (P.fused) {
        // position i decided (and ending the sequence, at K always): the update
        // completing the sequence's end posts its residual job
        const unsigned long long bits = (1ull << i) | ((ends || i == K) ? (1ull << (32 + i)) : 0ull);
        const unsigned long long old = vr_atom_or64(P.dw + b, bits);
        if (P.fused == 1 && !vr_ended(old) && vr_ended(old | bits))
            vr_post_end(P, b, old | bits);
    }
}

// ---------------------------------------------------------------- 1. row statistics
template <class E, int VT, bool SL>
__global__ void __launch_bounds__(VT) vr_stats(const __grid_constant__ RowsParams P)
{
    pdl_wait();
    pdl_trigger();
    constexpr int NW = VT / 32;
    __shared__ float sm_m[NW], sm_hi[NW], sm_lo[NW];
    __shared__ int sm_f[NW];
    __shared__ float sm_zd;
    __shared__ int sm_skip;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = P.K, V = P.V;
    // this launch's rows, position-major over [P.pos, P.pos + P.npos): the
    // target and draft rows of each sequence side by side (the target row
    // alone at position K), each cut into P.parts parts of P.span tokens, one
    // CTA each
    const int rpp = 2 * P.B;   // rows of a position below K
    const int rg = (int)blockIdx.x / P.parts, part = (int)blockIdx.x % P.parts;
    const int i = P.pos + rg / rpp;
    const int rl = rg % rpp;
    const int b = rl >> 1;
    const int kind = rl & 1;
    if (kind && i == K)
        return;   // position K has no draft row
    const size_t ridx = (size_t)b * (2 * K + 1) + (kind ? K + 1 + i : i);
    if (P.skip && i > 0) {
        // a rejection (or error) decided at an earlier position makes this row unneeded
        if (tid == 0) {
            const uint32_t m = __ldcg(P.rej + b);
            sm_skip = (m & ((1u << i) - 1u)) != 0u;
        }
        __syncthreads();
        if (sm_skip) {
            if (tid == 0 && part == 0)
                P.stat[ridx] = VrStat{-F_INF, 0.0f, 0.0f, VR_SKIP, 0.0f, 0, 0, 0};
            return;
        }
    }
    // a shortlisted draft row holds sl_len[i] logits, for the listed tokens
    const bool slrow = SL && kind;   // (SL: the call has a shortlisted draft)
    const int nrow = slrow ? P.sl_len[i] : V;
    const uint8_t *row =
        kind ? static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + i) * (size_t)(SL ? P.S : V) * E::ES
             : static_cast<const uint8_t *>(P.target) + ((size_t)b * (K + 1) + i) * (size_t)V * E::ES;
    const int32_t *lst = slrow ? P.sl + b * P.sl_seq + i * P.sl_pos : nullptr;
    const int dt = i < K ? __ldg(P.tokens + (size_t)b * K + i) : -1;
    // a shortlisted draft row is cut by its own length, so that its list
    // entries (the slow part of the row) spread over every part
    const int span = slrow ? ((nrow + P.parts - 1) / P.parts + 7) / 8 * 8 : P.span;
    const int t0 = min(nrow, part * span), t1 = min(nrow, t0 + span);
    const int u0 = t0 / 8, nu = (t1 - t0 + 7) / 8;   // this part's units of 8 tokens
    const float c = P.c;
    float mc = -F_INF, s = 0.0f, zd = 0.0f;
    int fl = 0;
    bool hz = false;
    // four units in flight per thread; each buffer is refilled right after its use
    Unit<E> u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (tid + k * VT < nu)
            u[k] = fetch_unit<E>(row, (u0 + tid + k * VT) * 8, t1, P.vec);
    for (int g0 = tid; g0 < nu; g0 += 4 * VT) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int g = g0 + k * VT;
            if (g < nu) {
                f2 X[4];
                unit_pairs<E>(u[k], X);
                if (g + 4 * VT < nu)
                    u[k] = fetch_unit<E>(row, (u0 + g + 4 * VT) * 8, t1, P.vec);
                const int x0 = (u0 + g) * 8;
                if (slrow) {
                    // the unit's list entries: strictly ascending inside [0, V); the
                    // drafted token's logit; the first entry of each 256-token segment
                    float x[8];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        upk(X[p], x[2 * p], x[2 * p + 1]);
                    int32_t *lb = P.lb + ((size_t)b * K + i) * (P.nseg + 1);
                    int prev = x0 > 0 ? __ldg(lst + x0 - 1) : -1;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int si = x0 + e;
                        if (si >= t1)
                            break;
                        const int cur = __ldg(lst + si);
                        if (cur < 0 || cur >= V || cur <= prev) {
                            fl |= VR_SLBAD;
                        } else {
                            if (cur == dt) {
                                zd = x[e];
                                hz = true;
                            }
                            for (int t = prev < 0 ? 0 : prev / VSEG + 1; t <= cur / VSEG; ++t)
                                lb[t] = si;
                            if (si == nrow - 1)
                                for (int t = cur / VSEG + 1; t <= P.nseg; ++t)
                                    lb[t] = nrow;
                        }
                        prev = cur;
                    }
                } else if ((unsigned)(dt - x0) < 8u) {
                    float x[8];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        upk(X[p], x[2 * p], x[2 * p + 1]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (dt == x0 + e) {
                            zd = x[e];
                            hz = true;
                        }
                    }
                }
                acc_group(X, c, mc, s, fl, VR_BAD);
            }
        }
    }
    if (hz) {
        sm_zd = zd;
        fl |= VR_HASD;
    }
    fl = warp_or(fl);
    {
        float M;
        DF S;
        merge_ms<32>(mc, DF{s, 0.0f}, c, M, S);
        if (lane == 0) {
            sm_m[warp] = M;
            sm_hi[warp] = S.hi;
            sm_lo[warp] = S.lo;
            sm_f[warp] = fl;
        }
    }
    __syncthreads();
    if (warp != 0)
        return;
    const bool in = lane < NW;
    VrStat st{};
    st.flags = warp_or(in ? sm_f[lane] : 0);
    // the drafted token's logit, from the thread that held it (VR_HASD); a
    // shortlisted draft row without it gives p(d) = 0
    st.zd = (st.flags & VR_HASD) ? sm_zd : (slrow ? -F_INF : 0.0f);
    {
        float M;
        DF S;
        merge_ms<NW>(in ? sm_m[lane] : -F_INF, in ? DF{sm_hi[lane], sm_lo[lane]} : DF{0.0f, 0.0f}, c, M, S);
        st.m = M;
        st.s_hi = S.hi;
        st.s_lo = S.lo;
    }
    if (lane == 0)
        vr_commit(P, ridx, b, i, kind, part, dt, st, slrow);
}

// ---------------------------------------------------------------- residual arithmetic
// q'(x) = 2^(xt c - Mt) and r'(x) = q'(x) (1 - 2^delta)_+ for 8 tokens as four
// float pairs, delta = (xd - xt) c - dL (both scaled by the target's
// normaliser, which cancels in the inverse CDF).  1 - 2^delta on [-1, 0) is
// 2^(delta/2) * (-2 sinh(delta ln2 / 2)) with sinh as its odd Taylor series to
// y^7 (|y| <= ln2 / 2, so the first term left out is below 6e-9 relative;
// the factor -2 is folded into the coefficients, an exact scaling), so
// nothing cancels as q -> p; below -1 it is 1 - 2^delta.  With qonly (the
// bonus row) r' = q'.
__device__ __forceinline__ void vr_res8(const f2 *XT, const f2 *XD, const ResK &k, bool qonly, f2 *R, f2 *Q)
{
    const f2 cc = pk(k.c, k.c), nMt = pk(-k.Mt, -k.Mt);
#pragma unroll
    for (int p = 0; p < 4; ++p)
        Q[p] = ex2x2(fma2(XT[p], cc, nMt));
    if (qonly) {
#pragma unroll
        for (int p = 0; p < 4; ++p)
            R[p] = Q[p];
        return;
    }
    const f2 ndh = pk(-k.dLhi, -k.dLhi), ndl = pk(-k.dLlo, -k.dLlo);
    const f2 hl = pk(0.34657359027997264f, 0.34657359027997264f);   // ln2 / 2
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const f2 dd = fma2(XT[p], pk(-1.0f, -1.0f), XD[p]);           // xd - xt
        float d0, d1;
        upk(add2(fma2(dd, cc, ndh), ndl), d0, d1);                    // delta
        d0 = fminf(d0, 0.0f);                                         // also maps NaN (both -inf) to 0
        d1 = fminf(d1, 0.0f);
        const bool far0 = d0 < -1.0f, far1 = d1 < -1.0f;
        float e0, e1;
        upk(ex2x2(pk(far0 ? d0 : 0.5f * d0, far1 ? d1 : 0.5f * d1)), e0, e1);
        const f2 y = mul2(pk(d0, d1), hl);
        const f2 y2 = mul2(y, y);
        f2 sp = pk(-2.0f / 5040.0f, -2.0f / 5040.0f);
        sp = fma2(sp, y2, pk(-2.0f / 120.0f, -2.0f / 120.0f));
        sp = fma2(sp, y2, pk(-2.0f / 6.0f, -2.0f / 6.0f));
        sp = fma2(sp, y2, pk(-2.0f, -2.0f));
        float s0, s1;
        upk(mul2(y, sp), s0, s1);                                     // -2 sinh(delta ln2 / 2)
        // far: 1 - e; near: e * (-2 sinh)
        const float o0 = fmaf(far0 ? -1.0f : s0, e0, far0 ? 1.0f : 0.0f);
        const float o1 = fmaf(far1 ? -1.0f : s1, e1, far1 ? 1.0f : 0.0f);
        R[p] = mul2(Q[p], pk(o0, o1));
    }
}
// The sum of a unit's 8 values held as four pairs, in a fixed order (the
// locate pass repeats it).
__device__ __forceinline__ float sum4p(const f2 *V)
{
    float lo, hi;
    upk(add2(add2(V[0], V[1]), add2(V[2], V[3])), lo, hi);
    return lo + hi;
}
// Sum each of 8 values over the 32 lanes (a transposed butterfly: 9 shuffles
// in place of 40); lane 4 v ends with the total of value v.
__device__ __forceinline__ float xpose8(const float *v, int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4], c[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        a[i] = (b4 ? v[4 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[4 + i], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        c[i] = (b3 ? a[2 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, b3 ? a[i] : a[2 + i], 8);
    float d = (b2 ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, b2 ? c[0] : c[1], 4);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}

// Sum each of NV (2 or 4) values over the 32 lanes, transposed: lane
// l * 32 / NV ends with the total of value l.
template <int NV>
__device__ __forceinline__ float xpose_sum(const float *v, int lane)
{
    static_assert(NV == 2 || NV == 4, "two or four values");
    float a;
    if constexpr (NV == 4) {
        const bool h4 = lane & 16;
        float a0 = h4 ? v[2] : v[0], a1 = h4 ? v[3] : v[1];
        const float s0 = h4 ? v[0] : v[2], s1 = h4 ? v[1] : v[3];
        a0 += __shfl_xor_sync(0xffffffffu, s0, 16);
        a1 += __shfl_xor_sync(0xffffffffu, s1, 16);
        const bool h3 = lane & 8;
        a = h3 ? a1 : a0;
        a += __shfl_xor_sync(0xffffffffu, h3 ? a0 : a1, 8);
#pragma unroll
        for (int o = 4; o; o >>= 1)
            a += __shfl_xor_sync(0xffffffffu, a, o);
    } else {
        const bool h4 = lane & 16;
        a = h4 ? v[1] : v[0];
        a += __shfl_xor_sync(0xffffffffu, h4 ? v[0] : v[1], 16);
#pragma unroll
        for (int o = 8; o; o >>= 1)
            a += __shfl_xor_sync(0xffffffffu, a, o);
    }
    return a;
}

// ---------------------------------------------------------------- residual coefficients
// The coefficients of the distribution sequence b samples at its end j, from
// the statistics t of its target row j and d of its draft row j (j < K).
__device__ __forceinline__ ResK res_coef(const RowsParams &P, const VrStat &t, const VrStat &d, int j)
{
    ResK k;
    k.Mt = t.m;
    k.c = P.c;
    k.dLhi = k.dLlo = 0.0f;
    if (j < P.K && P.probs) {
        // given probabilities: x_d c stands for log2 p(x) and dL = -(Mt + log2 St),
        // so that delta = log2(p St / q') as for logits
        int et;
        float ft;
        log2_split(DF{t.s_hi, t.s_lo}, et, ft);
        DF dl = two_sum(-t.m, -(float)et);
        dl = df_add(dl, DF{-ft, 0.0f});
        k.dLhi = dl.hi;
        k.dLlo = dl.lo;
    } else if (j < P.K) {
        // dL = (Md - Mt) + log2 Sd - log2 St as a float pair
        int et, ed;
        float ft, fd;
        log2_split(DF{t.s_hi, t.s_lo}, et, ft);
        log2_split(DF{d.s_hi, d.s_lo}, ed, fd);
        DF dl = two_sum(d.m, -t.m);
        dl = df_add(dl, DF{(float)(ed - et), 0.0f});
        dl = df_add(dl, DF{fd - ft, 0.0f});
        k.dLhi = dl.hi;
        k.dLlo = dl.lo;
    }
    return k;
}
// The same, loading the statistics (the draft row's only where it is used).
__device__ __forceinline__ ResK vr_coef(const RowsParams &P, int b, int j)
{
    const VrStat *st = P.stat + (size_t)b * (2 * P.K + 1);
    const VrStat t = ld_vrstat(st + j);
    const VrStat d = (j < P.K && !P.probs) ? ld_vrstat(st + P.K + 1 + j) : VrStat{};
    return res_coef(P, t, d, j);
}

// ---------------------------------------------------------------- 1b. row statistics from a bulk-copy stream
// The statistics and decisions of vr_stats for stochastic calls with aligned
// rows and draft logits, from one persistent launch (VS_CPS CTAs per SM).
// Rows are handed out position-major over every position from one counter,
// each cut into P.parts parts; a row whose sequence has ended before its
// position is skipped when its part is claimed, so the decisions of earlier
// positions are mostly known by then.  In each CTA:
//   - a producer thread claims parts and copies them in VS_STAGE-byte stages
//     (cp.async.bulk, completion on the stage's mbarrier) into a ring of
//     VS_NS stages, running ahead across parts;
//   - VS_NCW consumer warps reduce each stage from shared memory (the
//     per-token arithmetic of vr_stats), merge their partials at the end of
//     a part and hand the part's statistics over to
//   - an epilogue thread, which merges the parts of the row and decides the
//     position (vr_commit), so the consumers never wait on global memory.
// Every wait is bounded; one that runs out sets the timeout word, reported by
// vr_sample as ST_TIMEOUT.
constexpr int kMaxDevicesRows = 64;
constexpr int VS_NS = 4;          // stages in the ring
constexpr int VS_STAGE = 16384;   // bytes per stage
constexpr int VS_CPS = 3;         // CTAs per SM
constexpr int VS_NCW = 8;         // consumer warps
constexpr int VS_EPN = 4;         // epilogue slots
constexpr int VS_MB = 8;          // part-merge buffers (more than VS_NS)
constexpr int VR2_HALF = VS_STAGE / 2;   // bytes of each row in a residual stage
constexpr int VS_T = (VS_NCW + 2) * 32;
constexpr int VS_SMAX = 8;        // most parts per row of the stream

// A stage: type 0, tokens [tok0, tok0 + ntok) of the row of part `item`;
// type 1, a residual stage of sequence b's row pair j (target half, then draft
// half unless qonly) with its coefficients.
struct VsMeta {
    int item, tok0, ntok, last, dt;
    int type, b, j, qonly;
    float Mt, dLhi, dLlo;
};
struct VsEp {
    VrStat st;
    int item, dt, pad0, pad1;
};

// Bounded wait for the phase of parity `par` of one of the CTA's own
// barriers (its ring of copies and its hand-offs); sets the timeout word when
// it runs out.  The bound is the call's spin limit, but never below
// VS_RING_MIN polls, so a small limit cannot leave copies in flight when the
// CTA winds down: the waits on other CTAs (the end of every sequence, a
// posted job) are the ones a small limit exercises.
constexpr uint32_t VS_RING_MIN = 1u << 20;
__device__ __forceinline__ bool vs_wait(unsigned long long *bar, uint32_t par, uint32_t limit, uint32_t *tflag)
{
    limit = max(limit, VS_RING_MIN);
    for (uint32_t it = 0;; ++it) {
        if (mbar_test(bar, par))
            return true;
        if (it >= limit) {
            atomicExch(tflag, 1u);
            return false;
        }
        if (it > 16)
            __nanosleep(64);
    }
}

// Row r of the stream's order: positions 0..K-1 hold the target and draft rows
// of every sequence side by side, position K the B target rows.
__device__ __forceinline__ void vs_row(const RowsParams &P, int r, int &i, int &b, int &kind)
{
    if (P.probs) {
        // draft probabilities: the target rows alone, position-major
        i = r / P.B;
        b = r - i * P.B;
        kind = 0;
        return;
    }
    const int nk = 2 * P.B * P.K;
    if (r < nk) {
        i = r / (2 * P.B);
        const int rl = r - i * 2 * P.B;
        b = rl >> 1;
        kind = rl & 1;
    } else {
        i = P.K;
        b = r - nk;
        kind = 0;
    }
}

// A consumer thread's share of a stage of ntok tokens (its units of 8 tokens:
// g = tid, tid + CT, ...; float32 units are vectors g and g + CT of a group of
// 2 CT vectors): the terms 2^(x c - mc) are summed against the running
// reference mc and added to s in one step when the total is below 2^64 (no
// new maximum, NaN or +inf among them); otherwise the units go through
// acc_group one by one, which moves the reference and flags NaN / +inf.
template <class E, int CT>
__device__ __forceinline__ void vs_stage(const uint4 *p, int ntok, int tid, float c, float &mc, float &s, int &fl)
{
    const f2 cc = pk(c, c), nm = pk(-mc, -mc);
    f2 a0 = pk(0.0f, 0.0f), a1 = pk(0.0f, 0.0f);
    const uint4 ninf = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    if constexpr (E::ES == 2) {
        const int nv = ntok >> 3;   // whole units: ntok is a multiple of 8
#pragma unroll 4
        for (int g = tid; g < nv; g += CT) {
            const uint4 w = p[g];
            a0 = add2(a0, ex2x2(fma2(E::pair(w, 0), cc, nm)));
            a1 = add2(a1, ex2x2(fma2(E::pair(w, 1), cc, nm)));
            a0 = add2(a0, ex2x2(fma2(E::pair(w, 2), cc, nm)));
            a1 = add2(a1, ex2x2(fma2(E::pair(w, 3), cc, nm)));
        }
    } else {
        const int nv = ntok >> 2;
#pragma unroll 2
        for (int g = tid; g < nv; g += 2 * CT) {
            const uint4 w = p[g], w2 = g + CT < nv ? p[g + CT] : ninf;
            a0 = add2(a0, ex2x2(fma2(E::pair(w, 0), cc, nm)));
            a1 = add2(a1, ex2x2(fma2(E::pair(w, 1), cc, nm)));
            a0 = add2(a0, ex2x2(fma2(E::pair(w2, 0), cc, nm)));
            a1 = add2(a1, ex2x2(fma2(E::pair(w2, 1), cc, nm)));
        }
    }
    float l0, h0, l1, h1;
    upk(a0, l0, h0);
    upk(a1, l1, h1);
    const float t = (l0 + h0) + (l1 + h1);
    if (t < 18446744073709551616.0f) {
        s += t;
        return;
    }
    if constexpr (E::ES == 2) {
        const int nv = ntok >> 3;
        for (int g = tid; g < nv; g += CT) {
            Unit<E> u;
            u.a = p[g];
            f2 X[4];
            unit_pairs<E>(u, X);
            acc_group(X, c, mc, s, fl, VR_BAD);
        }
    } else {
        const int nv = ntok >> 2;
        for (int g = tid; g < nv; g += 2 * CT) {
            Unit<E> u;
            u.a = p[g];
            u.b = g + CT < nv ? p[g + CT] : ninf;
            f2 X[4];
            unit_pairs<E>(u, X);
            acc_group(X, c, mc, s, fl, VR_BAD);
        }
    }
}

__device__ __noinline__ void vs_commit(const RowsParams &P, int b, int i, int kind, int part, int dt, VrStat st)
{
    const int K = P.K;
    const size_t rt = (size_t)b * (2 * K + 1) + i, rd = (size_t)b * (2 * K + 1) + K + 1 + i;
    const int nrows = i < K && !P.probs ? 2 : 1;   // given probabilities: no draft row is streamed
    VrStat t = st, d{};
    if (P.parts > 1 || nrows > 1) {
        P.vpart[(kind ? rd : rt) * VR_SMAX + part] = st;
        if (vr_atom_add(P.pair + (size_t)b * (K + 1) + i, 1u) != (uint32_t)(nrows * P.parts - 1))
            return;
        t = merge_parts(P.vpart + rt * VR_SMAX, P.parts);
        if (nrows > 1)
            d = merge_parts(P.vpart + rd * VR_SMAX, P.parts);
    }
    P.stat[rt] = t;
    if (nrows > 1)
        P.stat[rd] = d;
    bool acc = false;
    const int code = vr_decide(P, b, i, dt, t, d, acc);
    const bool ends = code || (!acc && i < K);
    if (ends) {
        P.errc[(size_t)b * (K + 1) + i] = code;
        atomicOr(P.rej + b, 1u << i);
    }
    {
        // the word of decided (low half) and ending (high half) positions:
        // blind rows look at it, and with the residual pass in the stream the
        // update completing the sequence's end posts its residual job
        const unsigned long long bits = (1ull << i) | ((ends || i == K) ? (1ull << (32 + i)) : 0ull);
        const unsigned long long old = vr_atom_or64(P.dw + b, bits);
        if (P.fused && !vr_ended(old) && vr_ended(old | bits))
            vr_post_end(P, b, old | bits);
    }
}

// DM: the draft kind, fixed per instantiation so that each variant carries
// only its own stage types -- 0 draft logits, 1 given probabilities.
template <class E, int DM>
__global__ void __launch_bounds__(VS_T, VS_CPS) vr_stream(const __grid_constant__ RowsParams P)
{
    constexpr bool PROBS = DM == 1;
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(128) uint8_t vs_buf[];
    __shared__ unsigned long long full[VS_NS], empty[VS_NS], epf[VS_EPN], epe[VS_EPN], mg[VS_MB];
    __shared__ VsMeta meta[VS_NS];
    __shared__ VsEp ep[VS_EPN];
    __shared__ float rm[VS_MB][VS_NCW], rhi[VS_MB][VS_NCW], rlo[VS_MB][VS_NCW], rzd[VS_MB];
    __shared__ int rfl[VS_MB][VS_NCW];
    constexpr int STOK = VS_STAGE / E::ES;   // tokens per stage
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = P.K, V = P.V;
    const uint32_t lim = P.spin_limit;
    uint32_t *tflag = P.vctl + VC_TIMEOUT * VC_LINE;
    if (tid == 0) {
        for (int s = 0; s < VS_NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], VS_NCW);
        }
        for (int s = 0; s < VS_EPN; ++s) {
            mbar_init(&epf[s], 1);
            mbar_init(&epe[s], 1);
        }
        for (int s = 0; s < VS_MB; ++s)
            mbar_init(&mg[s], VS_NCW);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int nitems = P.B * (PROBS ? K + 1 : 2 * K + 1) * P.parts;

    if (warp == VS_NCW) {
        // ---- producer
        if (lane != 0)
            return;
        int st = 0;
        uint32_t ph = 0;
        bool ok = true;
        constexpr int RT = VR2_HALF / E::ES;   // tokens of each row in a residual stage
        // Work, in the order it is taken:
        //   1. with the residual pass (P.fused): residual chunks of sequences
        //      that have ended (the row pair was streamed recently, so part of
        //      it is still in L2);
        //   2. parts handed out position-major from one counter.
        // Without the residual pass the next part is claimed one ahead; with
        // it, a part is claimed only when it starts (a part held while
        // residual chunks go first would delay the decisions that post them).
        const bool dyn = P.fused != 0;
        const int nstatic = nitems;
        int item = dyn ? -1 : (int)atomicAdd(P.vctl + VC_CLAIM * VC_LINE, 1u);
        bool drained = false;
        uint32_t idle = 0;
        int pend = -1;      // a residual chunk number claimed ahead of its job
        bool stop = false;  // a wait on other CTAs gave up (ok: the ring is intact)
        // Stream part `part` of row r of the stream's order.
        auto stream_part = [&](int r, int part, int it) {
            int i, b, kind;
            vs_row(P, r, i, b, kind);
            const size_t ridx = (size_t)b * (2 * K + 1) + (kind ? K + 1 + i : i);
            const uint32_t m = (P.skip && i > 0) ? __ldcg(P.rej + b) : 0u;
            const int dt = i < K ? __ldg(P.tokens + (size_t)b * K + i) : -1;
            if (m & ((1u << i) - 1u)) {
                // a rejection (or error) decided at an earlier position makes this row unneeded
                if (part == 0)
                    P.stat[ridx] = VrStat{-F_INF, 0.0f, 0.0f, VR_SKIP, 0.0f, 0, 0, 0};
                return;
            }
            const uint8_t *row =
                kind ? static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + i) * (size_t)V * E::ES
                     : static_cast<const uint8_t *>(P.target) + ((size_t)b * (K + 1) + i) * (size_t)V * E::ES;
            const int t0 = part * P.span, t1 = min(V, t0 + P.span);
            // A row started before every earlier position of its sequence was
            // decided (and accepted) is read blind: before each stage the
            // producer looks again (the words loaded one stage ahead), and once
            // a rejection shows up the part is dropped -- its consumers get an
            // abort stage in place of the rest and post nothing.
            const uint32_t need = (1u << i) - 1u;
            bool blind = P.skip && i > 0 && ((uint32_t)__ldcg(P.dw + b) & need) != need;
            uint32_t rj = 0u, dd = 0u;
            for (int tok = t0; tok < t1; tok += STOK) {
                const int n = min(STOK, t1 - tok);
                if (blind) {
                    if (tok > t0) {
                        if (rj & need) {
                            if (!vs_wait(&empty[st], ph ^ 1u, lim, tflag)) {
                                ok = false;
                                break;
                            }
                            meta[st] = VsMeta{it, tok, 0, 1, dt, 2, 0, 0, 0, 0.0f, 0.0f, 0.0f};
                            mbar_arrive(&full[st]);
                            if (++st == VS_NS) {
                                st = 0;
                                ph ^= 1u;
                            }
                            break;
                        }
                        blind = (dd & need) != need;   // every earlier position decided: needed
                    }
                    rj = __ldcg(P.rej + b);
                    dd = (uint32_t)__ldcg(P.dw + b);
                }
                if (!vs_wait(&empty[st], ph ^ 1u, lim, tflag)) {
                    ok = false;
                    break;
                }
                meta[st] = VsMeta{it, tok, n, tok + STOK >= t1 ? 1 : 0, dt, 0, 0, 0, 0, 0.0f, 0.0f, 0.0f};
                mbar_arrive_tx(&full[st], (uint32_t)(n * E::ES));
                bulk_g2s(vs_buf + st * VS_STAGE, row + (size_t)tok * E::ES, (uint32_t)(n * E::ES), &full[st]);
                if (++st == VS_NS) {
                    st = 0;
                    ph ^= 1u;
                }
            }
        };
        // Take up a posted residual chunk, if there is one; true when it was
        // taken (streamed, or a wait gave up and ok is false).
        // Chunks are handed out by one counter (atomicAdd, no compare-and-swap
        // storms); a producer holds at most one number claimed ahead of the
        // posted jobs and takes it up once its job is posted.
        auto take_residual = [&]() -> bool {
            const uint32_t avail = ld_acq(P.vctl + VC_JOBS * VC_LINE) * (uint32_t)P.rnch;
            if (pend < 0 && (drained || __ldcg(P.vctl + VC_TICKETS * VC_LINE) < avail))
                pend = (int)atomicAdd(P.vctl + VC_TICKETS * VC_LINE, 1u);
            if (pend < 0 || (uint32_t)pend >= avail)
                return false;
            const int ticket = pend;
            pend = -1;
            const int e = ticket / P.rnch, ch = ticket - e * P.rnch;
            // the job was reserved before its chunks could be claimed: its
            // poster is writing it (a slot past the B a call can post means a
            // workspace that was not zeroed: give up without touching it)
            int b1 = 0;
            for (uint32_t it = 0; e < P.B && it <= lim; ++it) {
                b1 = ld_acq_s32(&P.jobs[e].b1);
                if (b1)
                    break;
                __nanosleep(32);
            }
            if (!b1) {
                // gave up on another CTA: stop claiming, wind down normally
                atomicExch(tflag, 1u);
                stop = true;
                return true;
            }
            const VrJob jb = P.jobs[e];
            const int b = b1 - 1, j = jb.j;
            const bool qonly = j == K;
            // tokens of each row per residual stage: half a stage of target
            // logits, or (given probabilities, 4 bytes each) a quarter
            const int rt = PROBS ? VR2_HALF / 4 : RT;
            const int des = PROBS ? 4 : E::ES;   // bytes of a draft element
            const uint8_t *trow =
                static_cast<const uint8_t *>(P.target) + ((size_t)b * (K + 1) + j) * (size_t)V * E::ES;
            const uint8_t *drow =
                qonly ? trow
                      : static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + j) * (size_t)V * des;
            for (int sg = 0; sg < P.rcs; ++sg) {
                const int tok0 = (ch * P.rcs + sg) * rt;
                if (tok0 >= V)
                    break;
                const int n = min(rt, V - tok0);
                if (!vs_wait(&empty[st], ph ^ 1u, lim, tflag)) {
                    ok = false;
                    break;
                }
                meta[st] = VsMeta{-2, tok0, n, 0, -1, 1, b, j, qonly ? 1 : 0, jb.Mt, jb.dLhi, jb.dLlo};
                const uint32_t nb = (uint32_t)(n * E::ES), nd = qonly ? 0u : (uint32_t)(n * des);
                mbar_arrive_tx(&full[st], nb + nd);
                bulk_g2s(vs_buf + st * VS_STAGE, trow + (size_t)tok0 * E::ES, nb, &full[st]);
                if (!qonly)
                    bulk_g2s(vs_buf + st * VS_STAGE + VR2_HALF, drow + (size_t)tok0 * des, nd, &full[st]);
                if (++st == VS_NS) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            return true;
        };
        while (ok) {
            if (P.fused && take_residual()) {
                if (stop)
                    break;
                idle = 0;
                continue;
            }
            if (dyn && !drained) {
                item = (int)atomicAdd(P.vctl + VC_CLAIM * VC_LINE, 1u);
                drained = item >= nstatic;
            }
            if (item >= nstatic || drained) {
                // no part left: with the residual pass, wait until every sequence
                // has ended and every posted chunk is claimed
                if (!dyn)
                    break;
                // every sequence ended: the jobs are final, and a number held
                // past them has no chunk
                if (ld_acq(P.vctl + VC_ENDED * VC_LINE) >= (uint32_t)P.B &&
                    (pend < 0 || (uint32_t)pend >= ld_acq(P.vctl + VC_JOBS * VC_LINE) * (uint32_t)P.rnch))
                    break;
                if (++idle > lim) {
                    // gave up on the other CTAs: stop claiming, wind down normally
                    atomicExch(tflag, 1u);
                    stop = true;
                    break;
                }
                __nanosleep(500);
                continue;
            }
            const int next = dyn ? nstatic : (int)atomicAdd(P.vctl + VC_CLAIM * VC_LINE, 1u);   // claimed ahead
            const int r = item / P.parts, part = item - r * P.parts;
            stream_part(r, part, item);
            item = next;
        }
        // end of the stream
        if (ok && vs_wait(&empty[st], ph ^ 1u, lim, tflag)) {
            meta[st] = VsMeta{-1, 0, 0, 0, -1, 0, 0, 0, 0, 0.0f, 0.0f, 0.0f};
            mbar_arrive(&full[st]);
        }
        return;
    }
    if (warp == VS_NCW + 1) {
        // ---- epilogue
        if (lane != 0)
            return;
        int es = 0;
        uint32_t eph = 0;
        while (vs_wait(&epf[es], eph, lim, tflag)) {
            const VsEp e = ep[es];
            mbar_arrive(&epe[es]);
            if (++es == VS_EPN) {
                es = 0;
                eph ^= 1u;
            }
            if (e.item < 0)
                break;
            const int r = e.item / P.parts, part = e.item - r * P.parts;
            int i, b, kind;
            vs_row(P, r, i, b, kind);
            vs_commit(P, b, i, kind, part, e.dt, e.st);
        }
        return;
    }
    // ---- consumers (threads 0 .. 32 VS_NCW - 1)
    constexpr int CT = VS_NCW * 32;
    const float c = P.c;
    int st = 0, nit = 0;
    uint32_t ph = 0;
    float mc = -F_INF, s = 0.0f, zd = 0.0f;
    int fl = 0;
    bool ok = true;
    for (;;) {
        if (lane == 0)
            ok = vs_wait(&full[st], ph, lim, tflag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok)
            break;
        (void)mbar_test(&full[st], ph);   // every lane observes the completed phase
        const VsMeta mt = meta[st];
        if (mt.type == 0 && mt.item < 0)
            break;
        if (mt.type == 2) {
            // the producer dropped the rest of a part read blind: nothing is posted
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
            if (++st == VS_NS) {
                st = 0;
                ph ^= 1u;
            }
            mc = -F_INF;
            s = 0.0f;
            zd = 0.0f;
            fl = 0;
            continue;
        }
        const uint8_t *sb = vs_buf + st * VS_STAGE;
        if (mt.type == 1 && PROBS) {
            // a residual stage with given probabilities: 2048 tokens, one
            // 256-token segment per warp; x_d c = log2 p (lg2 of each
            // probability); a probability that is negative, NaN or +inf puts
            // the sequence in error (its position j was a rejection)
            const ResK k{mt.Mt, mt.dLhi, mt.dLlo, c};
            const float ic = 1.0f / c;
            const int x = warp * VSEG + lane * 8;   // token within the stage
            float v0 = 0.0f, v1 = 0.0f;
            bool bad = false;
            if (x < mt.ntok) {
                const uint4 *pt = reinterpret_cast<const uint4 *>(sb + (size_t)x * E::ES);
                Unit<E> ut;
                ut.a = pt[0];
                if constexpr (E::ES == 4) {
                    const uint4 ninf = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
                    ut.b = x + 8 <= mt.ntok ? pt[1] : ninf;
                }
                f2 XT[4], XD[4], R[4], Q[4];
                unit_pairs<E>(ut, XT);
                if (mt.qonly) {
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        XD[p] = XT[p];
                } else {
                    const float4 *pp = reinterpret_cast<const float4 *>(sb + VR2_HALF + (size_t)x * 4);
                    const float4 pa = pp[0], pb = x + 8 <= mt.ntok ? pp[1] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float a0 = pv[2 * p], a1 = pv[2 * p + 1];
                        bad |= !(a0 >= 0.0f) || a0 == F_INF || !(a1 >= 0.0f) || a1 == F_INF;
                        XD[p] = pk(lg2a(a0) * ic, lg2a(a1) * ic);
                    }
                }
                vr_res8(XT, XD, k, mt.qonly != 0, R, Q);
                v0 = sum4p(R);
                v1 = sum4p(Q);
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0)
                P.errc[(size_t)mt.b * (K + 1) + mt.j] = ST_NONFINITE;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
            if (++st == VS_NS) {
                st = 0;
                ph ^= 1u;
            }
            const float vv[2] = {v0, v1};
            const float tot = xpose_sum<2>(vv, lane);   // lane 0: r', lane 16: q'
            if ((lane & 15) == 0 && warp * VSEG < mt.ntok)
                reinterpret_cast<float *>(P.segm + (size_t)mt.b * P.nseg + mt.tok0 / VSEG + warp)[lane >> 4] = tot;
            continue;
        }
        if (mt.type == 1) {
            // a residual stage: the masses of its 256-token segments
            constexpr int SPW = VR2_HALF / E::ES / VSEG / VS_NCW;   // segments per warp
            static_assert(SPW * VSEG * VS_NCW * E::ES == VR2_HALF, "a stage is whole segments");
            const ResK k{mt.Mt, mt.dLhi, mt.dLlo, c};
            float v[2 * SPW];
#pragma unroll
            for (int q = 0; q < SPW; ++q) {
                const int x = (warp + q * VS_NCW) * VSEG + lane * 8;   // token within the stage
                v[2 * q] = v[2 * q + 1] = 0.0f;
                if (x < mt.ntok) {
                    const uint4 *pt = reinterpret_cast<const uint4 *>(sb + (size_t)x * E::ES);
                    const uint4 *pd = reinterpret_cast<const uint4 *>(sb + VR2_HALF + (size_t)x * E::ES);
                    Unit<E> ut, ud;
                    ut.a = pt[0];
                    ud.a = mt.qonly ? ut.a : pd[0];
                    if constexpr (E::ES == 4) {
                        const uint4 ninf = make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
                        const bool whole = x + 8 <= mt.ntok;   // else its last four tokens are past the row
                        ut.b = whole ? pt[1] : ninf;
                        ud.b = mt.qonly ? ut.b : (whole ? pd[1] : ninf);
                    }
                    f2 XT[4], XD[4], R[4], Q[4];
                    unit_pairs<E>(ut, XT);
                    unit_pairs<E>(ud, XD);
                    vr_res8(XT, XD, k, mt.qonly != 0, R, Q);
                    v[2 * q] = sum4p(R);
                    v[2 * q + 1] = sum4p(Q);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
            if (++st == VS_NS) {
                st = 0;
                ph ^= 1u;
            }
            // lane (2q + w) * 32 / (2 SPW) holds value w of segment q (w = 0: r', 1: q')
            const float tot = xpose_sum<2 * SPW>(v, lane);
            const int vi = lane / (32 / (2 * SPW));
            const int sl = warp + (vi >> 1) * VS_NCW;
            if (lane % (32 / (2 * SPW)) == 0 && sl * VSEG < mt.ntok)
                reinterpret_cast<float *>(P.segm + (size_t)mt.b * P.nseg + mt.tok0 / VSEG + sl)[vi & 1] = tot;
            continue;
        }
        const uint4 *p = reinterpret_cast<const uint4 *>(sb);
        vs_stage<E, CT>(p, mt.ntok, tid, c, mc, s, fl);
        if (tid == 0 && (unsigned)(mt.dt - mt.tok0) < (unsigned)mt.ntok) {
            const int o = mt.dt - mt.tok0;
            zd = E::ES == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(sb)[o] << 16)
                            : reinterpret_cast<const float *>(sb)[o];
            fl |= VR_HASD;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
        if (++st == VS_NS) {
            st = 0;
            ph ^= 1u;
        }
        if (mt.last) {
            // the part's statistics: each warp posts its partial (buffer nit mod
            // VS_MB, whose mbarrier completes once all consumer warps posted);
            // warp nit mod VS_NCW merges them and hands the result to the
            // epilogue (slot nit mod VS_EPN), so the merges are spread over the
            // warps.  No warp runs more than VS_NS stages, so VS_NS parts,
            // ahead of another: the buffers never overlap.
            const int h = nit & (VS_MB - 1);
            const int wf = warp_or(fl);
            float M;
            DF S;
            merge_ms<32>(mc, DF{s, 0.0f}, c, M, S);
            if (lane == 0) {
                rm[h][warp] = M;
                rhi[h][warp] = S.hi;
                rlo[h][warp] = S.lo;
                rfl[h][warp] = wf;
                if (fl & VR_HASD)
                    rzd[h] = zd;   // thread 0 alone ever holds the drafted token
                mbar_arrive(&mg[h]);
            }
            if (warp == nit % VS_NCW) {
                bool got = true;
                if (lane == 0)
                    got = vs_wait(&mg[h], (uint32_t)(nit / VS_MB) & 1u, lim, tflag);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (got) {
                    (void)mbar_test(&mg[h], (uint32_t)(nit / VS_MB) & 1u);
                    const bool in = lane < VS_NCW;
                    VrStat r{};
                    r.flags = warp_or(in ? rfl[h][lane] : 0);
                    r.zd = (r.flags & VR_HASD) ? rzd[h] : 0.0f;
                    merge_ms<VS_NCW>(in ? rm[h][lane] : -F_INF,
                                     in ? DF{rhi[h][lane], rlo[h][lane]} : DF{0.0f, 0.0f}, c, M, S);
                    r.m = M;
                    r.s_hi = S.hi;
                    r.s_lo = S.lo;
                    const int es = nit % VS_EPN;
                    if (lane == 0 && vs_wait(&epe[es], ((uint32_t)(nit / VS_EPN) & 1u) ^ 1u, lim, tflag)) {
                        ep[es] = VsEp{r, mt.item, mt.dt, 0, 0};
                        mbar_arrive(&epf[es]);
                    }
                }
                __syncwarp();
            }
            mc = -F_INF;
            s = 0.0f;
            zd = 0.0f;
            fl = 0;
            ++nit;
        }
    }
    if (tid == 0 && vs_wait(&epe[nit % VS_EPN], ((uint32_t)(nit / VS_EPN) & 1u) ^ 1u, lim, tflag)) {
        ep[nit % VS_EPN].item = -1;
        mbar_arrive(&epf[nit % VS_EPN]);
    }
}

// Sequence b has ended (word w): post its residual job -- the position j it
// ended at and the coefficients of row pair j -- unless it ended in error
// (vr_sample writes those outputs); then count it as ended.
__device__ __noinline__ void vr_post_end(const RowsParams &P, int b, unsigned long long w)
{
    const int K = P.K;
    const int j = __ffs((uint32_t)(w >> 32)) - 1;
    const int code = (__ldcg(P.rej + b) >> j) & 1u ? __ldcg(P.errc + (size_t)b * (K + 1) + j) : 0;
    if (!code) {
        const ResK k = vr_coef(P, b, j);
        const uint32_t e = vr_atom_add(P.vctl + VC_JOBS * VC_LINE, 1u);
        VrJob *jb = P.jobs + e;
        jb->j = j;
        jb->Mt = k.Mt;
        jb->dLhi = k.dLhi;
        jb->dLlo = k.dLlo;
        st_rel_s32(&jb->b1, b + 1);
    }
    vr_atom_add(P.vctl + VC_ENDED * VC_LINE, 1u);
}

// Draft logits of the 8 tokens [seg * VSEG + 8 lane, +8) from a shortlisted
// draft row (b, j): the segment's list entries (lb gives their range) are
// scattered into a per-warp buffer of VSEG floats; tokens off the list read
// -inf, i.e. p = 0.
template <class E>
// lo, hi: the segment's list range when known (lo >= 0), else loaded here;
// pidx >= 0: this lane's first entry (list index lo + lane) already loaded,
// with its draft value pval.
__device__ __forceinline__ void sl_pairs(const RowsParams &P, int b, int j, int seg, int lane, float *buf, f2 *XD,
                                         int lo = -1, int hi = -1, int pidx = -1, float pval = 0.0f)
{
#pragma unroll
    for (int e = 0; e < 8; ++e)
        buf[lane * 8 + e] = -F_INF;
    __syncwarp();
    if (seg < P.nseg) {
        const int32_t *lb = P.lb + ((size_t)b * P.K + j) * (P.nseg + 1);
        const int32_t *lst = P.sl + b * P.sl_seq + j * P.sl_pos;
        const void *drow = static_cast<const uint8_t *>(P.draft) + ((size_t)b * P.K + j) * (size_t)P.S * E::ES;
        if (lo < 0) {
            lo = __ldcg(lb + seg);
            hi = __ldcg(lb + seg + 1);
        }
        int si0 = lo + lane;
        if (pidx >= 0) {
            const int pos = pidx - seg * VSEG;
            if ((unsigned)pos < (unsigned)VSEG)
                buf[pos] = pval;
            si0 += 32;
        }
        for (int si = si0; si < hi; si += 32) {
            const int pos = __ldg(lst + si) - seg * VSEG;
            if ((unsigned)pos < (unsigned)VSEG)
                buf[pos] = E::load(drow, (size_t)si);
        }
    }
    __syncwarp();
    float x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        x[e] = buf[lane * 8 + e];
    __syncwarp();
#pragma unroll
    for (int p = 0; p < 4; ++p)
        XD[p] = pk(x[2 * p], x[2 * p + 1]);
}

// SLR: the call has a shortlisted draft (its list code is compiled only then).
template <class E, bool SLR>
__global__ void __launch_bounds__(VRT, E::ES == 2 ? 3 : 1) vr_residual(const __grid_constant__ RowsParams P)
{
    pdl_wait();
    pdl_trigger();
    constexpr int NW = VRT / 32;
    constexpr int UPS = VSEG / 8;   // units per segment (one per lane)
    __shared__ int sm_j, sm_code;
    __shared__ float sl_buf[NW][VSEG];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / P.nch, ch = blockIdx.x % P.nch;
    const int K = P.K, V = P.V;
    if (tid == 0) {
        int j = 0;
        sm_code = vr_end(P, b, j);
        sm_j = j;
    }
    __syncthreads();
    if (sm_code)
        return;
    const int j = sm_j;
    const bool qonly = j == K;
    const bool slist = SLR && !qonly;   // draft values come from the shortlist
    const ResK k = vr_coef(P, b, j);
    const uint8_t *trow = static_cast<const uint8_t *>(P.target) + ((size_t)b * (K + 1) + j) * (size_t)V * E::ES;
    const uint8_t *drow =
        (qonly || slist) ? trow : static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + j) * (size_t)V * E::ES;
    // this chunk's segments [s_lo, s_hi); at step t warp w takes segment
    // s_lo + t * NW + w, lane l its unit l (tokens seg * VSEG + 8 l ..)
    const int spc = (P.nseg + P.nch - 1) / P.nch;
    const int s_lo = ch * spc, s_hi = min(P.nseg, s_lo + spc);
    const int nsteps = (s_hi - s_lo + NW - 1) / NW;
    VrSeg *out = P.segm + (size_t)b * P.nseg;
    auto unit_x0 = [&](int t) { return ((s_lo + t * NW + warp) * UPS + lane) * 8; };
    // a shortlisted draft: the list ranges of this warp's segments, one load
    // per lane up front, when the warp has at most 32 steps
    const bool pre = slist && nsteps <= 32;
    int blo = -1, bhi = -1;
    if (pre && lane < nsteps) {
        const int sg = s_lo + lane * NW + warp;
        if (sg < P.nseg) {
            const int32_t *lbp = P.lb + ((size_t)b * K + j) * (P.nseg + 1);
            blo = __ldcg(lbp + sg);
            bhi = __ldcg(lbp + sg + 1);
        }
    }
    // four steps in flight; each buffer is refilled right after its use
    Unit<E> ut[4], ud[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q < nsteps) {
            ut[q] = fetch_unit<E>(trow, unit_x0(q), V, P.vec);
            if (!qonly && !slist)
                ud[q] = fetch_unit<E>(drow, unit_x0(q), V, P.vec);
        }
    for (int t0 = 0; t0 < nsteps; t0 += 4) {
        // a shortlisted draft: each lane's first list entry of the four steps,
        // loaded at once (one round trip for the group, not one per step)
        int pidx[4];
        float pval[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            pidx[q] = -1;
            pval[q] = 0.0f;
            if (pre) {
                const int t = t0 + q;
                const int lo = __shfl_sync(0xffffffffu, blo, t & 31), hi = __shfl_sync(0xffffffffu, bhi, t & 31);
                if (t < nsteps && lo + lane < hi) {
                    pidx[q] = __ldg(P.sl + b * P.sl_seq + j * P.sl_pos + lo + lane);
                    pval[q] = E::load(static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + j) * (size_t)P.S * E::ES,
                                      (size_t)(lo + lane));
                }
            }
        }
        // the (r', q') sums of four steps' units, reduced over the lanes at once
        float v[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int t = t0 + q;
            v[2 * q] = v[2 * q + 1] = 0.0f;
            if (t < nsteps) {
                f2 XT[4], XD[4];
                unit_pairs<E>(ut[q], XT);
                if (slist) {
                    // the segment's list range: loaded up front (lane t holds step t's)
                    const int lo = __shfl_sync(0xffffffffu, blo, t & 31), hi = __shfl_sync(0xffffffffu, bhi, t & 31);
                    sl_pairs<E>(P, b, j, s_lo + t * NW + warp, lane, sl_buf[warp], XD, pre ? lo : -1, hi,
                                pidx[q], pval[q]);
                } else if (!qonly) {
                    unit_pairs<E>(ud[q], XD);
                }
                if (t + 4 < nsteps) {
                    ut[q] = fetch_unit<E>(trow, unit_x0(t + 4), V, P.vec);
                    if (!qonly && !slist)
                        ud[q] = fetch_unit<E>(drow, unit_x0(t + 4), V, P.vec);
                }
                f2 R[4], Q[4];
                vr_res8(XT, XD, k, qonly, R, Q);
                v[2 * q] = sum4p(R);
                v[2 * q + 1] = sum4p(Q);
            }
        }
        const float tot = xpose8(v, lane);
        const int vi = lane >> 2;
        const int seg = s_lo + (t0 + (vi >> 1)) * NW + warp;
        if ((lane & 3) == 0 && t0 + (vi >> 1) < nsteps && seg < s_hi)
            reinterpret_cast<float *>(out + seg)[vi & 1] = tot;
    }
}

// ---------------------------------------------------------------- 2b. small calls, rows resident
// When every row of the call fits in the shared memory of the GPU's resident
// CTAs, one cooperative launch reads each row once and keeps it: CTA
// (b, i, part) copies part `part` of target row i and draft row i of sequence
// b (position K: the target row alone) into shared memory with cp.async.bulk,
// reduces both, and commits the part (rs_commit: the last part of a position
// to count merges both rows and decides it, and the decision word records
// decided and ending positions).  Every CTA then waits (bounded) for its
// sequence's end; the parts of the pair the sequence ended at form the
// residual masses of their 256-token segments from the rows still in shared
// memory, and the others leave.  vr_sample draws the token.  Nothing is read
// twice, and a call's latency is one copy, one commit chain and one pass over
// shared memory.
constexpr int VRS_T = 256;          // threads of a resident CTA (the slice reductions' block size)
constexpr int VRS_SMEM = 65536;     // a part of both rows of a position
static_assert(VRS_T == CL_THREADS, "thread_stats strides by CL_THREADS");

__device__ __forceinline__ unsigned long long ld_acq64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One part of one row in shared memory (n tokens) as a part record: reference,
// sum, flags, and the drafted token's logit when it lies in the part.
template <class E>
__device__ VrStat rs_part_stats(const uint8_t *base, int n, int t0, int dt, float c, float *sm_m, float *sm_hi,
                                float *sm_lo, int *sm_f, int tid)
{
    constexpr int NW = VRS_T / 32;
    const int lane = tid & 31, warp = tid >> 5;
    float mc, sc;
    int fl = 0;
    thread_stats<E>(base, n, tid, c, mc, sc, fl, VR_BAD);
    float M;
    DF S;
    merge_ms<32>(mc, DF{sc, 0.0f}, c, M, S);
    fl = warp_or(fl);
    if (lane == 0) {
        sm_m[warp] = M;
        sm_hi[warp] = S.hi;
        sm_lo[warp] = S.lo;
        sm_f[warp] = fl;
    }
    __syncthreads();
    VrStat r{};
    const bool in = lane < NW;
    merge_ms<NW>(in ? sm_m[lane] : -F_INF, in ? DF{sm_hi[lane], sm_lo[lane]} : DF{0.0f, 0.0f}, c, M, S);
    r.m = M;
    r.s_hi = S.hi;
    r.s_lo = S.lo;
    r.flags = warp_or(in ? sm_f[lane] : 0);
    if ((unsigned)(dt - t0) < (unsigned)n) {
        const int o = dt - t0;
        r.zd = E::ES == 2 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(base)[o] << 16)
                          : reinterpret_cast<const float *>(base)[o];
        r.flags |= VR_HASD;
    }
    __syncthreads();   // the shared partials are free again
    return r;
}

// Warp 0 of a resident CTA: records its part of the position's rows (st, and
// sd when the position has a draft row) and counts it, once per CTA; the last
// part to count merges every part of both rows in one round trip (lane h
// loads target part h, lane 8 + h draft part h; S <= 8), writes the rows'
// statistics, decides the position and records it in the decision word.
__device__ __noinline__ void rs_commit(const RowsParams &P, int b, int i, int part, int dt, VrStat st, VrStat sd,
                                       bool two, int lane)
{
    const int K = P.K, S = P.parts;
    const size_t rt = (size_t)b * (2 * K + 1) + i, rd = (size_t)b * (2 * K + 1) + K + 1 + i;
    uint32_t prev = 0;
    if (lane == 0) {
        P.vpart[rt * VR_SMAX + part] = st;
        if (two)
            P.vpart[rd * VR_SMAX + part] = sd;
        prev = vr_atom_add(P.pair + (size_t)b * (K + 1) + i, 1u);
    }
    if (__shfl_sync(0xffffffffu, prev, 0) != (uint32_t)(S - 1))
        return;
    __syncwarp();   // the other lanes read the records after lane 0's acquire
    const int h = lane & 7;
    const bool isd = lane >= 8;
    float m = -F_INF, z = 0.0f;
    DF sv{0.0f, 0.0f};
    int f = 0;
    if (lane < 16 && h < S && (!isd || two)) {
        const VrStat *pp = P.vpart + (isd ? rd : rt) * VR_SMAX + h;
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(pp));
        z = __ldcg(&pp->zd);
        m = a.x;
        sv = DF{a.y, a.z};
        f = __float_as_int(a.w);
    }
    float M;
    DF Sm;
    merge_ms<8>(m, sv, 1.0f, M, Sm);   // lanes 0-7: the target row, 8-15: the draft row
    int fo = f;
#pragma unroll
    for (int o = 4; o; o >>= 1)
        fo |= __shfl_xor_sync(0xffffffffu, fo, o);
    // the drafted token's logit, from the part holding it
    const uint32_t hd = __ballot_sync(0xffffffffu, (f & VR_HASD) != 0);
    const int srcT = __ffs(hd & 0xffu) - 1, srcD = __ffs(hd & 0xff00u) - 1;
    const float zT = __shfl_sync(0xffffffffu, z, srcT < 0 ? 0 : srcT);
    const float zD = __shfl_sync(0xffffffffu, z, srcD < 0 ? 8 : srcD);
    const float MD = __shfl_sync(0xffffffffu, M, 8), hD = __shfl_sync(0xffffffffu, Sm.hi, 8),
                lD = __shfl_sync(0xffffffffu, Sm.lo, 8);
    const int fD = __shfl_sync(0xffffffffu, fo, 8);
    if (lane != 0)
        return;
    const VrStat t{M, Sm.hi, Sm.lo, fo, srcT < 0 ? 0.0f : zT, 0, 0, 0};
    const VrStat d{MD, hD, lD, fD, srcD < 0 ? 0.0f : zD, 0, 0, 0};
    P.stat[rt] = t;
    if (two)
        P.stat[rd] = d;
    bool acc = false;
    const int code = vr_decide(P, b, i, dt, t, d, acc);
    const bool ends = code || (!acc && i < K);
    if (ends) {
        P.errc[(size_t)b * (K + 1) + i] = code;
        atomicOr(P.rej + b, 1u << i);
    }
    const unsigned long long bits = (1ull << i) | ((ends || i == K) ? (1ull << (32 + i)) : 0ull);
    (void)vr_atom_or64(P.dw + b, bits);
}

template <class E>
__global__ void __launch_bounds__(VRS_T) vr_resident(const __grid_constant__ RowsParams P)
{
    constexpr int NW = VRS_T / 32;
    extern __shared__ __align__(128) uint8_t rs_buf[];
    __shared__ unsigned long long bar;
    __shared__ float sm_m[NW], sm_hi[NW], sm_lo[NW];
    __shared__ int sm_f[NW], sm_j;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();   // vr_sample's CTAs may launch now and wait for this launch to finish
    const int K = P.K, V = P.V, S = P.parts;
    const int part = (int)blockIdx.x % S, pi = (int)blockIdx.x / S;
    const int b = pi / (K + 1), i = pi - b * (K + 1);
    const bool two = i < K;   // a position with a draft row
    const int t0 = part * P.span, n = min(P.span, V - t0);
    uint8_t *ts = rs_buf, *ds = rs_buf + (size_t)P.span * E::ES;
    if (tid == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const uint32_t nb = (uint32_t)n * E::ES;
        mbar_arrive_tx(&bar, two ? 2 * nb : nb);
        const uint8_t *tr =
            static_cast<const uint8_t *>(P.target) + (((size_t)b * (K + 1) + i) * (size_t)V + t0) * E::ES;
        const uint8_t *dr = two ? static_cast<const uint8_t *>(P.draft) + (((size_t)b * K + i) * (size_t)V + t0) * E::ES
                                : nullptr;
        for (uint32_t o = 0; o < nb; o += 16384u) {
            const uint32_t m = min(16384u, nb - o);
            bulk_g2s(ts + o, tr + o, m, &bar);
            if (two)
                bulk_g2s(ds + o, dr + o, m, &bar);
        }
    }
    const int dt = two ? __ldg(P.tokens + (size_t)b * K + i) : -1;
    __syncthreads();
    if (!__syncthreads_and(ring_wait(&bar, 0u, P.spin_limit))) {
        // the copies did not land in time: no commit (the call reports a
        // timeout); wait for them before leaving
        if (tid == 0) {
            atomicExch(P.vctl + VC_TIMEOUT * VC_LINE, 1u);
            (void)mbar_wait(&bar, 0u, DRAIN_LIMIT, nullptr);
        }
        return;
    }
    const VrStat st = rs_part_stats<E>(ts, n, t0, dt, P.c, sm_m, sm_hi, sm_lo, sm_f, tid);
    VrStat sd{};
    if (two)
        sd = rs_part_stats<E>(ds, n, t0, dt, P.c, sm_m, sm_hi, sm_lo, sm_f, tid);
    if (warp == 0)
        rs_commit(P, b, i, part, dt, st, sd, two, lane);
    if (tid == 0) {
        // the sequence's end: the first ending position, every position up to
        // it decided (bounded: giving up reports a timeout for the call)
        int j = -1;
        for (uint32_t it = 0; it <= P.spin_limit; ++it) {
            const unsigned long long w = ld_acq64(P.dw + b);
            if (vr_ended(w)) {
                j = __ffs((uint32_t)(w >> 32)) - 1;
                break;
            }
            if (it > 16)
                __nanosleep(64);
        }
        if (j < 0)
            atomicExch(P.vctl + VC_TIMEOUT * VC_LINE, 1u);
        else if (j == i && ((__ldcg(P.rej + b) >> j) & 1u) && __ldcg(P.errc + (size_t)b * (K + 1) + j))
            j = -1;   // ended in error: no residual
        sm_j = j;
    }
    __syncthreads();
    if (sm_j != i)
        return;
    // the residual masses (r', q') of this part's 256-token segments
    const VrStat tS = ld_vrstat(P.stat + (size_t)b * (2 * K + 1) + i);
    const VrStat dS = two ? ld_vrstat(P.stat + (size_t)b * (2 * K + 1) + K + 1 + i) : VrStat{};
    const ResK k = res_coef(P, tS, dS, i);
    const bool qonly = !two;
    const uint4 ninf = E::neg_inf();
    const int nsg = (n + VSEG - 1) / VSEG;
    VrSeg *sg = P.segm + (size_t)b * P.nseg + t0 / VSEG;
    for (int q = warp; q < nsg; q += NW) {
        const int x = q * VSEG + lane * 8;   // token within the part
        Unit<E> ut, ud;
        const uint4 *pt = reinterpret_cast<const uint4 *>(ts + (size_t)x * E::ES);
        const uint4 *pd = reinterpret_cast<const uint4 *>(ds + (size_t)x * E::ES);
        ut.a = x < n ? pt[0] : ninf;
        ud.a = qonly ? ut.a : (x < n ? pd[0] : ninf);
        if constexpr (E::ES == 4) {
            const bool whole = x + 8 <= n;   // else its last four tokens are past the part
            ut.b = whole ? pt[1] : ninf;
            ud.b = qonly ? ut.b : (whole ? pd[1] : ninf);
        }
        f2 XT[4], XD[4], R[4], Q[4];
        unit_pairs<E>(ut, XT);
        unit_pairs<E>(ud, XD);
        vr_res8(XT, XD, k, qonly, R, Q);
        const float r = warp_sumf(sum4p(R)), qm = warp_sumf(sum4p(Q));
        if (lane == 0)
            sg[q] = VrSeg{r, qm};
    }
}

// ---------------------------------------------------------------- 3. sampling and outputs

// DK: the draft kind, fixed per instantiation so that each variant carries
// only its own locate code -- 0 draft logits, 1 given probabilities, 2 a
// shortlisted draft.
template <class E, int DK>
__global__ void __launch_bounds__(VST) vr_sample(const __grid_constant__ RowsParams P)
{
    constexpr bool PROBS = DK == 1, SLIST = DK == 2;
    pdl_wait();
    pdl_trigger();
    constexpr int NW = VST / 32;
    __shared__ int sm_seg, sm_last[NW], sm_x, sm_e[32];
    __shared__ uint32_t sm_m, sm_tf;
    __shared__ float sl_buf0[VSEG];
    __shared__ DF sm_r[NW], sm_q[NW], sm_before;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int K = P.K, V = P.V;
    // where the sequence ended, in one round trip: the mask, every position's
    // status and the timeout word together (vr_end's reading of them)
    if (tid <= K)
        sm_e[tid] = __ldcg(P.errc + (size_t)b * (K + 1) + tid);
    if (tid == 0) {
        sm_m = __ldcg(P.rej + b);
        sm_tf = __ldcg(P.vctl + VC_TIMEOUT * VC_LINE);
    }
    // the segment masses of the pair the sequence ended at (the residual pass
    // wrote them; they do not depend on where it ended), in the same round
    // trip: a thread's segments stay in registers when there are at most PC
    const int nseg = P.nseg;
    const VrSeg *sg = P.segm + (size_t)b * nseg;
    const int per = (nseg + VST - 1) / VST;
    const int s0 = min(nseg, tid * per), s1 = min(nseg, s0 + per);
    constexpr int PC = 8;
    const bool cached = per <= PC;
    float2 cg[PC];
    if (cached) {
#pragma unroll
        for (int k = 0; k < PC; ++k)
            cg[k] = s0 + k < s1 ? __ldcg(reinterpret_cast<const float2 *>(sg + s0 + k)) : make_float2(0.0f, 0.0f);
    }
    __syncthreads();
    const uint32_t msk = sm_m;
    const int j = msk ? __ffs(msk) - 1 : K;
    const int code = sm_tf ? (int)ST_TIMEOUT : ((msk >> j) & 1u ? sm_e[j] : 0);   // timeout: the stream gave up a wait
    const VrStat *st = P.stat + (size_t)b * (2 * K + 1);
    // the accepted drafts, emitted in parallel at the end
    const int tokv = tid < j ? __ldg(P.tokens + (size_t)b * K + tid) : -1;

    // per-position outputs (every row was computed when they are asked for)
    if (P.aux_q || P.aux_p || P.aux_lse) {
        // log2 of the row's sum 2^(x c); whether the row is usable
        auto row_l2 = [&](const VrStat &s, bool &ok) {
            ok = !(s.flags & (VR_BAD | VR_SKIP | VR_SLBAD)) && s.m > -F_INF && s.s_hi > 0.0f;
            int e;
            float f;
            log2_split(DF{s.s_hi, s.s_lo}, e, f);
            return s.m + ((float)e + f);
        };
        const float nan = __int_as_float(0x7fc00000);
        for (int i = tid; i < 2 * K + 1; i += VST) {
            bool ok;
            const float l2 = row_l2(ld_vrstat(st + i), ok);
            if (P.aux_lse)   // given probabilities have no draft logits: NaN there
                P.aux_lse[(size_t)b * (2 * K + 1) + i] = ok && !(PROBS && i > K) ? l2 * 0.6931471805599453f : nan;
        }
        // q_i(d_i) and p_i(d_i) where both rows of the position (given
        // probabilities: the target row and p_i(d_i)) and the token are usable
        for (int i = tid; i < K; i += VST) {
            const VrStat t = ld_vrstat(st + i);
            bool okt, okd;
            const float lt = row_l2(t, okt);
            const int dt = __ldg(P.tokens + (size_t)b * K + i);
            float pv;
            if (PROBS) {
                pv = dt >= 0 && dt < V ? __ldg(static_cast<const float *>(P.draft) + ((size_t)b * K + i) * (size_t)V + dt)
                                       : nan;
                okd = pv >= 0.0f && pv != F_INF;
            } else {
                const VrStat d = ld_vrstat(st + K + 1 + i);
                const float ld = row_l2(d, okd);
                pv = ex2a(fmaf(d.zd, P.c, -ld));
            }
            const bool ok = okt && okd && dt >= 0 && dt < V;
            if (P.aux_q)
                P.aux_q[(size_t)b * K + i] = ok ? ex2a(fmaf(t.zd, P.c, -lt)) : nan;
            if (P.aux_p)
                P.aux_p[(size_t)b * K + i] = ok ? pv : nan;
        }
    }
    if (tid == 0)
        sm_x = -1;
    if (code) {
        if (tid <= K)
            P.out_tokens[(size_t)b * (K + 1) + tid] = -1;
        if (tid == 0) {
            P.out_len[b] = -code;
            if (P.aux_R)
                P.aux_R[b] = __int_as_float(0x7fc00000);
            if (P.aux_status)
                atomicCAS(P.aux_status, 0, code);
        }
    } else {
        // the statistics of row pair j, loaded now for the coefficients used at the end
        VrStat tS{}, dS{};
        if (warp == 0) {
            tS = ld_vrstat(st + j);
            if (j < K)
                dS = ld_vrstat(st + K + 1 + j);
        }
        // totals of the residual and target masses of row pair j
        DF ownr{0.0f, 0.0f}, ownq{0.0f, 0.0f};
        if (cached) {
#pragma unroll
            for (int k = 0; k < PC; ++k)
                if (s0 + k < s1) {
                    ownr = df_add(ownr, DF{cg[k].x, 0.0f});
                    ownq = df_add(ownq, DF{cg[k].y, 0.0f});
                }
        } else {
            for (int s = s0; s < s1; ++s) {
                const float2 g = __ldcg(reinterpret_cast<const float2 *>(sg + s));
                ownr = df_add(ownr, DF{g.x, 0.0f});
                ownq = df_add(ownq, DF{g.y, 0.0f});
            }
        }
        const DF ir = warp_incl_scan_df(ownr, lane), iq = warp_incl_scan_df(ownq, lane);
        if (lane == 31) {
            sm_r[warp] = ir;
            sm_q[warp] = iq;
        }
        if (tid == 0)
            sm_seg = -1;
        __syncthreads();
        DF tr{0.0f, 0.0f}, tq{0.0f, 0.0f}, pr{0.0f, 0.0f}, pq{0.0f, 0.0f};
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (w == warp) {
                pr = tr;
                pq = tq;
            }
            tr = df_add(tr, sm_r[w]);
            tq = df_add(tq, sm_q[w]);
        }
        // R <= 0 (q == p up to rounding): sample q_j itself
        const bool useq = j < K && !(tr.hi > 0.0f);
        const DF F = useq ? tq : tr;
        const DF winc = useq ? iq : ir;
        DF wexc{__shfl_up_sync(0xffffffffu, winc.hi, 1), __shfl_up_sync(0xffffffffu, winc.lo, 1)};
        if (lane == 0)
            wexc = DF{0.0f, 0.0f};
        const DF incl = df_add(useq ? pq : pr, winc), excl = df_add(useq ? pq : pr, wexc);
        const uint4 wd = philox10((uint32_t)j, (uint32_t)b, 0u, 0u, P.key0, P.key1);
        const DF thr = u24_scale(wd.y, F);   // v R
        if (df_gt(incl, thr) && !df_gt(excl, thr)) {
            DF G = excl;
            if (cached) {
                bool found = false;
#pragma unroll
                for (int k = 0; k < PC; ++k) {
                    const float m = useq ? cg[k].y : cg[k].x;
                    const DF nG = df_add(G, DF{m, 0.0f});
                    if (!found && s0 + k < s1 && df_gt(nG, thr) && m > 0.0f) {
                        sm_seg = s0 + k;
                        sm_before = G;
                        found = true;
                    }
                    G = nG;
                }
            } else {
                for (int s = s0; s < s1; ++s) {
                    const float2 g = __ldcg(reinterpret_cast<const float2 *>(sg + s));
                    const float m = useq ? g.y : g.x;
                    const DF nG = df_add(G, DF{m, 0.0f});
                    if (df_gt(nG, thr) && m > 0.0f) {
                        sm_seg = s;
                        sm_before = G;
                        break;
                    }
                    G = nG;
                }
            }
        }
        __syncthreads();
        if (sm_seg < 0) {
            // rounding left no crossing: the last segment with mass
            int last = -1;
            for (int s = tid; s < nseg; s += VST) {
                const float2 g = __ldcg(reinterpret_cast<const float2 *>(sg + s));
                if ((useq ? g.y : g.x) > 0.0f)
                    last = s;
            }
            last = warp_maxi(last);
            if (lane == 0)
                sm_last[warp] = last;
            __syncthreads();
        }
        if (warp == 0) {
            // the token inside the segment: lane l holds tokens [s*256 + 8l, +8)
            int seg = sm_seg, fb = 0;
            if (seg < 0) {
                seg = -1;
                for (int w = 0; w < NW; ++w)
                    seg = max(seg, sm_last[w]);
                fb = 1;
            }
            int x = -1;
            if (seg >= 0) {
                const ResK k = res_coef(P, tS, dS, j);
                const bool qonly = j == K || useq;
                const bool slist = SLIST && !qonly;
                const uint8_t *trow =
                    static_cast<const uint8_t *>(P.target) + ((size_t)b * (K + 1) + j) * (size_t)V * E::ES;
                const int x0 = seg * VSEG + lane * 8;
                const Unit<E> ut = fetch_unit<E>(trow, x0, V, P.vec);
                Unit<E> ud{};
                Unit<F32> up{};
                if (!qonly && PROBS)
                    up = fetch_unit<F32>(static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + j) * (size_t)V * 4,
                                         x0, V, P.vec);
                else if (!qonly && !slist)
                    ud = fetch_unit<E>(static_cast<const uint8_t *>(P.draft) +
                                           ((size_t)b * K + j) * (size_t)V * E::ES, x0, V, P.vec);
                f2 XT[4], XD[4];
                unit_pairs<E>(ut, XT);
                if (slist) {
                    sl_pairs<E>(P, b, j, seg, lane, sl_buf0, XD);
                } else if (!qonly && PROBS) {
                    // x_d c = log2 p, as in the residual pass
                    f2 PP[4];
                    unit_pairs<F32>(up, PP);
                    const float ic = 1.0f / P.c;
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        float a0, a1;
                        upk(PP[p], a0, a1);
                        XD[p] = pk(lg2a(a0) * ic, lg2a(a1) * ic);
                    }
                } else if (!qonly) {
                    unit_pairs<E>(ud, XD);
                }
                f2 R[4], Q[4];
                vr_res8(XT, XD, k, qonly, R, Q);
                float r[8];
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    upk(R[p], r[2 * p], r[2 * p + 1]);
                const float ls = sum4p(R);
                if (!fb) {
                    const DF rel = df_add(thr, DF{-sm_before.hi, -sm_before.lo});
                    const float t = rel.hi + rel.lo;
                    float in = ls;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float u = __shfl_up_sync(0xffffffffu, in, o);
                        if (lane >= o)
                            in += u;
                    }
                    float ex = __shfl_up_sync(0xffffffffu, in, 1);
                    if (lane == 0)
                        ex = 0.0f;
                    const unsigned bal = __ballot_sync(0xffffffffu, in > t && ls > 0.0f);
                    if (bal) {
                        const int L = __ffs(bal) - 1;
                        if (lane == L) {
                            float cum = ex;
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                cum += r[e];
                                if (x < 0 && cum > t && r[e] > 0.0f)
                                    x = x0 + e;
                            }
                        }
                        x = __shfl_sync(0xffffffffu, x, L);
                    }
                }
                if (x < 0) {
                    // the last token of the segment with a positive weight
                    int lk = -1;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (r[e] > 0.0f)
                            lk = x0 + e;
                    x = warp_maxi(lk);
                }
            }
            if (lane == 0) {
                sm_x = x;
                if (P.aux_R) {
                    // R of the distribution drawn from (for q_j itself: the residual's, about 0)
                    const DF Rr = useq ? tr : F;
                    P.aux_R[b] = (Rr.hi + Rr.lo) / (tS.s_hi + tS.s_lo);
                }
            }
        }
    }
    __syncthreads();
    if (!code) {
        // accepted drafts 0..j-1, then x at j, -1 after
        if (tid <= K)
            P.out_tokens[(size_t)b * (K + 1) + tid] = tid < j ? tokv : (tid == j ? sm_x : -1);
        if (tid == 0)
            P.out_len[b] = j;
    }
    // the sequence's control words, for the next call
    for (int i = tid; i <= K; i += VST)
        P.pair[(size_t)b * (K + 1) + i] = 0u;
    for (int i = tid; i < 2 * K + 1; i += VST)
        P.rowcnt[(size_t)b * (2 * K + 1) + i] = 0u;
    if (tid == 0) {
        P.rej[b] = 0u;
        P.dw[b] = 0ull;
        P.jobs[b].b1 = 0;   // job slots are taken in posting order: slot b is some sequence's
        // the last CTA zeroes the call's counters (every CTA read the timeout word first)
        if (vr_atom_add(P.vctl + VC_SDONE * VC_LINE, 1u) == gridDim.x - 1) {
#pragma unroll
            for (int w = 0; w < VC_N; ++w)
                P.vctl[w * VC_LINE] = 0u;
        }
    }
}

// vr_sample for the call's draft kind.
template <class E>
cudaError_t launch_sample(const RowsParams &P, cudaStream_t stream)
{
    if (P.probs)
        return launch_after(vr_sample<E, 1>, P.B, VST, 0, stream, P);
    if (P.sl)
        return launch_after(vr_sample<E, 2>, P.B, VST, 0, stream, P);
    return launch_after(vr_sample<E, 0>, P.B, VST, 0, stream, P);
}

// A vr_stats launch over `rows` rows: each row is cut into parts so that the
// launch brings about as many threads as the GPU holds (the bytes in flight
// grow with them), with parts of at least 4096 tokens.
constexpr int VST_T = 256;   // threads of a vr_stats CTA
template <class E>
cudaError_t launch_stats(RowsParams P, int pos, int npos, int sms, cudaStream_t stream)
{
    const int rpp = 2 * P.B;
    // position K has the target row alone (B rows): launch it as rpp rows, the
    // draft half returning at once, to keep one row mapping
    const int rows = rpp * npos;
    const long long want = (long long)sms * 2048;
    int S = (int)std::min<long long>(VR_SMAX, (want + (long long)rows * VST_T - 1) / ((long long)rows * VST_T));
    // parts of at most 32768 tokens whatever the count of rows: most rows of a
    // later launch may skip, and those that do not should not be one CTA's
    // (a part that skips costs a launch and one load)
    S = std::max(S, (P.V + 32767) / 32768);
    S = std::max(1, std::min(std::min(S, VR_SMAX), P.V / 4096));
    P.pos = pos;
    P.npos = npos;
    P.span = ((P.V + S - 1) / S + 7) / 8 * 8;
    P.parts = (P.V + P.span - 1) / P.span;
    // the first launch of a call waits for whatever came before it in full
    if (P.sl)
        return launch_after(vr_stats<E, VST_T, true>, rows * P.parts, VST_T, 0, stream, P);
    return launch_after(vr_stats<E, VST_T, false>, rows * P.parts, VST_T, 0, stream, P);
}

// Whether vr_stream serves the call: stochastic, draft logits, aligned rows.
bool use_stream(const RowsParams &P)
{
    if (const char *ev = std::getenv("SPECVERIFY_ROWS_STREAM"))
        if (std::atoi(ev) == 0)
            return false;
    return !P.sl && P.vec;
}

constexpr long long kFusedMinRows = 1024;
constexpr long long kFusedSmallRows = 256;   // below this (small calls routed here): fused as well

// Whether vr_stream runs the residual pass: SPECVERIFY_ROWS_FUSED=1 always,
// =0 never (vr_residual does), unset by the call's size (-1); for
// measurement and tests.
int fused_mode()
{
    const char *ev = std::getenv("SPECVERIFY_ROWS_FUSED");
    if (!ev || !*ev)
        return -1;
    return std::atoi(ev) != 0 ? 1 : 0;
}

// The persistent statistics launch: VS_CPS CTAs per SM; parts per row so that
// there are about two parts per CTA, each at least two stages long (the
// epilogue's round trips per part make finer parts slower).
template <class E>
cudaError_t launch_stream(RowsParams P, int sms, cudaStream_t stream)
{
    static bool attr_set[kMaxDevicesRows][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int dm = P.probs ? 1 : 0;
    auto kern = dm ? vr_stream<E, 1> : vr_stream<E, 0>;
    const int smem = VS_NS * VS_STAGE;
    if (dev < kMaxDevicesRows && !attr_set[dev][dm]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        attr_set[dev][dm] = true;
    }
    const int ncta = sms * VS_CPS;
    const long long rows = (long long)P.B * (2 * P.K + 1);
    constexpr int STOK = VS_STAGE / E::ES;
    // at most VS_SMAX parts: 16 parts per row (B = 64, K = 4, residual pass in
    // its own launch) ran every call into the bounded waits' limit; the cause
    // is not known, and more than 8 parts never measured faster
    int S = (int)std::min<long long>(VS_SMAX, (2LL * ncta + rows - 1) / rows);
    S = std::max(1, std::min(S, P.V / (2 * STOK)));
    if (const char *ev = std::getenv("SPECVERIFY_ROWS_PARTS"))
        S = std::max(1, std::min(VS_SMAX, std::atoi(ev)));
    P.span = ((P.V + S - 1) / S + 7) / 8 * 8;
    P.parts = (P.V + P.span - 1) / P.span;
    return launch_after(kern, ncta, VS_T, smem, stream, P);
}

// Resident small calls: the parts per row S and tokens per part (whole
// 256-token segments) for which a part of both rows of a position fits
// VRS_SMEM, and whether the launch of B (K+1) S CTAs is resident at once.
// Returns the dynamic shared memory per CTA, or 0 when the call does not fit.
template <class E>
int resident_geometry(int B, int K, int V, int &S, int &span)
{
    static bool attr_set[kMaxDevicesRows] = {};
    static int occ_dev[kMaxDevicesRows] = {};
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevicesRows ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (!attr_set[dev]) {
        int occ = 0;
        if (cudaFuncSetAttribute(vr_resident<E>, cudaFuncAttributeMaxDynamicSharedMemorySize, VRS_SMEM) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, vr_resident<E>, VRS_T, VRS_SMEM) != cudaSuccess)
            return 0;
        occ_dev[dev] = occ;
        attr_set[dev] = true;
    }
    S = (int)((2LL * V * E::ES + VRS_SMEM - 1) / VRS_SMEM);
    for (;; ++S) {
        span = ((V + S - 1) / S + VSEG - 1) / VSEG * VSEG;
        if (2LL * span * E::ES <= VRS_SMEM)
            break;
    }
    S = (V + span - 1) / span;
    if (S > VR_SMAX || (long long)B * (K + 1) * S > (long long)sms * occ_dev[dev])
        return 0;
    return (int)(2LL * span * E::ES);
}

// Whether the resident path serves the call (stochastic, draft logits,
// aligned rows; SPECVERIFY_ROWS_RESIDENT=0 or SPECVERIFY_ROWS_STREAM=0 turn it off).
bool resident_enabled()
{
    const char *r = std::getenv("SPECVERIFY_ROWS_RESIDENT");
    const char *st = std::getenv("SPECVERIFY_ROWS_STREAM");
    return !(r && std::atoi(r) == 0) && !(st && std::atoi(st) == 0);
}

template <class E>
cudaError_t launch_resident(RowsParams P, int S, int span, int smem, cudaStream_t stream)
{
    P.parts = S;
    P.span = span;
    P.fused = 2;   // decisions recorded in the decision word, no residual jobs
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(P.B * (P.K + 1) * S));
    cfg.blockDim = dim3(VRS_T);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: they wait on each other
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, vr_resident<E>, P);
    if (e == cudaSuccess)
        e = launch_sample<E>(P, stream);
    return e;
}

template <class E>
cudaError_t launch_rows_t(RowsParams P, cudaStream_t stream, int &launches)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    launches = 0;
    if (!P.sl && !P.probs && P.vec && resident_enabled()) {
        int S = 0, span = 0;
        const int smem = resident_geometry<E>(P.B, P.K, P.V, S, span);
        if (smem > 0) {
            launches = 2;
            return launch_resident<E>(P, S, span, smem, stream);
        }
    }
    if (P.probs && !use_stream(P))
        return cudaErrorNotSupported;   // given probabilities: the stream alone serves them
    if (use_stream(P)) {
        // the residual pass in the same launch, in chunks of four stages, for
        // calls of at least kFusedMinRows rows (measured: B = 256, K = 4 at
        // 122 us against 138 us with vr_residual; B = 64, K = 4 at 64.5 us
        // against 61.5 us) and for the small calls the dispatch sends here
        // (B = 1, K = 4: 39 us against 44 us; B = 8, K = 8: 56 against 57)
        const int fm = fused_mode();
        const long long nrows = (long long)P.B * (2 * P.K + 1);
        P.fused = fm == 1 || (fm < 0 && (nrows >= kFusedMinRows || nrows < kFusedSmallRows)) ? 1 : 0;
        const int RT = P.probs ? VR2_HALF / 4 : VR2_HALF / E::ES;   // tokens of a row per residual stage
        const int nst = (P.V + RT - 1) / RT;
        if (P.probs)
            P.fused = 1;   // the residual pass over given probabilities runs in the stream only
        P.rcs = 4;
        P.rnch = (nst + P.rcs - 1) / P.rcs;
        e = launch_stream<E>(P, sms, stream);
        launches += 1;
    } else {
        // positions 0 and 1 first, then the rest: the second launch sees every
        // decision of the first (most of what skipping saves), at the cost of
        // one launch boundary
        const int first = std::min(2, P.K + 1);
        e = launch_stats<E>(P, 0, first, sms, stream);
        launches += 1;
        if (e == cudaSuccess && first <= P.K) {
            e = launch_stats<E>(P, first, P.K + 1 - first, sms, stream);
            launches += 1;
        }
    }
    if (e != cudaSuccess)
        return e;
    if (!P.fused) {
        // a shortlisted draft's segments scatter their list entries, a round
        // trip per step: four times the CTAs per sequence, a quarter of the steps
        if (P.sl)
            P.nch = 4 * VR_NCH;
        e = P.sl ? launch_after(vr_residual<E, true>, P.B * P.nch, VRT, 0, stream, P)
                 : launch_after(vr_residual<E, false>, P.B * P.nch, VRT, 0, stream, P);
        launches += 1;
        if (e != cudaSuccess)
            return e;
    }
    e = launch_sample<E>(P, stream);
    launches += 1;
    return e;
}

}  // namespace

bool rows_resident_fits(int B, int K, int V, int tdt)
{
    if (!resident_enabled())
        return false;
    int S = 0, span = 0;
    return (tdt == 0 ? resident_geometry<F32>(B, K, V, S, span) : resident_geometry<BF16>(B, K, V, S, span)) > 0;
}
int rows_chunks() { return VR_NCH; }
int rows_segment_tokens() { return VSEG; }
cudaError_t launch_rows(const RowsParams &P, int tdt, cudaStream_t stream, int *launches)
{
    if (P.greedy)
        return launch_greedy_rows(P, tdt, stream, launches);
    int n = 0;
    if (P.aux_status) {
        cudaError_t e = cudaMemsetAsync(P.aux_status, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return e;
    }
    const cudaError_t e = tdt == 0 ? launch_rows_t<F32>(P, stream, n) : launch_rows_t<BF16>(P, stream, n);
    if (launches)
        *launches = n;
    return e;
}

}  // namespace sv
