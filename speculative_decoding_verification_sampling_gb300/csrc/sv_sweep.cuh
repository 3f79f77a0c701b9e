// sv_sweep.cuh -- verification as a bandwidth sweep over (position, sequence, part) items.
//
// The rule is the one of the other kernels (nextadmin.net lesson "Speculative
// Decoding", § Core algorithm steps 4-6; aiengineeringfromscratch.com lesson
// 25, § The exact rule and § Greedy case; q = target, p = draft).  This kernel
// organises the work to keep HBM busy.
//
// Work items.  Item (i, b, h) is part h of the row pair at position i of
// sequence b: tokens [h*span, (h+1)*span) of target row i and draft row i
// (target only for greedy and for i = K).  Items are handed out from a global
// counter in position-major order.  A persistent CTA streams its item through
// a ring of shared-memory stages (cp.async.bulk, full/empty mbarriers) and
// reduces it to one SwStat: the maximum and the sum of 2^(x c - mc) per row,
// or for greedy the maximum and its lowest index.  Items of a sequence that
// has already ended before position i are skipped without reading; items
// ahead of the decisions are read anyway, a guess that costs at most the one
// row pair after each rejection.
//
// Decisions.  The CTA that completes the last part of (b, i) merges the parts
// into the row pair's statistics and marks them ready.  Under b's lock, it
// then advances b's decision frontier: position f is decided as soon as its
// statistics are ready, left to right, so statistics computed ahead are used
// when the frontier reaches them.  A CTA that finds the lock taken leaves; the
// holder looks again after releasing it, so no ready position is missed.
//
// Sampling.  The CTA whose decision ends b (first rejection j, or the bonus
// at j = K) samples at once.  It streams row pair j again (recently read, so
// from L2) and keeps the residual mass of every (stage, warp) chunk in token
// order.  The chunk whose running sum crosses v*R is reloaded, and its warp
// locates the token (inverse CDF over the unnormalised residual).
//
// Every wait and lock is bounded.  A wait that runs out records
// SPEC_ERR_TIMEOUT, and the last CTA out gives every unfinished sequence that
// error, reports the status and zeroes the workspace control region.
#pragma once
#include "sv_cluster.cuh"

namespace sv {

constexpr int WWARPS = 8;                  // warps per CTA
constexpr int WTHREADS = WWARPS * 32;
constexpr int WRING = 6;                   // ring stages
constexpr int WSBH = 8192;                 // bytes of one row in a stage
constexpr int WMAXST = 64;                 // stages per row (the residual streams a whole row)

struct alignas(16) SwShared {
    DF wm[WMAXST][WWARPS];                 // residual mass per (stage, warp), token order
    Rec wr[WWARPS];                        // per-warp partials
    unsigned long long full[WRING], empty[WRING];
    int item_b, item_pos, item_h, item_skip;   // the claimed item (thread 0 -> CTA)
    int end_b, end_j;                      // a sequence this CTA must sample (-1: none)
    int abort;
};
constexpr uint32_t SW_HDR = (uint32_t)((sizeof(SwShared) + 127) & ~size_t(127));
constexpr uint32_t SW_SMEM = SW_HDR + WRING * 2 * WSBH;

__device__ __forceinline__ void sw_status(const SweepParams &P, int code)
{
    atomicCAS(&P.ctl[CTL_STATUS], 0u, (uint32_t)code);
}
__device__ __forceinline__ void sw_error(const SweepParams &P, int b, int code)
{
    for (int i = 0; i <= P.K; ++i)
        P.out_tokens[(size_t)b * (P.K + 1) + i] = -1;
    P.out_len[b] = -code;
    if (P.aux_R)
        P.aux_R[b] = __int_as_float(0x7fc00000);
    sw_status(P, code);
}
// Accepted drafts 0..j-1, then x at j, -1 after.
__device__ __forceinline__ void sw_emit(const SweepParams &P, int b, int j, int x)
{
    int32_t *out = P.out_tokens + (size_t)b * (P.K + 1);
    for (int i = 0; i < j; ++i)
        out[i] = __ldg(P.tokens + (size_t)b * P.K + i);
    out[j] = x;
    for (int i = j + 1; i <= P.K; ++i)
        out[i] = -1;
    P.out_len[b] = j;
}
// A SwStat written by another CTA (read through L2).
__device__ __forceinline__ SwStat ld_stat(const SwStat *p)
{
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const int4 z = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    return SwStat{a.x, a.y, a.z, a.w, __int_as_float(z.x), __int_as_float(z.y), z.z, z.w};
}
__device__ __forceinline__ uint32_t ld_acq(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Merge the S part statistics of (b, i) in part order (thread 0).
__device__ __forceinline__ SwStat merge_parts(const SweepParams &P, size_t bp)
{
    const SwStat *pp = P.part + bp * P.S;
    if (P.greedy) {
        float v = -F_INF;
        int ix = -1, fl = 0;
        for (int h = 0; h < P.S; ++h) {
            const SwStat q = ld_stat(pp + h);
            fl |= q.flags;
            argmax_merge(v, ix, q.mt, __float_as_int(q.st_hi));
        }
        return SwStat{v, __int_as_float(ix), 0.0f, 0.0f, 0.0f, 0.0f, fl, 0};
    }
    float Mt = -F_INF, Md = -F_INF;
    int fl = 0;
    for (int h = 0; h < P.S; ++h) {
        const SwStat q = ld_stat(pp + h);
        fl |= q.flags;
        Mt = fmaxf(Mt, q.mt);
        Md = fmaxf(Md, q.md);
    }
    DF St{0.0f, 0.0f}, Sd{0.0f, 0.0f};
    for (int h = 0; h < P.S; ++h) {
        const SwStat q = ld_stat(pp + h);
        if (q.mt > -F_INF)
            St = df_add(St, df_scale_pow2(DF{q.st_hi, q.st_lo}, q.mt - Mt));
        if (q.md > -F_INF)
            Sd = df_add(Sd, df_scale_pow2(DF{q.sd_hi, q.sd_lo}, q.md - Md));
    }
    return SwStat{Mt, St.hi, St.lo, Md, Sd.hi, Sd.lo, fl, 0};
}

// Decide position f of sequence b from its merged statistics (thread 0).
// Returns 0 and sets accept, or a status code.
template <class E>
__device__ __forceinline__ int sw_decide(const SweepParams &P, int b, int f, bool &accept)
{
    const int K = P.K, V = P.V;
    const size_t bp = (size_t)b * (K + 1) + f;
    const SwStat s = ld_stat(P.stat + bp);
    accept = false;
    const int d = f < K ? __ldg(P.tokens + (size_t)b * K + f) : -1;
    if (f < K && !(d >= 0 && d < V))
        return ST_TOKEN;
    if (P.greedy) {
        const int g = __float_as_int(s.st_hi);
        if ((s.flags & 1) || !(s.mt > -F_INF) || g < 0)
            return ST_NONFINITE;
        accept = f < K && g == d;
        return 0;
    }
    if ((s.flags & 1) || !(s.mt > -F_INF) || !(s.st_hi > 0.0f))
        return ST_NONFINITE;
    if (f == K)
        return 0;
    if ((s.flags & 2) || !(s.md > -F_INF) || !(s.sd_hi > 0.0f))
        return ST_NONFINITE;
    const float zt = E::load(P.target, bp * (size_t)V + d);
    const float zd = E::load(P.draft, ((size_t)b * K + f) * (size_t)V + d);
    int et, ed;
    float ft, fd;
    log2_split(DF{s.st_hi, s.st_lo}, et, ft);
    log2_split(DF{s.sd_hi, s.sd_lo}, ed, fd);
    // p(d) == 0 (or below the float64 range) accepts
    const float lp = zd * P.c - s.md - ((float)ed + fd);
    if (zd == -F_INF || lp < -1074.5f) {
        accept = true;
        return 0;
    }
    // log2(q(d) / p(d)) = (zt - zd) c - (Mt - Md) - (log2 St - log2 Sd)
    const float X = (zt - zd) * P.c - ((s.mt - s.md) + ((float)(et - ed) + (ft - fd)));
    const uint4 w = philox10((uint32_t)f, (uint32_t)b, 0u, 0u, P.key0, P.key1);
    const float u = ((float)(w.x >> 8) + 0.5f) * (1.0f / 16777216.0f);
    accept = X >= 0.0f || u < ex2a(X);
    return 0;
}

// Advance b's decisions as far as ready statistics allow (thread 0).  Returns
// the position b ended at when this call ended it by a rejection or a bonus
// (the caller samples), else -1.  Errors write their outputs here.
template <class E>
__device__ int sw_advance(const SweepParams &P, int b, bool &timeout)
{
    SwSeq *sq = P.seq + b;
    const int K = P.K;
    for (;;) {
        uint32_t it = 0;
        while (atomicCAS(&sq->lock, 0u, 1u) != 0u) {
            // another CTA is advancing b: it looks again after releasing the lock
            if (++it > 64)
                return -1;
            __nanosleep(32);
        }
        __threadfence();
        uint32_t f = ld_vol(&sq->front), e = ld_vol(&sq->end);
        int ended = -1;
        while (e == 0u && (int)f <= K && (ld_acq(P.cnt + (size_t)b * (K + 1) + f) & SW_READY)) {
            bool accept = false;
            const int code = sw_decide<E>(P, b, (int)f, accept);
            if (code) {
                e = 0x80000000u | (uint32_t)code;
                sw_error(P, b, code);
                __threadfence();
                st_vol(&sq->fin, 1u);
                break;
            }
            if (accept && (int)f < K) {
                ++f;
                continue;
            }
            e = 1u + f;
            ended = (int)f;
            if (P.greedy) {
                const SwStat s = ld_stat(P.stat + (size_t)b * (K + 1) + f);
                sw_emit(P, b, (int)f, __float_as_int(s.st_hi));
                if (P.aux_R)
                    P.aux_R[b] = __int_as_float(0x7fc00000);
                __threadfence();
                st_vol(&sq->fin, 1u);
                ended = -1;
            }
            break;
        }
        st_vol(&sq->front, f);
        st_vol(&sq->end, e);
        __threadfence();
        atomicExch(&sq->lock, 0u);
        if (ended >= 0 || e != 0u)
            return ended;
        // statistics that became ready while the lock was held
        __threadfence();
        if ((int)f > K || !(ld_acq(P.cnt + (size_t)b * (K + 1) + f) & SW_READY))
            return -1;
        (void)timeout;
    }
}

template <class E>
__global__ void __launch_bounds__(WTHREADS, 2) sweep_kernel(const __grid_constant__ SweepParams P)
{
    extern __shared__ __align__(1024) uint8_t sw_smem[];
    SwShared &S = *reinterpret_cast<SwShared *>(sw_smem);
    uint8_t *ring = sw_smem + SW_HDR;
    constexpr int ST = WSBH / E::ES;           // tokens per stage
    constexpr int GPS = ST / 8;                // groups per stage
    constexpr int GW = GPS / WWARPS;           // groups per warp per stage
    constexpr int JL = GW / 32;                // groups per lane per stage
    static_assert(JL >= 1 && GW % 32 == 0, "stage geometry");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = P.K, V = P.V;
    const float c = P.c;

    if (tid == 0) {
        for (int i = 0; i < WRING; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], WWARPS);
        }
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    uint32_t kg = 0;      // stages consumed (the same in every thread)
    uint32_t kis = 0;     // stages issued (thread 0)

    // Thread 0: copy tokens [t0 + i*ST, ...) of the rows into ring stage k once
    // the warps have released it.
    auto issue = [&](uint32_t k, int t0, int nt, int i, const uint8_t *trow, const uint8_t *drow) -> bool {
        const uint32_t slot = k % WRING, use = k / WRING;
        if (use > 0 && !ring_wait(&S.empty[slot], (use - 1) & 1u, P.spin_limit))
            return false;
        const int cnt = min(ST, nt - i * ST);
        const uint32_t bytes = (uint32_t)cnt * E::ES;
        uint8_t *dst = ring + slot * 2 * WSBH;
        mbar_arrive_tx(&S.full[slot], drow ? 2u * bytes : bytes);
        bulk_g2s(dst, trow + (size_t)(t0 + i * ST) * E::ES, bytes, &S.full[slot]);
        if (drow)
            bulk_g2s(dst + WSBH, drow + (size_t)(t0 + i * ST) * E::ES, bytes, &S.full[slot]);
        kis = k + 1;
        return true;
    };
    // Stream tokens [t0, t0 + nt) of the rows through the ring; body(i, tb, db,
    // cnt) reduces stage i in every warp.  Returns false in every thread when a
    // wait ran out.
    auto pass = [&](int t0, int nt, const uint8_t *trow, const uint8_t *drow, auto &&body) -> bool {
        const int nst = (nt + ST - 1) / ST;
        bool ok = true;
        const uint32_t kb = kg;
        if (tid == 0)
            for (int i = 0; i < min(WRING, nst); ++i)
                ok = ok && issue(kb + i, t0, nt, i, trow, drow);
        for (int i = 0; i < nst; ++i) {
            const uint32_t k = kb + i, slot = k % WRING;
            const bool got = ok && ring_wait_warp(&S.full[slot], (k / WRING) & 1u, P.spin_limit, lane);
            if (got)
                body(i, ring + slot * 2 * WSBH, ring + slot * 2 * WSBH + WSBH, min(ST, nt - i * ST));
            ok = ok && got;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[slot]);
            if (tid == 0 && ok && i + WRING < nst)
                ok = issue(kb + i + WRING, t0, nt, i + WRING, trow, drow);
        }
        kg = kb + nst;
        return __syncthreads_and(ok);
    };

    for (;;) {
        // ---- claim an item
        if (tid == 0) {
            const uint32_t idx = atomicAdd(&P.ctl[CTL_STATS_NEXT], 1u);
            int b = -1, pos = 0, h = 0, skip = 0;
            if (idx < P.n_items && !ld_vol(&P.ctl[CTL_CL_ABORT])) {
                pos = (int)(idx / ((uint32_t)P.B * P.S));
                const uint32_t r = idx % ((uint32_t)P.B * P.S);
                b = (int)(r / P.S);
                h = (int)(r % P.S);
                // a sequence that ended before pos needs nothing more
                const uint32_t e = ld_vol(&P.seq[b].end);
                skip = e != 0u && ((e & 0x80000000u) || (int)(e - 1u) < pos);
            }
            S.item_b = b;
            S.item_pos = pos;
            S.item_h = h;
            S.item_skip = skip;
            S.end_b = -1;
        }
        __syncthreads();
        const int b = S.item_b, pos = S.item_pos, h = S.item_h;
        if (b < 0)
            break;
        if (S.item_skip) {
            __syncthreads();
            continue;
        }
        const size_t bp = (size_t)b * (K + 1) + pos;
        const int t0 = min(V, h * P.span), nt = min(P.span, V - t0);
        const uint8_t *trow = static_cast<const uint8_t *>(P.target) + bp * (size_t)V * E::ES;
        const uint8_t *drow = (!P.greedy && pos < K)
                                  ? static_cast<const uint8_t *>(P.draft) + ((size_t)b * K + pos) * (size_t)V * E::ES
                                  : nullptr;

        // ---- reduce the part
        bool ok;
        SwStat mine{};
        if (P.greedy) {
            float bv = -F_INF;
            int bi = -1, fl = 0;
            ok = pass(t0, nt, trow, nullptr, [&](int i, const uint8_t *tb, const uint8_t *, int cnt) {
#pragma unroll
                for (int jl = 0; jl < JL; ++jl) {
                    const int g = warp * GW + jl * 32 + lane;
                    if (g * 8 < cnt) {
                        f2 X[4];
                        const float vm = group8<E>(tb, g, cnt, X);
                        if (!(vm == vm) || vm == F_INF) {
                            fl = 1;
                        } else if (vm > bv) {
                            float x[8];
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                upk(X[p], x[2 * p], x[2 * p + 1]);
                            int e = 7;
#pragma unroll
                            for (int q = 7; q >= 0; --q)
                                if (x[q] == vm)
                                    e = q;
                            bv = vm;
                            bi = t0 + i * ST + g * 8 + e;
                        }
                    }
                }
            });
            warp_merge_argmax(bv, bi);
            fl = warp_or(fl);
            if (lane == 0)
                S.wr[warp] = Rec{bv, __int_as_float(bi), 0.0f, fl, 0.0f, 0.0f, 0.0f, 0};
            __syncthreads();
            if (warp == 0) {
                const bool in = lane < WWARPS;
                const Rec r = S.wr[in ? lane : 0];
                float v = in ? r.a0 : -F_INF;
                int ix = in ? __float_as_int(r.a1) : -1;
                warp_merge_argmax<WWARPS>(v, ix);
                mine = SwStat{v, __int_as_float(ix), 0.0f, 0.0f, 0.0f, 0.0f, warp_or(in ? r.i0 : 0), 0};
            }
        } else {
            float mt = -F_INF, st = 0.0f, md = -F_INF, sd = 0.0f;
            int fl = 0;
            ok = pass(t0, nt, trow, drow, [&](int, const uint8_t *tb, const uint8_t *db, int cnt) {
                if (cnt == ST) {
#pragma unroll
                    for (int jl = 0; jl < JL; ++jl) {
                        const int g = warp * GW + jl * 32 + lane;
                        f2 X[4];
                        Grp<E>::pairs(tb, g, X);
                        acc_group(X, c, mt, st, fl, 1);
                        if (drow) {
                            Grp<E>::pairs(db, g, X);
                            acc_group(X, c, md, sd, fl, 2);
                        }
                    }
                } else {
#pragma unroll
                    for (int jl = 0; jl < JL; ++jl) {
                        const int g = warp * GW + jl * 32 + lane;
                        if (g * 8 < cnt) {
                            f2 X[4];
                            (void)group8<E>(tb, g, cnt, X);
                            acc_group(X, c, mt, st, fl, 1);
                            if (drow) {
                                (void)group8<E>(db, g, cnt, X);
                                acc_group(X, c, md, sd, fl, 2);
                            }
                        }
                    }
                }
            });
            float Mt, Md;
            DF St, Sd;
            merge_ms<32>(mt, DF{st, 0.0f}, c, Mt, St);
            merge_ms<32>(md, DF{sd, 0.0f}, c, Md, Sd);
            fl = warp_or(fl);
            if (lane == 0)
                S.wr[warp] = Rec{Mt, St.hi, St.lo, fl, Md, Sd.hi, Sd.lo, 0};
            __syncthreads();
            if (warp == 0) {
                const bool in = lane < WWARPS;
                const Rec r = S.wr[in ? lane : 0];
                merge_ms<WWARPS>(in ? r.a0 : -F_INF, in ? DF{r.a1, r.a2} : DF{0.0f, 0.0f}, c, Mt, St);
                merge_ms<WWARPS>(in ? r.b0 : -F_INF, in ? DF{r.b1, r.b2} : DF{0.0f, 0.0f}, c, Md, Sd);
                mine = SwStat{Mt, St.hi, St.lo, Md, Sd.hi, Sd.lo, warp_or(in ? r.i0 : 0), 0};
            }
        }

        // ---- publish the part; the last part merges and advances the decisions
        if (tid == 0) {
            if (!ok) {
                sw_status(P, ST_TIMEOUT);
                atomicExch(&P.ctl[CTL_CL_ABORT], 1u);
                S.abort = 1;
            } else {
                P.part[bp * P.S + h] = mine;
                __threadfence();
                const uint32_t done = atomicAdd(P.cnt + bp, 1u) + 1u;
                if (done == (uint32_t)P.S) {
                    __threadfence();
                    P.stat[bp] = merge_parts(P, bp);
                    __threadfence();
                    atomicOr(P.cnt + bp, SW_READY);
                    bool to = false;
                    const int j = sw_advance<E>(P, b, to);
                    if (j >= 0) {
                        S.end_b = b;
                        S.end_j = j;
                    }
                }
            }
        }
        __syncthreads();
        if (S.abort)
            break;
        if (S.end_b < 0 || P.greedy)
            continue;

        // ---- sample the sequence this CTA ended (rejection at j, or the bonus at j = K)
        const int eb = S.end_b, j = S.end_j;
        const bool bonus = j == K;
        const size_t ebp = (size_t)eb * (K + 1) + j;
        const SwStat s = ld_stat(P.stat + ebp);
        const uint8_t *jt = static_cast<const uint8_t *>(P.target) + ebp * (size_t)V * E::ES;
        const uint8_t *jd =
            bonus ? nullptr : static_cast<const uint8_t *>(P.draft) + ((size_t)eb * K + j) * (size_t)V * E::ES;
        int et, ed;
        float ft, fd;
        log2_split(DF{s.st_hi, s.st_lo}, et, ft);
        ResK kc;
        kc.Mt = s.mt;
        kc.c = c;
        if (bonus) {
            kc.dLhi = kc.dLlo = 0.0f;
        } else {
            // dL = (Md - Mt) + log2 Sd - log2 St as a float pair
            log2_split(DF{s.sd_hi, s.sd_lo}, ed, fd);
            DF dl = two_sum(s.md, -s.mt);
            dl = df_add(dl, DF{(float)(ed - et), 0.0f});
            dl = df_add(dl, DF{fd - ft, 0.0f});
            kc.dLhi = dl.hi;
            kc.dLlo = dl.lo;
        }
        const uint4 wph = philox10((uint32_t)j, (uint32_t)eb, 0u, 0u, P.key0, P.key1);
        const float v = ((float)(wph.y >> 8) + 0.5f) * (1.0f / 16777216.0f);
        const int nst = (V + ST - 1) / ST;
        DF Rres{0.0f, 0.0f};
        bool useq = bonus, sampled = false, failed = false;
        for (int attempt = 0; attempt < 2 && !sampled && !failed; ++attempt) {
            const bool two = !(bonus || useq);
            const bool ok2 = pass(0, V, jt, two ? jd : nullptr, [&](int i, const uint8_t *tb, const uint8_t *db, int cnt) {
                const int ng = (cnt + 7) >> 3;
                const int g0 = min(ng, warp * GW), g1 = min(ng, g0 + GW);
                const DF W = warp_mass<E>(tb, db, cnt, g0, g1, kc, bonus, useq, lane);
                if (lane == 0)
                    S.wm[i][warp] = W;
            });
            if (!ok2) {
                failed = true;
                break;
            }
            // the total, and the (stage, warp) chunk whose running sum crosses t = v R
            DF F{0.0f, 0.0f};
            for (int i = 0; i < nst; ++i)
                for (int w = 0; w < WWARPS; ++w)
                    F = df_add(F, S.wm[i][w]);
            if (!useq || bonus)
                Rres = F;   // residual mass (kept when it is 0), or the total of q for a bonus
            if (!(F.hi > 0.0f)) {
                if (useq)
                    break;   // cannot happen for a finite row
                useq = true; // R <= 0: sample q_j itself
                continue;
            }
            const float th = v * F.hi;
            const DF t = df_add(DF{th, fmaf(v, F.hi, -th)}, DF{v * F.lo, 0.0f});
            int istar = -1, wstar = 0, ilast = -1, wlast = 0;
            DF G{0.0f, 0.0f}, Gc{0.0f, 0.0f}, Glast{0.0f, 0.0f};
            for (int i = 0; i < nst; ++i)
                for (int w = 0; w < WWARPS; ++w) {
                    const DF Wi = S.wm[i][w];
                    const DF nG = df_add(G, Wi);
                    if (Wi.hi > 0.0f) {
                        ilast = i;
                        wlast = w;
                        Glast = G;
                    }
                    if (istar < 0 && df_gt(nG, t)) {
                        istar = i;
                        wstar = w;
                        Gc = G;
                    }
                    G = nG;
                }
            const bool cfb = istar < 0;
            if (cfb) {
                istar = ilast;
                wstar = wlast;
                Gc = Glast;
            }
            if (istar >= 0 && warp == wstar) {
                // reload the chunk into ring stage 0 (the ring is idle) and locate in it
                const int cnt = min(ST, V - istar * ST);
                const int ng = (cnt + 7) >> 3;
                const int g0 = min(ng, wstar * GW), g1 = min(ng, g0 + GW);
                uint8_t *tb = ring, *db = ring + WSBH;
                constexpr int TPV = 16 / E::ES;   // tokens per 16-byte vector
                const size_t off = (size_t)istar * ST * E::ES;
                for (int g = g0 + lane; g < g1; g += 32) {
                    for (int hv = 0; hv < E::ES / 2; ++hv) {
                        if (g * 8 + hv * TPV >= cnt)   // vectors past the row are not read
                            break;
                        const size_t o = (size_t)g * 16 * (E::ES / 2) + (size_t)hv * 16;
                        *reinterpret_cast<uint4 *>(tb + o) = __ldcg(reinterpret_cast<const uint4 *>(jt + off + o));
                        if (two)
                            *reinterpret_cast<uint4 *>(db + o) = __ldcg(reinterpret_cast<const uint4 *>(jd + off + o));
                    }
                }
                // these generic stores precede later bulk copies into the same stage
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                const int xb = istar * ST;
                int xx = -1;
                if (!cfb)
                    xx = warp_locate<E>(tb, db, cnt, g0, g1, kc, bonus, useq, Gc, t, xb, lane);
                if (xx < 0)
                    xx = warp_last_positive<E>(tb, db, cnt, g0, g1, kc, bonus, useq, xb, lane);
                if (lane == 0) {
                    sw_emit(P, eb, j, xx);
                    if (P.aux_R)
                        P.aux_R[eb] = (Rres.hi + Rres.lo) / (s.st_hi + s.st_lo);
                    __threadfence();
                    st_vol(&P.seq[eb].fin, 1u);
                }
            }
            sampled = true;
        }
        if (failed && tid == 0) {
            sw_status(P, ST_TIMEOUT);
            atomicExch(&P.ctl[CTL_CL_ABORT], 1u);
            S.abort = 1;
        }
        __syncthreads();   // ring stage 0 is free again
        if (S.abort)
            break;
    }

    // ---- wind down: our own copies (only the last WRING issued can be in flight)
    if (tid == 0)
        for (uint32_t k = kis >= (uint32_t)WRING ? kis - WRING : 0u; k < kis; ++k)
            (void)mbar_wait(&S.full[k % WRING], (k / WRING) & 1u, DRAIN_LIMIT, nullptr);
    __syncthreads();
    __shared__ int last;
    if (tid == 0) {
        __threadfence();
        last = atomicAdd(&P.ctl[CTL_EXIT], 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    // sequences left without outputs (only after a wait ran out)
    for (int bb = tid; bb < P.B; bb += WTHREADS)
        if (ld_vol(&P.seq[bb].fin) == 0u)
            sw_error(P, bb, ST_TIMEOUT);
    __syncthreads();
    if (tid == 0 && P.aux_status)
        P.aux_status[0] = (int32_t)ld_vol(&P.ctl[CTL_STATUS]);
    __syncthreads();
    for (uint32_t i = tid; i < P.reset_words; i += WTHREADS)
        P.ctl[i] = 0u;
}

}  // namespace sv
