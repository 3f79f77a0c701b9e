// sv_sweep.cuh -- verification as a continuous bandwidth sweep.
//
// The rule is the one of the other kernels (nextadmin.net lesson "Speculative
// Decoding", § Core algorithm steps 4-6; aiengineeringfromscratch.com lesson
// 25, § The exact rule and § Greedy case; q = target, p = draft).  This kernel
// organises the work so that HBM never waits for a decision.
//
// Work items, and who takes them.
//   stats item (i, b, h):  part h of the row pair at position i of sequence b:
//                          tokens [h*span, (h+1)*span) of target row i and draft
//                          row i (the target alone for greedy and for i = K).
//                          Handed out from a global counter in position-major
//                          order; skipped without reading when b has already
//                          ended before i.
//   residual part (e, h):  part h of the row pair a sampling job e names
//                          (posted by the CTA whose decision ended a sequence).
//                          Residual parts are taken before new stats items.
//
// Warp roles.  Each CTA has one producer warp, eight consumer warps and one
// epilogue warp.
//   - The producer claims items and writes their descriptors into a small ring
//     of item slots.  It issues their stages (ST tokens of each row, by
//     cp.async.bulk) into a ring of shared-memory stages, running ahead across
//     item boundaries.
//   - The consumers reduce each stage and release it.  At an item's last stage
//     they merge their partials and hand the item to the epilogue warp through
//     a small queue.  They never wait on global-memory latency.
//   - The epilogue warp does the item's global work (publishing, decisions,
//     sampling jobs, locating tokens) while the ring keeps streaming.
//
// Epilogues.
//   - A stats item publishes its part's statistics.  The CTA completing the last
//     part of (b, i) merges the parts and advances b's decision frontier under b's
//     lock: positions are decided left to right as soon as their statistics are
//     ready.  A sequence that ends by a rejection or a bonus gets a sampling job.
//   - A residual part stores the residual mass of each (stage, warp) chunk in
//     token order.  The CTA completing a job's last part folds these masses, finds
//     the chunk whose running sum crosses v*R, reloads that chunk, and locates the
//     token (inverse CDF over the unnormalised residual r' = q' (1 - 2^delta)).
//
// Every wait and lock is bounded.  A wait that runs out records
// SPEC_ERR_TIMEOUT and stops the kernel; the last CTA out gives every
// unfinished sequence that error, reports the status and zeroes the workspace
// control region.
#pragma once
#include "sv_cluster.cuh"

namespace sv {

constexpr int WCONS = SW_WARPS;            // consumer warps (0 .. WCONS-1)
constexpr int WPROD = WCONS;               // the producer warp
constexpr int WEPI = WCONS + 1;            // the epilogue warp
constexpr int WTHREADS = (WCONS + 2) * 32;
constexpr int WEQ = 8;                     // epilogue queue entries
constexpr int WMASS = SW_MAXST * SW_WARPS;  // chunk masses of one sampling job (stages x warps)
constexpr int WRING = 6;                   // ring stages
constexpr int WSBH = 8192;                 // bytes of one row in a stage
constexpr int WSLOTS = 2;                  // item slots (work is claimed just in time)
enum { WK_STATS = 0, WK_RES = 1, WK_STOP = 2 };
enum { RF_BONUS = 1, RF_USEQ = 2 };


// An item as the producer hands it to the consumers.
struct alignas(16) WItem {
    int kind, b, pos, h;      // pos: the position (stats) or j (residual)
    int t0, nt, nst, e;       // tokens [t0, t0 + nt) in nst stages; e: sampling job
    float Mt, dLhi, dLlo, c;  // residual coefficients
    int flags, two, pad0, pad1;
};

// An item handed to the epilogue warp.
struct alignas(16) EpTask {
    int kind, b, pos, h, e, pad0, pad1, pad2;
    SwStat mine;                           // the part's statistics (stats items)
};

struct alignas(16) SwShared {
    WItem item[WSLOTS];
    EpTask ep[WEQ];
    int stage_slot[WRING];                 // item slot of the stage in each ring slot
    int stage_idx[WRING];                  // its stage index within the item
    Rec wr[WCONS];                         // per-warp partials of the current item
    unsigned long long full[WRING], empty[WRING], slot_free[WSLOTS], ep_full[WEQ], ep_empty[WEQ];
};
constexpr uint32_t SW_HDR = (uint32_t)((sizeof(SwShared) + 127) & ~size_t(127));
constexpr uint32_t SW_LOC = 2 * WSBH / WCONS;      // bytes of one row of the locate scratch (one chunk)
constexpr uint32_t SW_SMEM = SW_HDR + WRING * 2 * WSBH + 2 * SW_LOC + WMASS * sizeof(DF2);

__device__ __forceinline__ void sw_status(const SweepParams &P, int code)
{
    atomicCAS(&P.ctl[CTL_STATUS], 0u, (uint32_t)code);
}
__device__ __forceinline__ void sw_abort(const SweepParams &P)
{
    sw_status(P, ST_TIMEOUT);
    atomicExch(&P.swc[SWC_ABORT], 1u);
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
// The sequence's outputs are written: mark it finished.
__device__ __forceinline__ void sw_finish(const SweepParams &P, int b)
{
    __threadfence();
    st_vol(&P.seq[b].fin, 1u);
    atomicAdd(&P.swc[SWC_FIN], 1u);
}
// Records written by other CTAs (read through L2).
__device__ __forceinline__ SwStat ld_stat(const SwStat *p)
{
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const int4 z = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    return SwStat{a.x, a.y, a.z, a.w, __int_as_float(z.x), __int_as_float(z.y), z.z, z.w};
}
__device__ __forceinline__ SwRes ld_res(const SwRes *p)
{
    const int4 a = __ldcg(reinterpret_cast<const int4 *>(p));
    const float4 q = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    const float4 r = __ldcg(reinterpret_cast<const float4 *>(p) + 2);
    return SwRes{a.x, a.y, a.z, a.w, q.x, q.y, q.z, __float_as_uint(q.w), r.x, r.y, r.z, r.w};
}
__device__ __forceinline__ uint32_t ld_acq(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void cons_sync()   // the eight consumer warps
{
    asm volatile("bar.sync 1, %0;" ::"r"(WCONS * 32) : "memory");
}

// Merge the S part statistics of (b, i) in part order.
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

// Decide position f of sequence b from its merged statistics.  Returns 0 and
// sets accept, or a status code.
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
    accept = X >= 0.0f || u24_below(w.x, ex2a(X));
    return 0;
}

// Post a sampling job (flags: RF_*).  Rprev: the residual mass of an earlier
// attempt (reported as R when the job samples q_j itself).
__device__ void sw_post(const SweepParams &P, int b, int j, int flags, DF Rprev)
{
    const SwStat s = ld_stat(P.stat + (size_t)b * (P.K + 1) + j);
    SwRes r{};
    r.b = b;
    r.j = j;
    r.flags = flags;
    r.Mt = s.mt;
    int et, ed;
    float ft, fd;
    log2_split(DF{s.st_hi, s.st_lo}, et, ft);
    if (flags & RF_BONUS) {
        r.dLhi = r.dLlo = 0.0f;
    } else {
        // dL = (Md - Mt) + log2 Sd - log2 St as a float pair
        log2_split(DF{s.sd_hi, s.sd_lo}, ed, fd);
        DF dl = two_sum(s.md, -s.mt);
        dl = df_add(dl, DF{(float)(ed - et), 0.0f});
        dl = df_add(dl, DF{fd - ft, 0.0f});
        r.dLhi = dl.hi;
        r.dLlo = dl.lo;
    }
    const uint4 w = philox10((uint32_t)j, (uint32_t)b, 0u, 0u, P.key0, P.key1);
    r.vw = w.y;
    r.St_hi = s.st_hi;
    r.St_lo = s.st_lo;
    r.R_hi = Rprev.hi;
    r.R_lo = Rprev.lo;
    const uint32_t e = atomicAdd(&P.swc[SWC_RES_ALLOC], 1u);
    P.res[e] = r;
    __threadfence();
    st_vol(&P.res_ready[e], 1u);
}

// Advance b's decisions as far as ready statistics allow.  A sequence that
// ends by a rejection or a bonus gets a sampling job; greedy ends and errors
// write their outputs here.
template <class E>
__device__ void sw_advance(const SweepParams &P, int b)
{
    SwSeq *sq = P.seq + b;
    const int K = P.K;
    for (;;) {
        uint32_t it = 0;
        while (atomicCAS(&sq->lock, 0u, 1u) != 0u) {
            // another CTA is advancing b: it looks again after releasing the lock
            if (++it > 64)
                return;
            __nanosleep(32);
        }
        __threadfence();
        uint32_t f = ld_vol(&sq->front), e = ld_vol(&sq->end);
        while (e == 0u && (int)f <= K && (ld_acq(P.cnt + (size_t)b * (K + 1) + f) & SW_READY)) {
            bool accept = false;
            const int code = sw_decide<E>(P, b, (int)f, accept);
            if (code) {
                e = 0x80000000u | (uint32_t)code;
                sw_error(P, b, code);
                sw_finish(P, b);
                break;
            }
            if (accept && (int)f < K) {
                ++f;
                continue;
            }
            e = 1u + f;
            if (P.greedy) {
                const SwStat s = ld_stat(P.stat + (size_t)b * (K + 1) + f);
                sw_emit(P, b, (int)f, __float_as_int(s.st_hi));
                if (P.aux_R)
                    P.aux_R[b] = __int_as_float(0x7fc00000);
                sw_finish(P, b);
            } else {
                sw_post(P, b, (int)f, (int)f == K ? RF_BONUS : 0, DF{0.0f, 0.0f});
            }
            break;
        }
        st_vol(&sq->front, f);
        st_vol(&sq->end, e);
        __threadfence();
        atomicExch(&sq->lock, 0u);
        if (e != 0u)
            return;
        // statistics that became ready while the lock was held
        __threadfence();
        if ((int)f > K || !(ld_acq(P.cnt + (size_t)b * (K + 1) + f) & SW_READY))
            return;
    }
}

// Sample sequence r.b of job e once all its residual parts are stored: the
// total mass and the chunk whose running sum crosses v*R (a warp scan over
// the chunk masses in token order), then the token inside that chunk.  One
// warp; `loc` and `mass` are its shared-memory scratch.
template <class E>
__device__ void sw_locate(const SweepParams &P, int e, uint8_t *loc, DF2 *mass, int lane)
{
    constexpr int ST = WSBH / E::ES;
    constexpr int GPS = ST / 8;
    constexpr int GW = GPS / WCONS;
    const int K = P.K, V = P.V;
    const SwRes r = ld_res(P.res + e);
    const bool bonus = r.flags & RF_BONUS, useq = r.flags & RF_USEQ;
    // gather the chunk masses in token order: stage s of the row, warp w
    const int n = (V + ST - 1) / ST * SW_WARPS;
    {
        const DF2 *m = P.resm + (size_t)e * SW_MAXST * SW_WARPS;
        for (int i = lane; i < n; i += 32) {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(m) + i);   // written by other CTAs
            mass[i] = DF2{v.x, v.y};
        }
    }
    __syncwarp();
    // each lane sums a block of consecutive chunks; a scan over the lanes gives the running sums
    const int per = (n + 31) / 32;
    const int c0 = min(n, lane * per), c1 = min(n, c0 + per);
    DF blk{0.0f, 0.0f};
    for (int i = c0; i < c1; ++i)
        blk = df_add(blk, DF{mass[i].hi, mass[i].lo});
    const DF incl = warp_incl_scan_df(blk, lane);
    const DF F{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    if (!(F.hi > 0.0f) && !useq) {
        // R <= 0: sample q_j itself (a new job over the target row)
        if (lane == 0) {
            SwRes q = r;
            q.flags |= RF_USEQ;
            q.R_hi = F.hi;
            q.R_lo = F.lo;
            const uint32_t e2 = atomicAdd(&P.swc[SWC_RES_ALLOC], 1u);
            P.res[e2] = q;
            __threadfence();
            st_vol(&P.res_ready[e2], 1u);
        }
        return;
    }
    const DF R = (!useq || bonus) ? F : DF{r.R_hi, r.R_lo};
    const DF t = u24_scale(r.vw, F);
    // the crossing chunk: first lane whose running sum exceeds t, then inside its block
    int chunk = -1;
    DF Gc{0.0f, 0.0f};
    const unsigned bal = __ballot_sync(0xffffffffu, df_gt(incl, t) && c1 > c0);
    if (bal) {
        const int L = __ffs(bal) - 1;
        if (lane == L) {
            DF G = df_add(incl, DF{-blk.hi, -blk.lo});
            for (int i = c0; i < c1 && chunk < 0; ++i) {
                const DF nG = df_add(G, DF{mass[i].hi, mass[i].lo});
                if (df_gt(nG, t) && mass[i].hi > 0.0f) {
                    chunk = i;
                    Gc = G;
                }
                G = nG;
            }
        }
        chunk = __shfl_sync(0xffffffffu, chunk, L);
        Gc = DF{__shfl_sync(0xffffffffu, Gc.hi, L), __shfl_sync(0xffffffffu, Gc.lo, L)};
    }
    bool cfb = chunk < 0;
    if (cfb) {
        // rounding left no crossing: the last chunk with mass
        int lastc = -1;
        for (int i = lane; i < n; i += 32)
            if (mass[i].hi > 0.0f)
                lastc = i;
        chunk = warp_maxi(lastc);
    }
    int x = -1;
    if (chunk >= 0) {
        // chunk index -> stage of the row, warp
        const int ss = chunk / SW_WARPS, ws = chunk % SW_WARPS;
        const int t0 = 0;
        const int cnt = min(ST, V - ss * ST);
        const int ng = (cnt + 7) >> 3;
        const int g0 = min(ng, ws * GW), g1 = min(ng, g0 + GW);
        const uint8_t *jt = static_cast<const uint8_t *>(P.target) + ((size_t)r.b * (K + 1) + r.j) * (size_t)V * E::ES;
        const bool two = !(bonus || useq);
        const uint8_t *jd =
            two ? static_cast<const uint8_t *>(P.draft) + ((size_t)r.b * K + r.j) * (size_t)V * E::ES : nullptr;
        const size_t off = (size_t)(t0 + ss * ST) * E::ES;
        constexpr int TPV = 16 / E::ES;   // tokens per 16-byte vector
        // group g of the stage lands at byte (g - g0) * 8 * ES of the scratch
        uint8_t *lt = loc - (size_t)g0 * 8 * E::ES;
        uint8_t *ldp = loc + SW_LOC - (size_t)g0 * 8 * E::ES;
        for (int g = g0 + lane; g < g1; g += 32) {
            for (int hv = 0; hv < E::ES / 2; ++hv) {
                if (g * 8 + hv * TPV >= cnt)   // vectors past the row are not read
                    break;
                const size_t o = (size_t)g * 16 * (E::ES / 2) + (size_t)hv * 16;
                *reinterpret_cast<uint4 *>(lt + o) = __ldcg(reinterpret_cast<const uint4 *>(jt + off + o));
                if (two)
                    *reinterpret_cast<uint4 *>(ldp + o) = __ldcg(reinterpret_cast<const uint4 *>(jd + off + o));
            }
        }
        __syncwarp();
        ResK kc;
        kc.Mt = r.Mt;
        kc.dLhi = r.dLhi;
        kc.dLlo = r.dLlo;
        kc.c = P.c;
        const int xb = t0 + ss * ST;
        if (!cfb)
            x = warp_locate<E>(lt, ldp, cnt, g0, g1, kc, bonus, useq, Gc, t, xb, lane);
        if (x < 0)
            x = warp_last_positive<E>(lt, ldp, cnt, g0, g1, kc, bonus, useq, xb, lane);
    }
    if (lane == 0) {
        sw_emit(P, r.b, r.j, x);
        if (P.aux_R)
            P.aux_R[r.b] = (R.hi + R.lo) / (r.St_hi + r.St_lo);
        sw_finish(P, r.b);
    }
    __syncwarp();
}

template <class E>
__global__ void __launch_bounds__(WTHREADS, 2) sweep_kernel(const __grid_constant__ SweepParams P)
{
    extern __shared__ __align__(1024) uint8_t sw_smem[];
    SwShared &S = *reinterpret_cast<SwShared *>(sw_smem);
    uint8_t *ring = sw_smem + SW_HDR;
    uint8_t *loc = ring + WRING * 2 * WSBH;    // locate scratch: a target chunk, then a draft chunk
    DF2 *mass = reinterpret_cast<DF2 *>(loc + 2 * SW_LOC);   // a job's chunk masses, token order
    constexpr int ST = WSBH / E::ES;           // tokens per stage
    constexpr int GPS = ST / 8;                // groups per stage
    constexpr int GW = GPS / WCONS;            // groups per consumer warp per stage
    constexpr int JL = GW / 32;                // groups per lane per stage
    static_assert(JL >= 1 && GW % 32 == 0, "stage geometry");
    static_assert(GW * 8 * E::ES <= (int)SW_LOC, "locate scratch");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = P.K, V = P.V;
    const float c = P.c;

    if (tid == 0) {
        for (int i = 0; i < WRING; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], WCONS);
        }
        for (int i = 0; i < WSLOTS; ++i)
            mbar_init(&S.slot_free[i], 1);
        for (int i = 0; i < WEQ; ++i) {
            mbar_init(&S.ep_full[i], 1);
            mbar_init(&S.ep_empty[i], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == WPROD) {
        // ================================================================ producer
        if (lane == 0) {
            uint32_t k = 0, ni = 0, idle = 0, nap = 128;
            const uint32_t idle_limit = hinted_limit(P.spin_limit) * 64u;
            bool stop = false;
            while (!stop) {
                WItem it{};
                bool have = false;
                // 1. a residual part, if a sampling job is waiting (finishes sequences)
                const uint32_t alloc = ld_acq(&P.swc[SWC_RES_ALLOC]);
                uint32_t cl = ld_vol(&P.swc[SWC_RES_CLAIM]);
                while (cl < alloc * (uint32_t)P.RS) {
                    const uint32_t prev = atomicCAS(&P.swc[SWC_RES_CLAIM], cl, cl + 1u);
                    if (prev == cl)
                        break;
                    cl = prev;
                }
                if (cl < alloc * (uint32_t)P.RS) {
                    const uint32_t e = cl / (uint32_t)P.RS;
                    uint32_t w = 0;
                    while (!ld_acq(&P.res_ready[e]) && ++w < P.spin_limit)
                        __nanosleep(32);
                    const SwRes r = ld_res(P.res + e);
                    it.kind = WK_RES;
                    it.b = r.b;
                    it.pos = r.j;
                    it.h = (int)(cl % (uint32_t)P.RS);
                    it.e = (int)e;
                    it.flags = r.flags;
                    it.two = (r.flags & (RF_BONUS | RF_USEQ)) ? 0 : 1;
                    it.Mt = r.Mt;
                    it.dLhi = r.dLhi;
                    it.dLlo = r.dLlo;
                    have = true;
                }
                // 2. else the next stats item
                if (!have && ld_vol(&P.swc[SWC_ITEMS]) < P.n_items && !ld_vol(&P.swc[SWC_ABORT])) {
                    const uint32_t idx = atomicAdd(&P.swc[SWC_ITEMS], 1u);
                    if (idx < P.n_items) {
                        const int pos = (int)(idx / ((uint32_t)P.B * P.S));
                        const uint32_t rr = idx % ((uint32_t)P.B * P.S);
                        const int b = (int)(rr / P.S);
                        const uint32_t en = ld_vol(&P.seq[b].end);
                        idle = 0;
                        // a sequence that ended before pos needs nothing more
                        if (en != 0u && ((en & 0x80000000u) || (int)(en - 1u) < pos))
                            continue;
                        it.kind = WK_STATS;
                        it.b = b;
                        it.pos = pos;
                        it.h = (int)(rr % P.S);
                        it.two = (!P.greedy && pos < K) ? 1 : 0;
                        have = true;
                    }
                }
                if (!have) {
                    // nothing to hand out now: done once every sequence is finished
                    if (ld_vol(&P.swc[SWC_FIN]) >= (uint32_t)P.B || ld_vol(&P.swc[SWC_ABORT])) {
                        it.kind = WK_STOP;
                        stop = true;
                    } else if (++idle > idle_limit) {
                        sw_abort(P);
                        it.kind = WK_STOP;
                        stop = true;
                    } else {
                        // back off: idle producers poll the shared counters less and less often
                        __nanosleep(nap);
                        nap = min(nap * 2u, 4096u);
                        continue;
                    }
                }
                idle = 0;
                nap = 128;
                if (it.kind != WK_STOP) {
                    const int sp = it.kind == WK_RES ? P.rspan : P.span;
                    it.t0 = min(V, it.h * sp);
                    it.nt = min(sp, V - it.t0);
                    it.nst = (it.nt + ST - 1) / ST;
                    it.c = c;
                    if (it.nst == 0) {
                        // an empty part: publish a neutral part without streaming
                        it.nst = 1;
                        it.nt = 0;
                    }
                }
                // an item slot, once the consumers are done with its previous item
                const uint32_t slot = ni % WSLOTS, use = ni / WSLOTS;
                if (use > 0 && !ring_wait(&S.slot_free[slot], (use - 1) & 1u, P.spin_limit)) {
                    sw_abort(P);
                    it.kind = WK_STOP;
                    stop = true;
                }
                S.item[slot] = it;
                ++ni;
                const uint8_t *trow = nullptr, *drow = nullptr;
                if (it.kind != WK_STOP) {
                    const size_t bp = (size_t)it.b * (K + 1) + it.pos;
                    trow = static_cast<const uint8_t *>(P.target) + bp * (size_t)V * E::ES;
                    if (it.two)
                        drow = static_cast<const uint8_t *>(P.draft) +
                               ((size_t)it.b * K + it.pos) * (size_t)V * E::ES;
                }
                // its stages (a STOP, or an empty part, takes one stage without data)
                const int nst = it.kind == WK_STOP ? 1 : it.nst;
                for (int i = 0; i < nst; ++i) {
                    const uint32_t rs = k % WRING, ru = k / WRING;
                    if (ru > 0 && !ring_wait(&S.empty[rs], (ru - 1) & 1u, P.spin_limit)) {
                        sw_abort(P);
                        stop = true;   // the consumers time out on the missing stage
                        break;
                    }
                    S.stage_slot[rs] = (int)slot;
                    S.stage_idx[rs] = i;
                    const int cnt = it.kind == WK_STOP ? 0 : min(ST, it.nt - i * ST);
                    if (cnt <= 0) {
                        mbar_arrive(&S.full[rs]);
                    } else {
                        const uint32_t bytes = (uint32_t)cnt * E::ES;
                        uint8_t *dst = ring + rs * 2 * WSBH;
                        mbar_arrive_tx(&S.full[rs], drow ? 2u * bytes : bytes);
                        bulk_g2s(dst, trow + (size_t)(it.t0 + i * ST) * E::ES, bytes, &S.full[rs]);
                        if (drow)
                            bulk_g2s(dst + WSBH, drow + (size_t)(it.t0 + i * ST) * E::ES, bytes, &S.full[rs]);
                    }
                    ++k;
                }
            }
            // wind down: the copies still in flight
            for (uint32_t q = k >= (uint32_t)WRING ? k - WRING : 0u; q < k; ++q)
                (void)mbar_wait(&S.full[q % WRING], (q / WRING) & 1u, DRAIN_LIMIT, nullptr);
        }
        __syncwarp();
    } else if (warp < WCONS) {
        // ================================================================ consumers
        uint32_t k = 0, eqn = 0;
        float mt = -F_INF, st = 0.0f, md = -F_INF, sd = 0.0f, bv = -F_INF;
        int fl = 0, bi = -1;
        for (;;) {
            const uint32_t rs = k % WRING;
            if (!ring_wait_warp(&S.full[rs], (k / WRING) & 1u, P.spin_limit, lane)) {
                if (lane == 0)
                    sw_abort(P);
                break;   // the producer stops on the abort flag
            }
            const int slot = S.stage_slot[rs], i = S.stage_idx[rs];
            const WItem it = S.item[slot];
            if (it.kind == WK_STOP)
                break;
            const uint8_t *tb = ring + rs * 2 * WSBH, *db = tb + WSBH;
            const int cnt = max(0, min(ST, it.nt - i * ST));
            if (it.kind == WK_STATS) {
                if (i == 0) {
                    mt = md = bv = -F_INF;
                    st = sd = 0.0f;
                    fl = 0;
                    bi = -1;
                }
                if (P.greedy) {
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
                                bi = it.t0 + i * ST + g * 8 + e;
                            }
                        }
                    }
                } else if (cnt == ST) {
#pragma unroll
                    for (int jl = 0; jl < JL; ++jl) {
                        const int g = warp * GW + jl * 32 + lane;
                        f2 X[4];
                        Grp<E>::pairs(tb, g, X);
                        acc_group(X, c, mt, st, fl, 1);
                        if (it.two) {
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
                            if (it.two) {
                                (void)group8<E>(db, g, cnt, X);
                                acc_group(X, c, md, sd, fl, 2);
                            }
                        }
                    }
                }
            } else {
                // residual part: this warp's chunk of the stage, in token order
                ResK kc;
                kc.Mt = it.Mt;
                kc.dLhi = it.dLhi;
                kc.dLlo = it.dLlo;
                kc.c = it.c;
                const bool bonus = it.flags & RF_BONUS, useq = it.flags & RF_USEQ;
                const int ng = (cnt + 7) >> 3;
                const int g0 = min(ng, warp * GW), g1 = min(ng, g0 + GW);
                const DF W = warp_mass<E>(tb, db, cnt, g0, g1, kc, bonus, useq, lane);
                if (lane == 0) {
                    DF2 *m = P.resm + ((size_t)it.e * SW_MAXST + it.t0 / ST + i) * SW_WARPS + warp;
                    *m = DF2{W.hi, W.lo};
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.empty[rs]);
            ++k;
            if (i + 1 < it.nst)
                continue;

            // ---- the item's end: merge, and hand it to the epilogue warp
            EpTask task{};
            task.kind = it.kind;
            task.b = it.b;
            task.pos = it.pos;
            task.h = it.h;
            task.e = it.e;
            if (it.kind == WK_STATS) {
                if (P.greedy) {
                    float v = bv;
                    int ix = bi;
                    warp_merge_argmax(v, ix);
                    const int f = warp_or(fl);
                    if (lane == 0)
                        S.wr[warp] = Rec{v, __int_as_float(ix), 0.0f, f, 0.0f, 0.0f, 0.0f, 0};
                    cons_sync();
                    if (warp == 0) {
                        const bool in = lane < WCONS;
                        const Rec r = S.wr[in ? lane : 0];
                        float vv = in ? r.a0 : -F_INF;
                        int ii = in ? __float_as_int(r.a1) : -1;
                        warp_merge_argmax<WCONS>(vv, ii);
                        task.mine = SwStat{vv, __int_as_float(ii), 0.0f, 0.0f, 0.0f, 0.0f, warp_or(in ? r.i0 : 0), 0};
                    }
                } else {
                    float Mt, Md;
                    DF St, Sd;
                    merge_ms<32>(mt, DF{st, 0.0f}, c, Mt, St);
                    merge_ms<32>(md, DF{sd, 0.0f}, c, Md, Sd);
                    const int f = warp_or(fl);
                    if (lane == 0)
                        S.wr[warp] = Rec{Mt, St.hi, St.lo, f, Md, Sd.hi, Sd.lo, 0};
                    cons_sync();
                    if (warp == 0) {
                        const bool in = lane < WCONS;
                        const Rec r = S.wr[in ? lane : 0];
                        merge_ms<WCONS>(in ? r.a0 : -F_INF, in ? DF{r.a1, r.a2} : DF{0.0f, 0.0f}, c, Mt, St);
                        merge_ms<WCONS>(in ? r.b0 : -F_INF, in ? DF{r.b1, r.b2} : DF{0.0f, 0.0f}, c, Md, Sd);
                        task.mine = SwStat{Mt, St.hi, St.lo, Md, Sd.hi, Sd.lo, warp_or(in ? r.i0 : 0), 0};
                    }
                }
            } else {
                // the chunk masses this warp stored must be visible before the part counts as done
                if (lane == 0)
                    __threadfence();
                cons_sync();
            }
            if (tid == 0) {
                const uint32_t q = eqn % WEQ, u = eqn / WEQ;
                if (u > 0 && !ring_wait(&S.ep_empty[q], (u - 1) & 1u, P.spin_limit))
                    sw_abort(P);
                S.ep[q] = task;
                mbar_arrive(&S.ep_full[q]);
            }
            ++eqn;
            cons_sync();   // S.wr is free again
            if (tid == 0)
                mbar_arrive(&S.slot_free[slot]);
        }
        // tell the epilogue warp to stop
        if (tid == 0) {
            const uint32_t q = eqn % WEQ, u = eqn / WEQ;
            if (u > 0)
                (void)ring_wait(&S.ep_empty[q], (u - 1) & 1u, P.spin_limit);
            S.ep[q].kind = WK_STOP;
            mbar_arrive(&S.ep_full[q]);
        }
    } else {
        // ================================================================ epilogue warp
        uint32_t eq = 0;
        for (;;) {
            const uint32_t q = eq % WEQ;
            if (!ring_wait_warp(&S.ep_full[q], (eq / WEQ) & 1u, P.spin_limit, lane)) {
                if (lane == 0)
                    sw_abort(P);
                break;
            }
            const EpTask task = S.ep[q];
            if (task.kind == WK_STOP)
                break;
            if (task.kind == WK_STATS) {
                if (lane == 0) {
                    const size_t bp = (size_t)task.b * (K + 1) + task.pos;
                    P.part[bp * P.S + task.h] = task.mine;
                    __threadfence();
                    const uint32_t done = atomicAdd(P.cnt + bp, 1u) + 1u;
                    if (done == (uint32_t)P.S) {
                        __threadfence();
                        P.stat[bp] = merge_parts(P, bp);
                        __threadfence();
                        atomicOr(P.cnt + bp, SW_READY);
                        sw_advance<E>(P, task.b);
                    }
                }
            } else {
                // a residual part is done: the last part of its job locates the token
                int last = 0;
                if (lane == 0) {
                    __threadfence();
                    last = atomicAdd(P.res_done + task.e, 1u) + 1u == (uint32_t)P.RS;
                    __threadfence();
                }
                if (__shfl_sync(0xffffffffu, last, 0))
                    sw_locate<E>(P, task.e, loc, mass, lane);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&S.ep_empty[q]);
            ++eq;
        }
    }

    // ---- the last CTA out finalises
    __syncthreads();
    __shared__ int last;
    if (tid == 0) {
        __threadfence();
        last = atomicAdd(&P.swc[SWC_EXIT], 1u) == gridDim.x - 1;
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
