// sv_cluster.cuh -- verification with one sequence per thread-block cluster.
//
// The rule is the one of verify_kernel (nextadmin.net lesson "Speculative
// Decoding", § Core algorithm steps 4-6; aiengineeringfromscratch.com lesson
// 25, § The exact rule and § Greedy case; q = target, p = draft); this kernel
// organises the work around the sequence instead of the chunk.
//
// A cluster of C CTAs verifies one sequence at a time, left to right.  CTA r
// owns tokens [r*chunk, (r+1)*chunk) of every row.  For position i it copies
// its slice of target row i (and draft row i) into shared memory with
// cp.async.bulk, and reduces it: the maximum and the sum of 2^((x - m) c) per
// row, or for greedy the maximum and its lowest index.  It then sends a
// 32-byte record to every CTA of the cluster: st.async into the peers'
// shared memory, with completion counted on their mbarriers.  Each CTA merges
// the C records in rank order, so all of them reach the same decision without
// another exchange.  Rows after a rejection are never read.
//
// At the first rejection j the residual r(x) = max(0, q_j(x) - p_j(x)) comes
// from the slices still held in shared memory (a bonus samples q_{K+1}):
//   - each warp forms its mass in token order, one 256-token segment at a time;
//   - one more exchange carries the per-CTA masses;
//   - the CTA, then the warp, whose running sum crosses v*R locates the token.
// No row is read twice and no probability is stored.
//
// Sequences come from a global counter.  Each claim is made during the first
// position of the sequence before it, so the atomic's latency is hidden.
// Several clusters share an SM (about 64 KB of shared memory each), so one
// cluster's decision latency is covered by the others' copies.  Every wait is
// bounded: one that runs out gives SPEC_ERR_TIMEOUT for the unfinished
// sequences and ends the kernel.
#pragma once
#include "sv_kernel.cuh"

namespace sv {

constexpr int CL_WARPS = 8;
constexpr int CL_THREADS = CL_WARPS * 32;
constexpr int CL_MAX = 16;   // largest cluster
constexpr int SEGB = 4;      // residual segments whose lane sums are formed together

// One CTA's contribution to one exchange round.
//   stats:   a = (target max, sum hi, sum lo, flags), b = (draft max, sum hi, sum lo, claimed sequence)
//   greedy:  a = (max, -, -, flags), b = (-, -, -, claimed sequence), index in a1's bits
//   masses:  a = (mass hi, mass lo, -, -)
struct alignas(16) Rec {
    float a0, a1, a2;
    int i0;
    float b0, b1, b2;
    int i1;
};

struct alignas(16) ClShared {
    Rec rx[2][CL_MAX];            // records received, by round parity and sender rank
    Rec wr[CL_WARPS];             // this CTA's per-warp partials / masses
    unsigned long long full;      // slice copies of the current position
    unsigned long long xbar[2];   // exchange rounds, by parity
};
constexpr uint32_t CL_HDR = (uint32_t)((sizeof(ClShared) + 127) & ~size_t(127));

// Flags carried in Rec::i0.
enum { FL_T = 1, FL_D = 2, FL_TIMEOUT = 4 };

// ------------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cl_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_count()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cl_map(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void cl_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 16-byte store into a peer's shared memory, counted on the peer's mbarrier.
__device__ __forceinline__ void st_async16(uint32_t dst, uint4 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     dst),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                 : "memory");
}
// Suspend time hint (ns) for the waits below: the warp sleeps in hardware
// until the phase completes or this much time has passed, instead of
// spinning and taking issue slots from the warps that compute.
constexpr uint32_t WAIT_HINT_NS = 20000;

__device__ __forceinline__ bool cl_test(unsigned long long *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity), "r"(WAIT_HINT_NS)
        : "memory");
    return ok != 0;
}
// A CTA-local phase wait with the suspend hint (the data came by cp.async.bulk).
__device__ __forceinline__ bool mbar_test_hint(unsigned long long *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity), "r"(WAIT_HINT_NS)
        : "memory");
    return ok != 0;
}
// The same test without suspending: one poll.
__device__ __forceinline__ bool cl_poll(unsigned long long *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Number of hinted waits that make up a spin limit of `limit` polls.
__device__ __forceinline__ uint32_t hinted_limit(uint32_t limit) { return (limit >> 8) + 16u; }
// Bounded wait on one of the CTA's own mbarriers (its ring of copies, its
// hand-offs between warps): hinted try_wait sleeps the thread in hardware
// until the phase completes (or the hint runs out).  Returns false when the
// waits allowed by `limit` ran out.  The bound never goes below OWN_WAIT_MIN
// polls, so a small spin limit runs out only the waits on other CTAs, and a
// CTA never winds down with its own copies still landing.
__device__ __forceinline__ bool ring_wait(unsigned long long *bar, uint32_t parity, uint32_t limit)
{
    const uint32_t lim = hinted_limit(limit > OWN_WAIT_MIN ? limit : OWN_WAIT_MIN);
    for (uint32_t it = 0;; ++it) {
        if (mbar_test_hint(bar, parity))
            return true;
        if (it >= lim)
            return false;
    }
}
// Warp-uniform form: lane 0 waits, then every lane observes the phase.
__device__ __forceinline__ bool ring_wait_warp(unsigned long long *bar, uint32_t parity, uint32_t limit, int lane)
{
    bool ok = true;
    if (lane == 0)
        ok = ring_wait(bar, parity, limit);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok)
        (void)mbar_test(bar, parity);
    __syncwarp();
    return ok;
}

// Warp-uniform bounded wait for an exchange round (records written by peers).
// Gives up after `limit` polls, or early once another CTA has aborted.  A
// limit below CL_PLAIN_POLLS is that many plain polls (a spin limit of 1 gives
// up unless the records are already there); above it, hinted waits.
constexpr uint32_t CL_PLAIN_POLLS = 64;
__device__ __forceinline__ bool cl_wait(unsigned long long *bar, uint32_t parity, uint32_t limit,
                                        const uint32_t *abortw, int lane)
{
    bool ok = true;
    if (lane == 0) {
        if (limit < CL_PLAIN_POLLS) {
            for (uint32_t it = 0;; ++it) {
                if (cl_poll(bar, parity))
                    break;
                if (it + 1 >= limit || ld_vol(abortw)) {
                    ok = false;
                    break;
                }
            }
        } else {
            const uint32_t lim = hinted_limit(limit);
            for (uint32_t it = 0;; ++it) {
                if (cl_test(bar, parity))
                    break;
                if (it >= lim || ld_vol(abortw)) {
                    ok = false;
                    break;
                }
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok)
        (void)cl_test(bar, parity);
    __syncwarp();
    return ok;
}

// ------------------------------------------------------------------ small numerics
__device__ __forceinline__ float lg2a(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// a > b for float pairs
__device__ __forceinline__ bool df_gt(DF a, DF b)
{
    const DF d = two_sum(a.hi, -b.hi);
    return d.hi + (d.lo + (a.lo - b.lo)) > 0.0f;
}
__device__ __forceinline__ DF warp_incl_scan_df(DF v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const DF t{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
        if (lane >= o)
            v = df_add(v, t);
    }
    return v;
}
__device__ __forceinline__ float warp_maxf(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// log2 of a positive float pair S >= 1 as an exact integer e plus a fraction
// f in [-1, 0): S = 2^e * m with m in [1/2, 1), f = log2(m).
__device__ __forceinline__ void log2_split(DF S, int &e, float &f)
{
    e = ((__float_as_int(S.hi) >> 23) & 0xff) - 126;
    const float sc = __int_as_float((127 - e) << 23);   // 2^-e, exact
    const float mh = S.hi * sc, ml = S.lo * sc;
    f = lg2a(mh) + ml / mh * 1.4426950408889634f;
}
// Merge per-lane (reference mc, sum relative to 2^mc) partials over aligned
// groups of W lanes (W a power of two): every lane gets its group's largest
// reference M and the sum relative to 2^M, as a float pair.
template <int W>
__device__ __forceinline__ void merge_ms(float m, DF s, float c, float &M, DF &S)
{
    (void)c;
    M = m;
#pragma unroll
    for (int o = W / 2; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    S = (m > -F_INF) ? df_scale_pow2(s, m - M) : DF{0.0f, 0.0f};
#pragma unroll
    for (int o = W / 2; o; o >>= 1)
        S = df_add(S, DF{__shfl_xor_sync(0xffffffffu, S.hi, o), __shfl_xor_sync(0xffffffffu, S.lo, o)});
}
// The same for a runtime group width w in {1, 2, 4, 8, 16}.
__device__ __forceinline__ void merge_ms_w(int w, float m, DF s, float c, float &M, DF &S)
{
    if (w <= 8)
        merge_ms<8>(m, s, c, M, S);
    else
        merge_ms<16>(m, s, c, M, S);
}
template <int W = 32>
__device__ __forceinline__ void warp_merge_argmax(float &v, int &i)
{
#pragma unroll
    for (int o = W / 2; o; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        argmax_merge(v, i, v2, i2);
    }
}

// ------------------------------------------------------------------ slice access
// Group g (8 tokens) of a slice of n tokens in shared memory as 4 float pairs
// (tokens past n read as -inf); returns the group's NaN-propagating maximum.
template <class E>
__device__ __forceinline__ float group8(const uint8_t *base, int g, int n, f2 *X);

template <>
__device__ __forceinline__ float group8<BF16>(const uint8_t *base, int g, int n, f2 *X)
{
    uint4 v = reinterpret_cast<const uint4 *>(base)[g];
    const int k = n - g * 8;
    if (k < 8) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (2 * i >= k)
                w[i] = 0xff80ff80u;
            else if (2 * i + 1 >= k)
                w[i] = (w[i] & 0x0000ffffu) | 0xff800000u;
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
        X[p] = BF16::pair(v, p);
    return BF16::vec_max(v);
}
template <>
__device__ __forceinline__ float group8<F32>(const uint8_t *base, int g, int n, f2 *X)
{
    uint4 v0 = reinterpret_cast<const uint4 *>(base)[2 * g];
    uint4 v1 = reinterpret_cast<const uint4 *>(base)[2 * g + 1];
    const int k = n - g * 8;
    if (k < 8) {
        uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i >= k)
                w[i] = 0xff800000u;
        v0 = make_uint4(w[0], w[1], w[2], w[3]);
        v1 = make_uint4(w[4], w[5], w[6], w[7]);
    }
    X[0] = F32::pair(v0, 0);
    X[1] = F32::pair(v0, 1);
    X[2] = F32::pair(v1, 0);
    X[3] = F32::pair(v1, 1);
    return fmax_nan(F32::vec_max(v0), F32::vec_max(v1));
}

// Full groups (8 tokens, no masking) for the slice reductions.
//   acc_max: fold the group into a packed running maximum (NaN-propagating);
//   pairs:   the group as 4 float pairs.
template <class E> struct Grp;
template <> struct Grp<BF16> {
    typedef uint32_t Acc;
    static __device__ __forceinline__ Acc acc_init() { return 0xff80ff80u; }
    static __device__ __forceinline__ Acc acc_max(const uint8_t *base, int g, Acc a)
    {
        const uint4 v = reinterpret_cast<const uint4 *>(base)[g];
        return bmax2(a, bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w)));
    }
    static __device__ __forceinline__ float acc_value(Acc a) { return BF16::word_max(a); }
    static __device__ __forceinline__ void pairs(const uint8_t *base, int g, f2 *X)
    {
        const uint4 v = reinterpret_cast<const uint4 *>(base)[g];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            X[p] = BF16::pair(v, p);
    }
};
template <> struct Grp<F32> {
    typedef float Acc;
    static __device__ __forceinline__ Acc acc_init() { return -F_INF; }
    static __device__ __forceinline__ Acc acc_max(const uint8_t *base, int g, Acc a)
    {
        const uint4 v0 = reinterpret_cast<const uint4 *>(base)[2 * g];
        const uint4 v1 = reinterpret_cast<const uint4 *>(base)[2 * g + 1];
        return fmax_nan(a, fmax_nan(F32::vec_max(v0), F32::vec_max(v1)));
    }
    static __device__ __forceinline__ float acc_value(Acc a) { return a; }
    static __device__ __forceinline__ void pairs(const uint8_t *base, int g, f2 *X)
    {
        const uint4 v0 = reinterpret_cast<const uint4 *>(base)[2 * g];
        const uint4 v1 = reinterpret_cast<const uint4 *>(base)[2 * g + 1];
        X[0] = F32::pair(v0, 0);
        X[1] = F32::pair(v0, 1);
        X[2] = F32::pair(v1, 0);
        X[3] = F32::pair(v1, 1);
    }
};

// Sum over one group of 2^(x c - mc), as a float pair (lo, hi lanes).
__device__ __forceinline__ f2 sum_exp8(const f2 *X, f2 cc, f2 nmc)
{
    f2 e[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
        e[p] = ex2x2(fma2(X[p], cc, nmc));
    return add2(add2(e[0], e[2]), add2(e[1], e[3]));
}

// Adds one group (4 float pairs) to a running partial (reference mc in log2
// units, s = sum 2^(x c - mc)).  The common case is one packed FMA, one ex2
// and one add per token plus a single compare on the group's sum.  The slow
// path is taken when that sum is not below 2^32, which covers:
//   - the first group (mc = -inf),
//   - a group more than about 2^29 above the reference,
//   - NaN or +inf (which set `bit` in fl).
// There the group maximum moves the reference.  Below 2^32 the sum simply
// grows, so the reference rarely moves.
__device__ __forceinline__ void acc_group(const f2 *X, float c, float &mc, float &s, int &fl, int bit)
{
    const f2 cc = pk(c, c);
    float lo, hi;
    upk(sum_exp8(X, cc, pk(-mc, -mc)), lo, hi);
    const float t = lo + hi;
    if (t < 4294967296.0f) {
        s += t;
        return;
    }
    float x[8];
#pragma unroll
    for (int p = 0; p < 4; ++p)
        upk(X[p], x[2 * p], x[2 * p + 1]);
    float gm = x[0];
#pragma unroll
    for (int e = 1; e < 8; ++e)
        gm = fmax_nan(gm, x[e]);
    if (!(gm == gm) || gm == F_INF) {
        fl |= bit;
        return;
    }
    if (!(gm > -F_INF))
        return;
    const float gmc = gm * c;
    if (gmc > mc) {
        s = (mc > -F_INF) ? s * ex2a(mc - gmc) : 0.0f;
        mc = gmc;
    }
    upk(sum_exp8(X, cc, pk(-mc, -mc)), lo, hi);
    s += lo + hi;
}

// One thread's partial over the groups tid, tid + T, ... of a slice of n
// tokens: a reference mc (a maximum logit times c, rounded) and
// s = sum 2^(x c - mc), in one pass.  The last, partial group (n not a
// multiple of 8) is masked to -inf.  NaN or +inf sets `bit` in fl.
template <class E>
__device__ __forceinline__ void thread_stats(const uint8_t *base, int n, int tid, float c, float &mc, float &s,
                                             int &fl, int bit)
{
    const int nf = n >> 3;
    mc = -F_INF;
    s = 0.0f;
    int g = tid;
    for (; g + CL_THREADS < nf; g += 2 * CL_THREADS) {
        f2 X[4], Y[4];
        Grp<E>::pairs(base, g, X);
        Grp<E>::pairs(base, g + CL_THREADS, Y);
        acc_group(X, c, mc, s, fl, bit);
        acc_group(Y, c, mc, s, fl, bit);
    }
    if (g < nf) {
        f2 X[4];
        Grp<E>::pairs(base, g, X);
        acc_group(X, c, mc, s, fl, bit);
    }
    if ((n & 7) != 0 && tid == nf % CL_THREADS) {
        f2 T[4];
        (void)group8<E>(base, nf, n, T);
        acc_group(T, c, mc, s, fl, bit);
    }
}

// Residual coefficients of the position a sequence ended at, in log2 units:
// Mt = the target reference (largest mc), dL = log2 of (Z_draft / Z_target)
// relative to the references, as a float pair: dL = (Md - Mt) + log2 Sd - log2 St.
struct ResK {
    float Mt, dLhi, dLlo, c;
};

// r'(x) (or q'(x) when `useq`) for the 8 tokens of group g, scaled by the
// target's normaliser (r' = r * St, so the normaliser drops out of the
// inverse CDF):
//   q'(x) = 2^(xt c - Mt),
//   delta = log2(p(x) / q(x)) = (xd - xt) c - dL,
//   r'(x) = q'(x) (1 - 2^delta) for delta < 0, else 0.
// 1 - 2^delta has no cancellation on [-1, 0) in the form
// -2 * 2^(delta/2) * sinh(delta ln2 / 2), where sinh is its odd Taylor series
// to y^9 (|y| <= ln2/2: truncation below 3e-10 relative; about 5e-7 relative
// with ex2.approx).  Below -1 it is 1 - ex2(delta), where 2^delta < 1/2.  One
// ex2 serves both branches.  Tokens with xt = -inf give 0.
template <class E>
__device__ __forceinline__ void res_group(const uint8_t *bt, const uint8_t *bd, int n, int g, const ResK &k,
                                          bool bonus, bool useq, float *v)
{
    f2 XT[4], XD[4];
    (void)group8<E>(bt, g, n, XT);
    const f2 cc = pk(k.c, k.c), nMt = pk(-k.Mt, -k.Mt);
    f2 Q[4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
        Q[p] = ex2x2(fma2(XT[p], cc, nMt));
    if (bonus || useq) {
#pragma unroll
        for (int p = 0; p < 4; ++p)
            upk(Q[p], v[2 * p], v[2 * p + 1]);
        return;
    }
    (void)group8<E>(bd, g, n, XD);
    const f2 ndh = pk(-k.dLhi, -k.dLhi), ndl = pk(-k.dLlo, -k.dLlo);
    const f2 hl = pk(0.34657359027997264f, 0.34657359027997264f);   // ln2 / 2
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const f2 dd = fma2(XT[p], pk(-1.0f, -1.0f), XD[p]);           // xd - xt (exact for bf16 inputs)
        float d0, d1;
        upk(add2(fma2(dd, cc, ndh), ndl), d0, d1);                    // delta
        d0 = fminf(d0, 0.0f);                                         // also maps NaN (both -inf) to 0
        d1 = fminf(d1, 0.0f);
        const bool far0 = d0 < -1.0f, far1 = d1 < -1.0f;
        float e0, e1;
        upk(ex2x2(pk(far0 ? d0 : 0.5f * d0, far1 ? d1 : 0.5f * d1)), e0, e1);
        const f2 y = mul2(pk(d0, d1), hl);
        const f2 y2 = mul2(y, y);
        f2 sp = pk(1.0f / 362880.0f, 1.0f / 362880.0f);
        sp = fma2(sp, y2, pk(1.0f / 5040.0f, 1.0f / 5040.0f));
        sp = fma2(sp, y2, pk(1.0f / 120.0f, 1.0f / 120.0f));
        sp = fma2(sp, y2, pk(1.0f / 6.0f, 1.0f / 6.0f));
        sp = fma2(sp, y2, pk(1.0f, 1.0f));
        float s0, s1;
        upk(mul2(y, sp), s0, s1);                                     // sinh(delta ln2 / 2)
        const float o0 = far0 ? 1.0f - e0 : -2.0f * e0 * s0;
        const float o1 = far1 ? 1.0f - e1 : -2.0f * e1 * s1;
        upk(mul2(Q[p], pk(o0, o1)), v[2 * p], v[2 * p + 1]);
    }
}
__device__ __forceinline__ float tree8(const float *v)
{
    return ((v[0] + v[4]) + (v[2] + v[6])) + ((v[1] + v[5]) + (v[3] + v[7]));
}

// Sum of one lane's 8 values of segment sg (groups g0 + 32 sg + lane), 0 past g1.
template <class E>
__device__ __forceinline__ float lane_seg(const uint8_t *bt, const uint8_t *bd, int n, int g0, int g1, int sg,
                                          const ResK &k, bool bonus, bool useq, int lane)
{
    const int g = g0 + sg * 32 + lane;
    if (g >= g1)
        return 0.0f;
    float v[8];
    res_group<E>(bt, bd, n, g, k, bonus, useq, v);
    return tree8(v);
}

// Mass of groups [g0, g1): each lane sums its groups (one per 256-token
// segment) as a float pair, then one float-pair butterfly over the lanes.
template <class E>
__device__ DF warp_mass(const uint8_t *bt, const uint8_t *bd, int n, int g0, int g1, const ResK &k, bool bonus,
                        bool useq, int lane)
{
    const int nseg = (g1 - g0 + 31) / 32;
    DF W{0.0f, 0.0f};
    for (int sb = 0; sb < nseg; sb += SEGB) {
        float ls[SEGB];
#pragma unroll
        for (int i = 0; i < SEGB; ++i)
            ls[i] = sb + i < nseg ? lane_seg<E>(bt, bd, n, g0, g1, sb + i, k, bonus, useq, lane) : 0.0f;
#pragma unroll
        for (int i = 0; i < SEGB; ++i)
            W = df_add(W, DF{ls[i], 0.0f});
    }
    return warp_sum_df(W);
}

// Largest token in groups [g0, g1) with positive mass (-1 if none).
template <class E>
__device__ int warp_last_positive(const uint8_t *bt, const uint8_t *bd, int n, int g0, int g1, const ResK &k,
                                  bool bonus, bool useq, int x0, int lane)
{
    int best = -1;
    for (int g = g0 + lane; g < g1; g += 32) {
        float v[8];
        res_group<E>(bt, bd, n, g, k, bonus, useq, v);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (v[e] > 0.0f)
                best = x0 + g * 8 + e;
    }
    return warp_maxi(best);
}

// Inverse CDF inside one warp's groups [g0, g1): the smallest token whose
// running sum (starting at G) exceeds t.  Segment totals are formed exactly
// as in warp_mass; inside the crossing segment a lane scan finds the lane and
// a scan over its 8 values the token.  Returns -1 when rounding leaves no
// crossing.
template <class E>
__device__ int warp_locate(const uint8_t *bt, const uint8_t *bd, int n, int g0, int g1, const ResK &k,
                           bool bonus, bool useq, DF G, DF t, int x0, int lane)
{
    const int nseg = (g1 - g0 + 31) / 32;
    int sstar = -1;
    for (int sb = 0; sb < nseg && sstar < 0; sb += SEGB) {
        float ls[SEGB];
#pragma unroll
        for (int i = 0; i < SEGB; ++i)
            ls[i] = sb + i < nseg ? lane_seg<E>(bt, bd, n, g0, g1, sb + i, k, bonus, useq, lane) : 0.0f;
#pragma unroll
        for (int i = 0; i < SEGB; ++i) {
            if (sstar < 0 && sb + i < nseg) {
                const DF Gn = df_add(G, warp_sum_df(DF{ls[i], 0.0f}));
                if (df_gt(Gn, t))
                    sstar = sb + i;
                else
                    G = Gn;
            }
        }
    }
    if (sstar < 0)
        return -1;
    const int g = g0 + sstar * 32 + lane;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (g < g1)
        res_group<E>(bt, bd, n, g, k, bonus, useq, v);
    const float ls = tree8(v);
    const DF incl = warp_incl_scan_df(DF{ls, 0.0f}, lane);
    int last = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (v[e] > 0.0f)
            last = x0 + g * 8 + e;
    const bool cross = df_gt(df_add(G, incl), t) && ls > 0.0f;
    const unsigned bal = __ballot_sync(0xffffffffu, cross);
    if (!bal)
        return warp_maxi(last);
    const int L = __ffs(bal) - 1;
    int x = -1;
    if (lane == L) {
        DF cum = df_add(G, df_add(incl, DF{-ls, 0.0f}));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            cum = df_add(cum, DF{v[e], 0.0f});
            if (x < 0 && v[e] > 0.0f && df_gt(cum, t))
                x = x0 + g * 8 + e;
        }
        if (x < 0)
            x = last;
    }
    return __shfl_sync(0xffffffffu, x, L);
}

// ------------------------------------------------------------------ outputs
__device__ __forceinline__ void cl_status(const ClusterParams &P, int code)
{
    atomicCAS(&P.ctl[CTL_STATUS], 0u, (uint32_t)code);
}
__device__ __forceinline__ void cl_error(const ClusterParams &P, int b, int code)
{
    for (int i = 0; i <= P.K; ++i)
        P.out_tokens[(size_t)b * (P.K + 1) + i] = -1;
    P.out_len[b] = -code;
    if (P.aux_R)
        P.aux_R[b] = __int_as_float(0x7fc00000);
    cl_status(P, code);
}
// Accepted drafts 0..j-1, then (if x >= 0) the emitted token at j; -1 after.
__device__ __forceinline__ void cl_emit(const ClusterParams &P, int b, int j, int x)
{
    int32_t *out = P.out_tokens + (size_t)b * (P.K + 1);
    for (int i = 0; i < j; ++i)
        out[i] = __ldg(P.tokens + (size_t)b * P.K + i);
    if (x >= 0)
        out[j] = x;
    for (int i = j + 1; i <= P.K; ++i)
        out[i] = -1;
    P.out_len[b] = j;
}

// Send lane 0's record to every CTA of the cluster (lane l writes CTA l's
// copy): `slot` is this CTA's own receive slot for the sender (the same offset
// in every CTA), `bar` the round's mbarrier.
__device__ __forceinline__ void send_rec_to(Rec *slot, unsigned long long *bar, uint32_t C, const Rec &r0, int lane)
{
    Rec r;
    r.a0 = __shfl_sync(0xffffffffu, r0.a0, 0);
    r.a1 = __shfl_sync(0xffffffffu, r0.a1, 0);
    r.a2 = __shfl_sync(0xffffffffu, r0.a2, 0);
    r.i0 = __shfl_sync(0xffffffffu, r0.i0, 0);
    r.b0 = __shfl_sync(0xffffffffu, r0.b0, 0);
    r.b1 = __shfl_sync(0xffffffffu, r0.b1, 0);
    r.b2 = __shfl_sync(0xffffffffu, r0.b2, 0);
    r.i1 = __shfl_sync(0xffffffffu, r0.i1, 0);
    if ((uint32_t)lane < C) {
        const uint32_t dst = cl_map(saddr(slot), (uint32_t)lane);
        const uint32_t rb = cl_map(saddr(bar), (uint32_t)lane);
        st_async16(dst, make_uint4(__float_as_uint(r.a0), __float_as_uint(r.a1), __float_as_uint(r.a2), (uint32_t)r.i0),
                   rb);
        st_async16(dst + 16,
                   make_uint4(__float_as_uint(r.b0), __float_as_uint(r.b1), __float_as_uint(r.b2), (uint32_t)r.i1),
                   rb);
    }
}

// Send lane 0's record of the round with parity `par` to every CTA (lane l
// writes CTA l's copy).
__device__ __forceinline__ void send_rec(ClShared &S, uint32_t par, uint32_t me, uint32_t C, const Rec &r0, int lane)
{
    Rec r;
    r.a0 = __shfl_sync(0xffffffffu, r0.a0, 0);
    r.a1 = __shfl_sync(0xffffffffu, r0.a1, 0);
    r.a2 = __shfl_sync(0xffffffffu, r0.a2, 0);
    r.i0 = __shfl_sync(0xffffffffu, r0.i0, 0);
    r.b0 = __shfl_sync(0xffffffffu, r0.b0, 0);
    r.b1 = __shfl_sync(0xffffffffu, r0.b1, 0);
    r.b2 = __shfl_sync(0xffffffffu, r0.b2, 0);
    r.i1 = __shfl_sync(0xffffffffu, r0.i1, 0);
    if ((uint32_t)lane < C) {
        const uint32_t dst = cl_map(saddr(&S.rx[par][me]), (uint32_t)lane);
        const uint32_t bar = cl_map(saddr(&S.xbar[par]), (uint32_t)lane);
        st_async16(dst, make_uint4(__float_as_uint(r.a0), __float_as_uint(r.a1), __float_as_uint(r.a2), (uint32_t)r.i0),
                   bar);
        st_async16(dst + 16,
                   make_uint4(__float_as_uint(r.b0), __float_as_uint(r.b1), __float_as_uint(r.b2), (uint32_t)r.i1),
                   bar);
    }
}

// =================================================================== kernel
template <class E, int MODE>
__global__ void __launch_bounds__(CL_THREADS, 3) cluster_kernel(const __grid_constant__ ClusterParams P)
{
    extern __shared__ __align__(1024) uint8_t cl_smem[];
    ClShared &S = *reinterpret_cast<ClShared *>(cl_smem);
    uint8_t *bt = cl_smem + CL_HDR;                                   // target slice
    uint8_t *bd = bt + (size_t)P.chunk * E::ES;                      // draft slice
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t me = cl_rank(), C = cl_size(), ncl = cl_count();
    const int K = P.K, V = P.V;
    const int x0 = min(V, (int)me * P.chunk);
    const int n = min(P.chunk, V - x0);                              // tokens of this CTA's slice
    const int ng = (n + 7) >> 3;
    const uint32_t rec_bytes = 32u * C;
    const float c = P.c;

    if (tid == 0) {
        mbar_init(&S.full, 1);
        mbar_init(&S.xbar[0], 1);
        mbar_init(&S.xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_tx(&S.xbar[0], rec_bytes);
        mbar_arrive_tx(&S.xbar[1], rec_bytes);
    }
    __syncthreads();
    cl_sync();   // every CTA's barriers are armed before any record is sent

    uint32_t round = 0, loads = 0;
    bool load_pending = false, abort = false;
    int ab_b = -1;   // the sequence this CTA gave up on (an exchange wait ran out)
    int b = (int)cl_id();
    int claimed = P.B;   // rank 0's claim for the next sequence (held by thread 0)

    while (b < P.B && !abort) {
        int next_b = P.B;
        for (int pos = 0;; ++pos) {
            const bool has_d = MODE == MODE_STOCH && pos < K;
            const size_t bp = (size_t)b * (K + 1) + pos;
            // ---- copy this CTA's slices of row pos (target, and draft)
            if (tid == 0 && n > 0) {
                const uint32_t bytes = (uint32_t)n * E::ES;
                mbar_arrive_tx(&S.full, has_d ? 2u * bytes : bytes);
                bulk_g2s(bt, static_cast<const uint8_t *>(P.target) + (bp * (size_t)V + x0) * E::ES, bytes, &S.full);
                if (has_d)
                    bulk_g2s(bd,
                             static_cast<const uint8_t *>(P.draft) +
                                 (((size_t)b * K + pos) * (size_t)V + x0) * E::ES,
                             bytes, &S.full);
                load_pending = true;
            }
            if (tid == 0 && me == 0 && pos == 0)
                claimed = (int)min((uint32_t)P.B, ncl + atomicAdd(&P.ctl[CTL_CL_NEXT], 1u));
            // the drafted token and its two logits (every warp decides for itself)
            int d = -1;
            float zt_d = 0.0f, zd_d = 0.0f;
            if (pos < K) {
                d = __ldg(P.tokens + (size_t)b * K + pos);
                if (MODE == MODE_STOCH && lane == 0 && d >= 0 && d < V) {
                    zt_d = E::load(P.target, bp * (size_t)V + d);
                    zd_d = E::load(P.draft, ((size_t)b * K + pos) * (size_t)V + d);
                }
            }
            // ---- reduce the slice
            bool ok = true;
            if (n > 0) {
                ok = ring_wait_warp(&S.full, loads & 1u, P.spin_limit, lane);
                ok = __syncthreads_and(ok);
                if (ok) {
                    ++loads;
                    if (tid == 0)
                        load_pending = false;
                }
            }
            Rec mine{};
            if (MODE == MODE_GREEDY) {
                float bv = -F_INF;
                int bi = -1, fl = 0;
                if (ok)
                    for (int g = tid; g < ng; g += CL_THREADS) {
                        f2 X[4];
                        const float vm = group8<E>(bt, g, n, X);
                        if (!(vm == vm) || vm == F_INF) {
                            fl = FL_T;
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
                            bi = x0 + g * 8 + e;
                        }
                    }
                warp_merge_argmax(bv, bi);
                fl = warp_or(fl);
                if (lane == 0)
                    S.wr[warp] = Rec{bv, __int_as_float(bi), 0.0f, fl, 0.0f, 0.0f, 0.0f, 0};
                __syncthreads();
                if (warp == 0) {
                    Rec r = S.wr[lane < CL_WARPS ? lane : 0];
                    float v = lane < CL_WARPS ? r.a0 : -F_INF;
                    int i = lane < CL_WARPS ? __float_as_int(r.a1) : -1;
                    int f = lane < CL_WARPS ? r.i0 : 0;
                    warp_merge_argmax<CL_WARPS>(v, i);
                    f = warp_or(f) | (ok ? 0 : FL_TIMEOUT);
                    mine = Rec{v, __int_as_float(i), 0.0f, f, 0.0f, 0.0f, 0.0f,
                               __shfl_sync(0xffffffffu, claimed, 0)};
                }
            } else {
                float mt = -F_INF, st = 0.0f, md = -F_INF, sd = 0.0f;
                int fl = 0;
                if (ok) {
                    thread_stats<E>(bt, n, tid, c, mt, st, fl, FL_T);
                    if (has_d)
                        thread_stats<E>(bd, n, tid, c, md, sd, fl, FL_D);
                }
                float Mt, Md;
                DF St, Sd;
                merge_ms<32>(mt, DF{st, 0.0f}, c, Mt, St);
                merge_ms<32>(md, DF{sd, 0.0f}, c, Md, Sd);
                fl = warp_or(fl);
                if (lane == 0)
                    S.wr[warp] = Rec{Mt, St.hi, St.lo, fl, Md, Sd.hi, Sd.lo, 0};
                __syncthreads();
                if (warp == 0) {
                    const bool in = lane < CL_WARPS;
                    const Rec r = S.wr[in ? lane : 0];
                    merge_ms<CL_WARPS>(in ? r.a0 : -F_INF, in ? DF{r.a1, r.a2} : DF{0.0f, 0.0f}, c, Mt, St);
                    merge_ms<CL_WARPS>(in ? r.b0 : -F_INF, in ? DF{r.b1, r.b2} : DF{0.0f, 0.0f}, c, Md, Sd);
                    const int f = warp_or(in ? r.i0 : 0) | (ok ? 0 : FL_TIMEOUT);
                    mine = Rec{Mt, St.hi, St.lo, f, Md, Sd.hi, Sd.lo, __shfl_sync(0xffffffffu, claimed, 0)};
                }
            }
            // this position's uniforms (word 0 accepts, word 1 samples)
            const uint4 wph = philox10((uint32_t)pos, (uint32_t)b, 0u, 0u, P.key0, P.key1);
            // ---- exchange (the slice stays in shared memory for the residual)
            const uint32_t par = round & 1u;
            if (warp == 0)
                send_rec(S, par, me, C, mine, lane);
            const bool got = __syncthreads_and(
                cl_wait(&S.xbar[par], (round >> 1) & 1u, P.spin_limit, &P.ctl[CTL_CL_ABORT], lane));
            // every lane < C holds one record; merge in rank order
            const bool in = (uint32_t)lane < C;
            const Rec r = S.rx[par][in ? lane : 0];
            int flags = warp_or(in ? r.i0 : 0);
            if (!got)
                flags |= FL_TIMEOUT;
            next_b = __shfl_sync(0xffffffffu, r.i1, 0);
            if (tid == 0 && got)
                mbar_arrive_tx(&S.xbar[par], rec_bytes);   // re-arm for round + 2
            ++round;

            int code = 0;
            bool accept = false;
            float Mt = 0.0f, Md = 0.0f;
            DF St{0.0f, 0.0f}, Sd{0.0f, 0.0f};
            int g_tok = -1;
            if (MODE == MODE_GREEDY) {
                float v = in ? r.a0 : -F_INF;
                int i = in ? __float_as_int(r.a1) : -1;
                if (C <= 8)
                    warp_merge_argmax<8>(v, i);
                else
                    warp_merge_argmax<16>(v, i);
                v = __shfl_sync(0xffffffffu, v, 0);
                i = __shfl_sync(0xffffffffu, i, 0);
                g_tok = i;
                if (flags & FL_TIMEOUT)
                    code = ST_TIMEOUT;
                else if (pos < K && !(d >= 0 && d < V))
                    code = ST_TOKEN;
                else if ((flags & FL_T) || !(v > -F_INF) || i < 0)
                    code = ST_NONFINITE;
                accept = !code && pos < K && i == d;
            } else {
                merge_ms_w((int)C, in ? r.a0 : -F_INF, in ? DF{r.a1, r.a2} : DF{0.0f, 0.0f}, c, Mt, St);
                merge_ms_w((int)C, in ? r.b0 : -F_INF, in ? DF{r.b1, r.b2} : DF{0.0f, 0.0f}, c, Md, Sd);
                // lanes of other groups hold copies of garbage: take lane 0's
                Mt = __shfl_sync(0xffffffffu, Mt, 0);
                Md = __shfl_sync(0xffffffffu, Md, 0);
                St = DF{__shfl_sync(0xffffffffu, St.hi, 0), __shfl_sync(0xffffffffu, St.lo, 0)};
                Sd = DF{__shfl_sync(0xffffffffu, Sd.hi, 0), __shfl_sync(0xffffffffu, Sd.lo, 0)};
                if (flags & FL_TIMEOUT)
                    code = ST_TIMEOUT;
                else if (pos < K && !(d >= 0 && d < V))
                    code = ST_TOKEN;
                else if ((flags & FL_T) || !(Mt > -F_INF) || !(St.hi > 0.0f))
                    code = ST_NONFINITE;
                else if (pos < K && ((flags & FL_D) || !(Md > -F_INF) || !(Sd.hi > 0.0f)))
                    code = ST_NONFINITE;
                if (!code && pos < K) {
                    zt_d = __shfl_sync(0xffffffffu, zt_d, 0);
                    zd_d = __shfl_sync(0xffffffffu, zd_d, 0);
                    int et, ed;
                    float ft, fd;
                    log2_split(St, et, ft);
                    log2_split(Sd, ed, fd);
                    // p(d) == 0 (or below the float64 range) accepts
                    const float lp = zd_d * c - Md - ((float)ed + fd);
                    if (zd_d == -F_INF || lp < -1074.5f) {
                        accept = true;
                    } else {
                        // log2(q(d) / p(d)) = (zt - zd) c - (Mt - Md) - (log2 St - log2 Sd),
                        // the large parts cancelled before rounding
                        const float X = (zt_d - zd_d) * c - ((Mt - Md) + ((float)(et - ed) + (ft - fd)));
                        accept = X >= 0.0f || u24_below(wph.x, ex2a(X));
                    }
                }
            }

            if (code) {
                if (code == ST_TIMEOUT) {
                    abort = true;
                    ab_b = b;
                }
                if (me == 0 && tid == 0) {
                    cl_error(P, b, code);
                    if (abort && claimed < P.B)
                        cl_error(P, claimed, ST_TIMEOUT);
                }
                if (abort && tid == 0)
                    atomicExch(&P.ctl[CTL_CL_ABORT], 1u);
                break;
            }
            if (pos < K && accept)
                continue;

            // ---- the sequence ends at position j = pos
            const int j = pos;
            if (MODE == MODE_GREEDY) {
                if (me == 0 && tid == 0) {
                    cl_emit(P, b, j, g_tok);
                    if (P.aux_R)
                        P.aux_R[b] = __int_as_float(0x7fc00000);
                }
                break;
            }
            const bool bonus = j == K;
            int et, ed;
            float ft, fd;
            log2_split(St, et, ft);
            log2_split(Sd, ed, fd);
            ResK kc;
            kc.Mt = Mt;
            kc.c = c;
            if (bonus) {
                kc.dLhi = kc.dLlo = 0.0f;
            } else {
                // dL = (Md - Mt) + log2 Sd - log2 St as a float pair
                DF dl = two_sum(Md, -Mt);
                dl = df_add(dl, DF{(float)(ed - et), 0.0f});
                dl = df_add(dl, DF{fd - ft, 0.0f});
                kc.dLhi = dl.hi;
                kc.dLlo = dl.lo;
            }
            const int gpw = (ng + CL_WARPS - 1) / CL_WARPS;
            const int g0 = min(ng, warp * gpw), g1 = min(ng, g0 + gpw);
            DF Rres{0.0f, 0.0f};
            bool useq = bonus;
            for (int attempt = 0; attempt < 2 && !abort; ++attempt) {
                // per-warp masses in token order, then per-CTA, then the cluster
                const DF Wm = warp_mass<E>(bt, bd, n, g0, g1, kc, bonus, useq, lane);
                if (lane == 0)
                    S.wr[warp] = Rec{Wm.hi, Wm.lo, 0.0f, 0, 0.0f, 0.0f, 0.0f, 0};
                __syncthreads();
                if (warp == 0) {
                    DF F{0.0f, 0.0f};
                    for (int i = 0; i < CL_WARPS; ++i)
                        F = df_add(F, DF{S.wr[i].a0, S.wr[i].a1});
                    send_rec(S, round & 1u, me, C, Rec{F.hi, F.lo, 0.0f, 0, 0.0f, 0.0f, 0.0f, 0}, lane);
                }
                const uint32_t rp = round & 1u;
                const bool got2 = __syncthreads_and(
                    cl_wait(&S.xbar[rp], (round >> 1) & 1u, P.spin_limit, &P.ctl[CTL_CL_ABORT], lane));
                if (tid == 0 && got2)
                    mbar_arrive_tx(&S.xbar[rp], rec_bytes);
                ++round;
                if (!got2) {
                    // gave up on a peer's record: the sequence and rank 0's
                    // claimed next one end in a timeout, and the grid winds down
                    abort = true;
                    ab_b = b;
                    if (tid == 0) {
                        if (me == 0 && claimed < P.B)
                            cl_error(P, claimed, ST_TIMEOUT);
                        atomicExch(&P.ctl[CTL_CL_ABORT], 1u);
                    }
                    break;
                }
                // cluster total and the CTA whose running sum crosses t = v R
                DF F{0.0f, 0.0f};
                for (uint32_t i = 0; i < C; ++i)
                    F = df_add(F, DF{S.rx[rp][i].a0, S.rx[rp][i].a1});
                if (!useq || bonus)
                    Rres = F;   // residual mass (kept when it is 0), or the total of q for a bonus
                if (!(F.hi > 0.0f)) {
                    if (useq)
                        break;   // cannot happen for a finite row; leaves x = -1
                    useq = true; // R <= 0: sample q_j itself
                    continue;
                }
                const DF t = u24_scale(wph.y, F);   // v R
                int rstar = -1, rlast = -1;
                DF pre{0.0f, 0.0f}, prelast{0.0f, 0.0f}, acc{0.0f, 0.0f};
                for (uint32_t i = 0; i < C; ++i) {
                    const DF Ri{S.rx[rp][i].a0, S.rx[rp][i].a1};
                    const DF nacc = df_add(acc, Ri);
                    if (Ri.hi > 0.0f) {
                        rlast = (int)i;
                        prelast = acc;
                    }
                    if (rstar < 0 && df_gt(nacc, t)) {
                        rstar = (int)i;
                        pre = acc;
                    }
                    acc = nacc;
                }
                const bool fallback = rstar < 0;
                if (fallback) {
                    rstar = rlast;
                    pre = prelast;
                }
                if (rstar == (int)me) {
                    // the warp whose running sum crosses t
                    int wstar = -1, wlast = -1;
                    DF G = pre, Gw{0.0f, 0.0f}, Glast{0.0f, 0.0f};
                    for (int i = 0; i < CL_WARPS; ++i) {
                        const DF Wi{S.wr[i].a0, S.wr[i].a1};
                        const DF nG = df_add(G, Wi);
                        if (Wi.hi > 0.0f) {
                            wlast = i;
                            Glast = G;
                        }
                        if (!fallback && wstar < 0 && df_gt(nG, t)) {
                            wstar = i;
                            Gw = G;
                        }
                        G = nG;
                    }
                    const bool wfb = wstar < 0;
                    if (wfb) {
                        wstar = wlast;
                        Gw = Glast;
                    }
                    if (warp == wstar) {
                        int xx = -1;
                        if (!wfb)
                            xx = warp_locate<E>(bt, bd, n, g0, g1, kc, bonus, useq, Gw, t, x0, lane);
                        if (xx < 0)
                            xx = warp_last_positive<E>(bt, bd, n, g0, g1, kc, bonus, useq, x0, lane);
                        if (lane == 0)
                            P.out_tokens[(size_t)b * (K + 1) + j] = xx;
                    }
                }
                break;
            }
            if (abort)
                break;
            if (me == 0 && tid == 0) {
                cl_emit(P, b, j, -1);
                if (P.aux_R) {
                    // R of the distribution the token came from: the residual
                    // mass, or the total of q_{K+1} for a bonus (normalised by St)
                    P.aux_R[b] = (Rres.hi + Rres.lo) / (St.hi + St.lo);
                }
            }
            break;
        }
        __syncthreads();   // the slices are free for the next sequence
        b = next_b;
    }

    // ---- wind down: our own copies, then the cluster (peers may still write records)
    if (tid == 0 && load_pending)
        (void)mbar_wait(&S.full, loads & 1u, DRAIN_LIMIT, nullptr);
    __syncthreads();
    cl_sync();
    if (tid == 0) {
        // a CTA that gave up marks its sequence after the cluster barrier, so
        // its error comes after anything rank 0 wrote for it (a peer may have
        // finished the sequence without the part this CTA did not do)
        if (ab_b >= 0)
            cl_error(P, ab_b, ST_TIMEOUT);
        if (abort)
            cl_status(P, ST_TIMEOUT);
        __threadfence();
        const uint32_t prev = atomicAdd(&P.ctl[CTL_CL_EXIT], 1u);
        if (prev == gridDim.x - 1) {
            __threadfence();
            if (ld_vol(&P.ctl[CTL_CL_ABORT])) {
                // sequences no cluster claimed
                for (uint32_t s = ncl + ld_vol(&P.ctl[CTL_CL_NEXT]); s < (uint32_t)P.B; ++s)
                    cl_error(P, (int)s, ST_TIMEOUT);
            }
            if (P.aux_status)
                P.aux_status[0] = (int32_t)ld_vol(&P.ctl[CTL_STATUS]);
            P.ctl[CTL_STATUS] = 0u;
            P.ctl[CTL_CL_NEXT] = 0u;
            P.ctl[CTL_CL_ABORT] = 0u;
            P.ctl[CTL_CL_EXIT] = 0u;
        }
    }
}

}  // namespace sv
