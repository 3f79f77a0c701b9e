// k_draft.cu -- fused draft-token sampler.
//
// The drafting step before verification (nextadmin.net lesson "Speculative
// Decoding", § Core algorithm step 2 and § Build it, spec_step: each drafted
// token d is drawn from the draft distribution and p_dist[d] is kept;
// aiengineeringfromscratch.com lesson 25, § Build it: the distribution is the
// softmax of the logits divided by the temperature).  For row (b, i) of the
// draft logits: d_i = the smallest x whose running sum of softmax(z / T) in
// ascending token order exceeds v * R, v = word 0 of Philox4x32-10 with counter
// (i, b, 1, 0); the row also yields p_i(d_i).  T == 0 takes the first argmax.
//
// One CTA per row, one pass over HBM:
//   - each warp owns segments of 4 * 32 16-byte vectors of contiguous tokens
//     (1024 bfloat16 or 512 float32 tokens); lane l reads vector l of each
//     quarter, so every load instruction of a warp covers 512 contiguous bytes;
//   - a segment's reference ref = floor(max * c) (log2 units) and its mass
//     sum 2^(x c - ref) go to shared memory, so segment masses are in token
//     order; the next segment's loads are in flight while one is reduced;
//   - the row's total is the exact power-of-two rescaling of the segment
//     masses to the largest reference; a block scan over them finds the
//     segment whose running sum crosses v * R;
//   - one warp reads that segment again (from L2) and locates the token.
// The block has 128, 256 or 512 threads, chosen by occupancy: preferably one
// with every row of the call resident at once, then the most threads.
#include "sv_cluster.cuh"
#include "sv_launch.h"

#include <algorithm>

namespace sv {
namespace {

struct DraftParams {
    const void *draft;      // [rows][V]
    int rows, K, V;
    float c;                // log2(e) / T
    uint32_t key0, key1;
    int greedy;
    int vec;                // rows start 16-byte aligned
    int32_t *out_tokens;    // [rows]
    float *out_prob;        // [rows] or nullptr
    int32_t *status;        // [1] or nullptr
};

constexpr int DQ = 4;   // vectors per lane per segment

// Tokens [x0, x0 + TPV) of a row as one 16-byte vector (TPV = 16 / element
// size); tokens at or past V read as -inf.
template <class E>
__device__ __forceinline__ uint4 fetch_vec(const DraftParams &P, const uint8_t *row, int x0)
{
    constexpr int TPV = 16 / E::ES;
    if (P.vec && x0 + TPV <= P.V)
        return __ldg(reinterpret_cast<const uint4 *>(row + (size_t)x0 * E::ES));
    uint32_t w[4];
    if constexpr (E::ES == 2) {
        const uint16_t *h = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = x0 + 2 * k < P.V ? (uint32_t)__ldg(h + x0 + 2 * k) : 0xff80u;
            const uint32_t hi = x0 + 2 * k + 1 < P.V ? (uint32_t)__ldg(h + x0 + 2 * k + 1) : 0xff80u;
            w[k] = lo | (hi << 16);
        }
    } else {
        const uint32_t *f = reinterpret_cast<const uint32_t *>(row);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = x0 + k < P.V ? __ldg(f + x0 + k) : 0xff800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sum of 2^(x c - ref) over one vector, in a fixed order (the locate pass
// repeats it exactly).
template <class E>
__device__ __forceinline__ float vec_mass(const uint4 &v, f2 cc, f2 nref)
{
    if constexpr (E::ES == 2) {
        f2 e[4];
#pragma unroll
        for (int p = 0; p < 4; ++p)
            e[p] = ex2x2(fma2(E::pair(v, p), cc, nref));
        float lo, hi;
        upk(add2(add2(e[0], e[2]), add2(e[1], e[3])), lo, hi);
        return lo + hi;
    } else {
        f2 e[2];
#pragma unroll
        for (int p = 0; p < 2; ++p)
            e[p] = ex2x2(fma2(E::pair(v, p), cc, nref));
        float lo, hi;
        upk(add2(e[0], e[1]), lo, hi);
        return lo + hi;
    }
}

__device__ __forceinline__ void draft_error(const DraftParams &P, int r)
{
    P.out_tokens[r] = -1;
    if (P.out_prob)
        P.out_prob[r] = __int_as_float(0x7fc00000);
    if (P.status)
        atomicCAS(P.status, 0, (int)ST_NONFINITE);
}

template <class E, int DT>
__global__ void __launch_bounds__(DT) draft_sample_kernel(const __grid_constant__ DraftParams P)
{
    // a kernel launched after this one (the tree walk) may start launching
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int DWARPS = DT / 32;
    constexpr int TPV = 16 / E::ES;    // tokens per 16-byte vector
    constexpr int QT = 32 * TPV;       // tokens per quarter of a segment (one load per lane)
    constexpr int GT = DQ * QT;        // tokens per segment
    constexpr int CT = DWARPS * GT;    // tokens per step of the CTA
    extern __shared__ __align__(16) float2 dseg[];   // [nseg]: (reference, mass) per segment
    __shared__ float red_f[DWARPS];
    __shared__ int red_i[DWARPS];
    __shared__ DF red_df[DWARPS];
    __shared__ int s_seg, s_fb;
    __shared__ DF s_before;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x;
    const int b = r / P.K, i = r % P.K;
    const uint8_t *row = static_cast<const uint8_t *>(P.draft) + (size_t)r * P.V * E::ES;
    const int nsteps = (P.V + CT - 1) / CT;
    const int nseg = nsteps * DWARPS;
    const float c = P.c;

    // this lane's four vectors of segment (step g, this warp)
    auto load_seg = [&](int g, uint4 *v) {
        const int x = g * CT + warp * GT + lane * TPV;
#pragma unroll
        for (int q = 0; q < DQ; ++q)
            v[q] = fetch_vec<E>(P, row, x + q * QT);
    };

    if (P.greedy) {
        // first index of the largest logit (ties to the lowest index)
        float bv = -F_INF;
        int bi = -1;
        bool bad = false;
        auto step = [&](int g, const uint4 *v) {
            const float lm = E::quad_max(v);
            if (!(lm == lm) || lm == F_INF) {
                bad = true;
            } else if (lm > bv) {
                const int x = g * CT + warp * GT + lane * TPV;
                int idx = -1;
#pragma unroll
                for (int q = DQ - 1; q >= 0; --q) {
                    float f[TPV];
                    E::unpack(v[q], f);
#pragma unroll
                    for (int j = TPV - 1; j >= 0; --j)
                        if (f[j] == lm)
                            idx = x + q * QT + j;
                }
                bv = lm;
                bi = idx;
            }
        };
        // two segments in flight; each buffer is refilled right after its use
        uint4 A[DQ], Bv[DQ];
        load_seg(0, A);
        if (nsteps > 1)
            load_seg(1, Bv);
        for (int g = 0; g < nsteps; g += 2) {
            step(g, A);
            if (g + 2 < nsteps)
                load_seg(g + 2, A);
            if (g + 1 < nsteps) {
                step(g + 1, Bv);
                if (g + 3 < nsteps)
                    load_seg(g + 3, Bv);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
            argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
        if (lane == 0) {
            red_f[warp] = bv;
            red_i[warp] = bi;
        }
        bad = __syncthreads_or(bad);
        if (tid == 0) {
            for (int w = 1; w < DWARPS; ++w)
                argmax_merge(bv, bi, red_f[w], red_i[w]);
            if (bad || bi < 0) {
                draft_error(P, r);
            } else {
                P.out_tokens[r] = bi;
                if (P.out_prob)
                    P.out_prob[r] = 1.0f;
            }
        }
        return;
    }

    // ---- pass 1: segment references and masses, in token order
    bool bad = false;
    {
        const f2 cc = pk(c, c);
        auto step = [&](int g, const uint4 *v) {
            const float lm = E::quad_max(v);
            bad |= !(lm == lm) || lm == F_INF;
            const float wm = warp_maxf(lm);
            const float ref = wm > -F_INF ? floorf(wm * c) : -F_INF;
            float ls = 0.0f;
            if (ref > -F_INF && ref < F_INF) {
                const f2 nref = pk(-ref, -ref);
#pragma unroll
                for (int q = 0; q < DQ; ++q)
                    ls += vec_mass<E>(v[q], cc, nref);
            }
            const float ws = warp_sumf(ls);
            if (lane == 0)
                dseg[g * DWARPS + warp] = make_float2(ref, ws);
        };
        uint4 A[DQ], Bv[DQ];
        load_seg(0, A);
        if (nsteps > 1)
            load_seg(1, Bv);
        for (int g = 0; g < nsteps; g += 2) {
            step(g, A);
            if (g + 2 < nsteps)
                load_seg(g + 2, A);
            if (g + 1 < nsteps) {
                step(g + 1, Bv);
                if (g + 3 < nsteps)
                    load_seg(g + 3, Bv);
            }
        }
    }
    bad = __syncthreads_or(bad);
    // the largest reference
    float M = -F_INF;
    for (int s = tid; s < nseg; s += DT)
        M = fmaxf(M, dseg[s].x);
    M = warp_maxf(M);
    if (lane == 0)
        red_f[warp] = M;
    __syncthreads();
    M = red_f[0];
#pragma unroll
    for (int w = 1; w < DWARPS; ++w)
        M = fmaxf(M, red_f[w]);
    if (bad || !(M > -F_INF) || M == F_INF) {
        if (tid == 0)
            draft_error(P, r);
        return;
    }

    // ---- the total and the crossing segment: a block scan over the segment
    //      masses rescaled to 2^M (each thread sums a run of consecutive segments)
    const int per = (nseg + DT - 1) / DT;
    const int s0 = min(nseg, tid * per), s1 = min(nseg, s0 + per);
    DF own{0.0f, 0.0f};
    for (int s = s0; s < s1; ++s) {
        const float2 g = dseg[s];
        if (g.x > -F_INF)
            own = df_add(own, df_scale_pow2(DF{g.y, 0.0f}, g.x - M));
    }
    const DF wincl = warp_incl_scan_df(own, lane);
    DF wexcl{__shfl_up_sync(0xffffffffu, wincl.hi, 1), __shfl_up_sync(0xffffffffu, wincl.lo, 1)};
    if (lane == 0)
        wexcl = DF{0.0f, 0.0f};
    if (lane == 31)
        red_df[warp] = wincl;
    if (tid == 0) {
        s_seg = -1;
        s_fb = 0;
    }
    __syncthreads();
    DF wpre{0.0f, 0.0f}, total{0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < DWARPS; ++w) {
        if (w == warp)
            wpre = total;
        total = df_add(total, red_df[w]);
    }
    const DF incl = df_add(wpre, wincl), excl = df_add(wpre, wexcl);
    const uint4 wd = philox10((uint32_t)i, (uint32_t)b, 1u, 0u, P.key0, P.key1);
    const DF thr = u24_scale(wd.x, total);   // v R
    if (df_gt(incl, thr) && !df_gt(excl, thr)) {
        // this thread's run holds the crossing: walk it with the same sums
        DF G = excl;
        for (int s = s0; s < s1; ++s) {
            const float2 g = dseg[s];
            const DF m = g.x > -F_INF ? df_scale_pow2(DF{g.y, 0.0f}, g.x - M) : DF{0.0f, 0.0f};
            const DF nG = df_add(G, m);
            if (df_gt(nG, thr) && m.hi > 0.0f) {
                s_seg = s;
                s_before = G;
                break;
            }
            G = nG;
        }
    }
    __syncthreads();
    if (s_seg < 0) {
        // rounding left no crossing: the last segment with mass
        int last = -1;
        for (int s = tid; s < nseg; s += DT)
            if (dseg[s].y > 0.0f && dseg[s].x > -F_INF)
                last = s;
        last = warp_maxi(last);
        if (lane == 0)
            red_i[warp] = last;
        __syncthreads();
        if (tid == 0) {
            int l = red_i[0];
            for (int w = 1; w < DWARPS; ++w)
                l = max(l, red_i[w]);
            s_seg = l;
            s_fb = 1;
        }
        __syncthreads();
    }
    if (warp != 0)
        return;

    // ---- pass 2 (one warp): the token inside the segment, in token order
    const int seg = s_seg;
    const int xs = (seg / DWARPS) * CT + (seg % DWARPS) * GT;   // the segment's first token
    const float ref = dseg[seg].x;
    const f2 cc = pk(c, c), nref = pk(-ref, -ref);
    uint4 vv[DQ];
    float m[DQ];
#pragma unroll
    for (int q = 0; q < DQ; ++q) {
        vv[q] = fetch_vec<E>(P, row, xs + q * QT + lane * TPV);
        m[q] = vec_mass<E>(vv[q], cc, nref);
    }
    int tok = -1;
    float ztok = 0.0f;
    if (!s_fb) {
        // the threshold in units of 2^ref, relative to the segment's start
        const DF rel = df_add(thr, DF{-s_before.hi, -s_before.lo});
        const float tr = (rel.hi + rel.lo) * __int_as_float(((int)(M - ref) + 127) << 23);
        float run = 0.0f;
#pragma unroll
        for (int q = 0; q < DQ; ++q) {
            if (tok >= 0)
                break;
            float in = m[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, in, o);
                if (lane >= o)
                    in += u;
            }
            in += run;
            float ex = __shfl_up_sync(0xffffffffu, in, 1);
            if (lane == 0)
                ex = run;
            const unsigned bal = __ballot_sync(0xffffffffu, in > tr && m[q] > 0.0f);
            if (bal) {
                const int L = __ffs(bal) - 1;
                if (lane == L) {
                    float f[TPV];
                    E::unpack(vv[q], f);
                    float cum = ex;
#pragma unroll
                    for (int j = 0; j < TPV; ++j) {
                        const float e = ex2a(fmaf(f[j], c, -ref));
                        cum += e;
                        if (tok < 0 && cum > tr && e > 0.0f) {
                            tok = xs + q * QT + L * TPV + j;
                            ztok = f[j];
                        }
                    }
                }
                tok = __shfl_sync(0xffffffffu, tok, L);
                ztok = __shfl_sync(0xffffffffu, ztok, L);
                if (tok < 0)
                    break;   // rounding inside the vector: the fallback below
            }
            run = __shfl_sync(0xffffffffu, in, 31);
        }
    }
    if (tok < 0) {
        // the last token of the segment with a positive weight
        int lk = -1;
        float lz = 0.0f;
#pragma unroll
        for (int q = 0; q < DQ; ++q) {
            float f[TPV];
            E::unpack(vv[q], f);
#pragma unroll
            for (int j = 0; j < TPV; ++j)
                if (ex2a(fmaf(f[j], c, -ref)) > 0.0f)
                    lk = xs + q * QT + lane * TPV + j, lz = f[j];
        }
        tok = warp_maxi(lk);
        const unsigned ob = __ballot_sync(0xffffffffu, lk == tok && lk >= 0);
        ztok = __shfl_sync(0xffffffffu, lz, ob ? __ffs(ob) - 1 : 0);
    }
    if (lane == 0) {
        if (tok < 0) {
            draft_error(P, r);
        } else {
            P.out_tokens[r] = tok;
            if (P.out_prob)
                P.out_prob[r] = ex2a(fmaf(ztok, c, -M)) / (total.hi + total.lo);
        }
    }
}

template <class E, int DT>
cudaError_t launch_draft_dt(const DraftParams &P, cudaStream_t stream)
{
    constexpr int CT = (DT / 32) * DQ * 32 * (16 / E::ES);
    const int nsteps = (P.V + CT - 1) / CT;
    const size_t smem = (size_t)nsteps * (DT / 32) * sizeof(float2);
    auto kern = draft_sample_kernel<E, DT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<P.rows, DT, smem, stream>>>(P);
    return cudaGetLastError();
}

// Bytes in flight grow with the threads working on the rows.  Score a block
// size by the threads it keeps resident (by the kernel's occupancy), first by
// whether every row of the call is resident at once.
template <class E, int DT>
long long draft_score(int sms, int rows)
{
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, draft_sample_kernel<E, DT>, DT, 0) != cudaSuccess)
        return -1;
    const long long slots = (long long)sms * occ;
    return (slots >= rows ? (1LL << 40) : 0LL) + std::min<long long>(slots, rows) * DT;
}
template <class E>
cudaError_t launch_draft(const DraftParams &P, cudaStream_t stream)
{
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    const long long s512 = draft_score<E, 512>(sms, P.rows), s256 = draft_score<E, 256>(sms, P.rows),
                    s128 = draft_score<E, 128>(sms, P.rows);
    if (s512 >= s256 && s512 >= s128)
        return launch_draft_dt<E, 512>(P, stream);
    if (s256 >= s128)
        return launch_draft_dt<E, 256>(P, stream);
    return launch_draft_dt<E, 128>(P, stream);
}

}  // namespace

// Largest vocabulary: the segment table (8 bytes per segment of 512 or more
// tokens) stays far below the shared-memory limit.
int draft_max_v() { return 2093056; }

cudaError_t launch_draft_sample(const void *draft, int tdt, int B, int K, int V, float T, uint64_t seed,
                                int32_t *out_tokens, float *out_prob, int32_t *status, cudaStream_t stream)
{
    DraftParams P{};
    P.draft = draft;
    P.rows = B * K;
    P.K = K;
    P.V = V;
    P.greedy = T == 0.0f ? 1 : 0;
    P.c = P.greedy ? 1.0f : (float)(1.4426950408889634 / (double)T);
    P.key0 = (uint32_t)(seed & 0xffffffffu);
    P.key1 = (uint32_t)(seed >> 32);
    const int es = tdt == 0 ? 4 : 2;
    P.vec = ((long long)V * es) % 16 == 0 && reinterpret_cast<uintptr_t>(draft) % 16 == 0;
    P.out_tokens = out_tokens;
    P.out_prob = out_prob;
    P.status = status;
    if (status) {
        cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return e;
    }
    return tdt == 0 ? launch_draft<F32>(P, stream) : launch_draft<BF16>(P, stream);
}

}  // namespace sv
