// k_greedy_rows.cu -- greedy verification (T = 0) in one launch.
//
// The rule (aiengineeringfromscratch.com lesson 25, § Greedy case; the bonus
// of nextadmin.net lesson "Speculative Decoding", § Core algorithm step 6):
// g_i = the first index of the largest target logit of position i; accept d_i
// while g_i == d_i; at the first mismatch emit g_i and stop; if all K match,
// emit g_K.  Draft rows are not read.
//
// Every target row is needed up to the first mismatch, and the batches this
// serves fit in about one wave of the GPU, so every row is read, all at once,
// with no decision to wait for:
//   - a CTA takes one part of one row (rows [B][K+1], parts of `span` tokens)
//     and finds the first index of its maximum: each warp reads segments of
//     4 x 32 16-byte vectors (every load instruction of a warp covers 512
//     contiguous bytes), several segments in flight per lane;
//   - the last part of a row to finish merges the parts' results (the
//     largest value, ties to the lower index) and records the row;
//   - the last row of a sequence to finish walks the rule over the sequence's
//     K + 1 rows and writes its outputs, one warp lane per position; the last
//     sequence to finish reports the call's status and zeroes the counters for
//     the next call.
// Errors follow the rule's order at the positions it reaches: the drafted
// token (outside [0, V)), then the row (NaN or +inf, or -inf everywhere).
#include "sv_cluster.cuh"
#include "sv_launch.h"

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace sv {
namespace {

constexpr int GQ = 4;   // vectors per lane per segment

__device__ __forceinline__ uint32_t g_atom_add(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Tokens [x0, x0 + TPV) of a row as one 16-byte vector, -inf at or past t1.
template <class E>
__device__ __forceinline__ uint4 g_fetch(const uint8_t *row, int x0, int t1, bool vec)
{
    constexpr int TPV = 16 / E::ES;
    if (vec && x0 + TPV <= t1)
        return __ldg(reinterpret_cast<const uint4 *>(row + (size_t)x0 * E::ES));
    uint32_t w[4];
    if constexpr (E::ES == 2) {
        const uint16_t *h = reinterpret_cast<const uint16_t *>(row);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = x0 + 2 * k < t1 ? (uint32_t)__ldg(h + x0 + 2 * k) : 0xff80u;
            const uint32_t hi = x0 + 2 * k + 1 < t1 ? (uint32_t)__ldg(h + x0 + 2 * k + 1) : 0xff80u;
            w[k] = lo | (hi << 16);
        }
    } else {
        const uint32_t *f = reinterpret_cast<const uint32_t *>(row);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = x0 + k < t1 ? __ldg(f + x0 + k) : 0xff800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Sequence b's outputs from its rows' argmax records (every row recorded), by
// one warp: lane i loads position i's record and drafted token, and the walk
// stops at the first position where a check fails or the argmax differs from
// the drafted token (position K always stops it).
__device__ void g_walk(const RowsParams &P, int b, int lane)
{
    const int K = P.K;
    bool stop = false, tok_bad = false, row_bad = false;
    int g = -1, d = -1;
    if (lane <= K) {
        const VrStat *st = P.stat + (size_t)b * (2 * K + 1);
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(st + lane));
        g = __float_as_int(a.y);
        row_bad = (__float_as_int(a.w) & VR_BAD) || g < 0;
        if (lane < K) {
            d = __ldg(P.tokens + (size_t)b * K + lane);
            tok_bad = !(d >= 0 && d < P.V);
        }
        stop = tok_bad || row_bad || lane == K || g != d;
    }
    const int j = __ffs(__ballot_sync(0xffffffffu, stop)) - 1;   // K at the latest
    const int code = __shfl_sync(0xffffffffu, tok_bad ? (int)ST_TOKEN : (row_bad ? (int)ST_NONFINITE : 0), j);
    const int gj = __shfl_sync(0xffffffffu, g, j);
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    if (lane <= K)
        out[lane] = code ? -1 : (lane < j ? d : (lane == j ? gj : -1));
    if (lane == 0) {
        P.out_len[b] = code ? -code : j;
        if (code)
            atomicCAS(P.ctl + CTL_STATUS, 0u, (uint32_t)code);
        if (P.aux_R)
            P.aux_R[b] = __int_as_float(0x7fc00000);
    }
}

template <class E, int DT, int NSEG>
__global__ void __launch_bounds__(DT) vg_argmax(const __grid_constant__ RowsParams P)
{
    constexpr int NW = DT / 32;
    constexpr int TPV = 16 / E::ES;   // tokens per 16-byte vector
    constexpr int QT = 32 * TPV;      // tokens of one load instruction of a warp
    constexpr int GT = GQ * QT;       // tokens per segment (one warp)
    constexpr int CT = NW * GT;       // tokens per step of the CTA
    __shared__ float sm_v[NW];
    __shared__ int sm_i[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = P.K;
    const int r = (int)blockIdx.x / P.parts, part = (int)blockIdx.x % P.parts;   // row r = b (K + 1) + i
    const int b = r / (K + 1), i = r - b * (K + 1);
    const uint8_t *row = static_cast<const uint8_t *>(P.target) + (size_t)r * (size_t)P.V * E::ES;
    const int t0 = min(P.V, part * P.span), t1 = min(P.V, t0 + P.span);
    const int nsteps = (t1 - t0 + CT - 1) / CT;
    const bool vec = P.vec != 0;

    auto load_seg = [&](int g, uint4 *v) {
        const int x = t0 + g * CT + warp * GT + lane * TPV;
#pragma unroll
        for (int q = 0; q < GQ; ++q)
            v[q] = g_fetch<E>(row, x + q * QT, t1, vec);
    };
    float bv = -F_INF;
    int bi = -1;
    bool bad = false;
    auto step = [&](int g, const uint4 *v) {
        const float lm = E::quad_max(v);
        if (!(lm == lm) || lm == F_INF) {
            bad = true;
        } else if (lm > bv) {
            // the first of this lane's tokens holding the new maximum
            const int x = t0 + g * CT + warp * GT + lane * TPV;
            int idx = -1;
#pragma unroll
            for (int q = GQ - 1; q >= 0; --q) {
                float f[TPV];
                E::unpack(v[q], f);
#pragma unroll
                for (int e = TPV - 1; e >= 0; --e)
                    if (f[e] == lm)
                        idx = x + q * QT + e;
            }
            bv = lm;
            bi = idx;
        }
    };
    // NSEG segments in flight; each buffer is refilled right after its use
    // (static buffer indices: rotating the registers would wait on every load)
    uint4 buf[NSEG][GQ];
#pragma unroll
    for (int k = 0; k < NSEG; ++k)
        if (k < nsteps)
            load_seg(k, buf[k]);
    for (int g0 = 0; g0 < nsteps; g0 += NSEG) {
#pragma unroll
        for (int k = 0; k < NSEG; ++k) {
            const int g = g0 + k;
            if (g < nsteps) {
                step(g, buf[k]);
                if (g + NSEG < nsteps)
                    load_seg(g + NSEG, buf[k]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if (lane == 0) {
        sm_v[warp] = bv;
        sm_i[warp] = bi;
    }
    bad = __syncthreads_or(bad);
    if (warp != 0)
        return;
    // ---- warp 0: the part's result, then (last part) the row's, then (last
    //      row) the sequence's outputs, then (last sequence) the call's status
    bv = lane < NW ? sm_v[lane] : -F_INF;
    bi = lane < NW ? sm_i[lane] : -1;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
    const size_t srow = (size_t)b * (2 * K + 1) + i;   // the row's record (target rows 0..K)
    int fl = bad ? (int)VR_BAD : 0;
    if (P.parts > 1) {
        // the last part of the row to finish merges every part's result
        VrStat *pp = P.vpart + srow * VR_SMAX;
        uint32_t prev = 0;
        if (lane == 0) {
            pp[part] = VrStat{bv, __int_as_float(bi), 0.0f, fl, 0.0f, 0, 0, 0};
            prev = g_atom_add(P.rowcnt + srow, 1u);
        }
        if (__shfl_sync(0xffffffffu, prev, 0) != (uint32_t)(P.parts - 1))
            return;
        if (lane == 0)
            P.rowcnt[srow] = 0u;   // every part has counted: ready for the next call
        bv = -F_INF;
        bi = -1;
        fl = 0;
        if (lane < P.parts) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(pp + lane));
            bv = a.x;
            bi = __float_as_int(a.y);
            fl = __float_as_int(a.w);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
            fl |= __shfl_xor_sync(0xffffffffu, fl, o);
        }
    }
    // the last row of the sequence to finish walks the rule
    uint32_t *seqc = P.pair + (size_t)b * (K + 1);
    uint32_t prev = 0;
    if (lane == 0) {
        P.stat[srow] = VrStat{bv, __int_as_float(bi), 0.0f, fl, 0.0f, 0, 0, 0};
        prev = g_atom_add(seqc, 1u);
    }
    if (__shfl_sync(0xffffffffu, prev, 0) != (uint32_t)K)
        return;
    if (lane == 0)
        *seqc = 0u;
    g_walk(P, b, lane);
    // the last sequence reports the status and zeroes it
    if (lane == 0) {
        uint32_t *done = P.vctl + VC_SDONE * VC_LINE;
        if (g_atom_add(done, 1u) == (uint32_t)(P.B - 1)) {
            const uint32_t s = __ldcg(P.ctl + CTL_STATUS);
            if (P.aux_status)
                *P.aux_status = (int32_t)s;
            P.ctl[CTL_STATUS] = 0u;
            *done = 0u;
        }
    }
}

template <class E, int DT, int NSEG>
cudaError_t launch_greedy_t(RowsParams P, cudaStream_t stream, int *launches)
{
    int dev = 0, sms = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, vg_argmax<E, DT, NSEG>, DT, 0);
    if (e != cudaSuccess)
        return e;
    // parts per row: one while every row fits the resident CTAs (a part per
    // CTA, long enough for its loads to stream); more only when the rows are
    // too few to fill the GPU, with parts of at least 16384 tokens
    const long long rows = (long long)P.B * (P.K + 1);
    const long long slots = (long long)sms * std::max(occ, 1);
    int S = (int)std::min<long long>(VR_SMAX, std::max<long long>(1, slots / rows));
    S = std::max(1, std::min(S, P.V / 16384));
    if (const char *ev = std::getenv("SPECVERIFY_GREEDY_PARTS"))
        S = std::max(1, std::min(VR_SMAX, std::atoi(ev)));
    P.span = ((P.V + S - 1) / S + 7) / 8 * 8;
    P.parts = (P.V + P.span - 1) / P.span;
    const long long grid = rows * P.parts;
    if (grid > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    vg_argmax<E, DT, NSEG><<<(unsigned)grid, DT, 0, stream>>>(P);
    if (launches)
        *launches = 1;
    return cudaGetLastError();
}

// Block size and segments in flight; SPECVERIFY_GREEDY_CFG = "threads,depth"
// picks another instantiation, for measurement.
template <class E>
cudaError_t launch_greedy_e(const RowsParams &P, cudaStream_t stream, int *launches)
{
    int dt = 256, depth = 2;
    if (const char *ev = std::getenv("SPECVERIFY_GREEDY_CFG")) {
        dt = std::atoi(ev);
        if (const char *c = std::strchr(ev, ','))
            depth = std::atoi(c + 1);
    }
    if (dt == 512 && depth == 2)
        return launch_greedy_t<E, 512, 2>(P, stream, launches);
    if (dt == 512 && depth == 3)
        return launch_greedy_t<E, 512, 3>(P, stream, launches);
    if (dt == 256 && depth == 3)
        return launch_greedy_t<E, 256, 3>(P, stream, launches);
    if (dt == 256 && depth == 4)
        return launch_greedy_t<E, 256, 4>(P, stream, launches);
    if (dt == 128 && depth == 4)
        return launch_greedy_t<E, 128, 4>(P, stream, launches);
    return launch_greedy_t<E, 256, 2>(P, stream, launches);
}

}  // namespace

cudaError_t launch_greedy_rows(const RowsParams &P, int tdt, cudaStream_t stream, int *launches)
{
    return tdt == 0 ? launch_greedy_e<F32>(P, stream, launches) : launch_greedy_e<BF16>(P, stream, launches);
}

}  // namespace sv
