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
// with no decision to wait for.  Two kernels find the first index of each
// row's maximum in parts:
//   - vg_bulk (rows 16-byte aligned, 2.5 or more rows per SM, rows of 64 KB
//     or more): one CTA per row streams it through a shared-memory ring by
//     bulk copies;
//   - vg_argmax (any rows): a CTA takes one part of one row (parts of `span`
//     tokens, several per row when the rows are few); each warp reads
//     segments of 4 x 32 16-byte vectors (every load instruction of a warp
//     covers 512 contiguous bytes), several segments in flight per lane.
// Each part is recorded and counted once per sequence; the last part of a
// sequence to count merges its rows' parts (the largest value, ties to the
// lower index) and walks the rule over the K + 1 rows, one warp lane per
// position.  With a status output, the last sequence to finish reports the
// call's status and zeroes it for the next call.  Both kernels are launched
// as programmatic dependents: the launch overlaps the end of the kernel
// before them in the stream, and they read nothing before it has finished.
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
constexpr int kMaxDevicesGreedy = 64;
constexpr int VG_TMO = 64;   // row flag: a wait on the CTA's own copies ran out (reported as a timeout)

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

// Sequence b's outputs from its rows' part records (every part recorded), by
// one warp: lane i merges the `nparts` parts of position i's row (the largest value,
// ties to the lower index) and loads the drafted token, and the walk stops at
// the first position where a check fails or the argmax differs from the
// drafted token (position K always stops it).
__device__ void g_walk(const RowsParams &P, int b, int lane, int nparts)
{
    const int K = P.K;
    bool stop = false, tok_bad = false, row_bad = false, tmo = false;
    int g = -1, d = -1;
    if (lane <= K) {
        const VrStat *pp = P.vpart + ((size_t)b * (2 * K + 1) + lane) * VR_SMAX;
        float v = -F_INF;
        int fl = 0;
#pragma unroll
        for (int q = 0; q < VR_SMAX; ++q) {
            if (q < nparts) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(pp + q));
                argmax_merge(v, g, a.x, __float_as_int(a.y));
                fl |= __float_as_int(a.w);
            }
        }
        row_bad = (fl & (VR_BAD | VG_TMO)) || g < 0;
        tmo = (fl & VG_TMO) != 0;
        if (lane < K) {
            d = __ldg(P.tokens + (size_t)b * K + lane);
            tok_bad = !(d >= 0 && d < P.V);
        }
        stop = tok_bad || row_bad || lane == K || g != d;
    }
    const int j = __ffs(__ballot_sync(0xffffffffu, stop)) - 1;   // K at the latest
    const int code = __shfl_sync(0xffffffffu,
                                 tok_bad ? (int)ST_TOKEN : (tmo ? (int)ST_TIMEOUT : (row_bad ? (int)ST_NONFINITE : 0)), j);
    const int gj = __shfl_sync(0xffffffffu, g, j);
    int32_t *out = P.out_tokens + (size_t)b * (K + 1);
    if (lane <= K)
        out[lane] = code ? -1 : (lane < j ? d : (lane == j ? gj : -1));
    if (lane == 0) {
        P.out_len[b] = code ? -code : j;
        if (code && P.aux_status)
            atomicCAS(P.ctl + CTL_STATUS, 0u, (uint32_t)code);
        if (P.aux_R)
            P.aux_R[b] = __int_as_float(0x7fc00000);
    }
}

// After a sequence's walk, with a status output: the last sequence to finish
// reports the call's status and zeroes it for the next call.
__device__ __forceinline__ void g_done(const RowsParams &P, int lane)
{
    if (lane == 0 && P.aux_status) {
        uint32_t *done = P.vctl + VC_SDONE * VC_LINE;
        if (g_atom_add(done, 1u) == (uint32_t)(P.B - 1)) {
            const uint32_t s = __ldcg(P.ctl + CTL_STATUS);
            *P.aux_status = (int32_t)s;
            P.ctl[CTL_STATUS] = 0u;
            *done = 0u;
        }
    }
}

// Warp 0 of a CTA that reduced part `part` of row (b, i): the warps' maxima
// are in sm_v / sm_i; flags are the part's VR_BAD / VG_TMO.  The part's record
// goes out, then one count per sequence over all its rows' parts: the last
// part to count walks the rule.
template <int NW>
__device__ __forceinline__ void vg_finish(const RowsParams &P, int b, int i, int part, float bv, int bi, int flags,
                                          const float *sm_v, const int *sm_i, int lane)
{
    const int K = P.K;
    bv = lane < NW ? sm_v[lane] : -F_INF;
    bi = lane < NW ? sm_i[lane] : -1;
#pragma unroll
    for (int o = 16; o; o >>= 1)
        argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
    uint32_t *seqc = P.pair + (size_t)b * (K + 1);
    uint32_t prev = 0;
    if (lane == 0) {
        P.vpart[((size_t)b * (2 * K + 1) + i) * VR_SMAX + part] = VrStat{bv, __int_as_float(bi), 0.0f, flags, 0.0f, 0, 0, 0};
        prev = g_atom_add(seqc, 1u);
    }
    if (__shfl_sync(0xffffffffu, prev, 0) != (uint32_t)((K + 1) * P.parts - 1))
        return;
    if (lane == 0)
        *seqc = 0u;   // every part has counted: ready for the next call
    __syncwarp();     // the other lanes read the records after lane 0's acquire
    g_walk(P, b, lane, P.parts);
    g_done(P, lane);
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
    pdl_wait();
    pdl_trigger();
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
    vg_finish<NW>(P, b, i, part, bv, bi, bad ? (int)VR_BAD : 0, sm_v, sm_i, lane);
}

// The same for rows that start 16-byte aligned, when the rows are many
// (2.5 or more per SM): one CTA per row, thread 0 keeps VGB_NS bulk copies of
// VGB_STAGE bytes in flight into a shared-memory ring (completion on each
// stage's mbarrier), and every thread takes the maximum of its vectors of
// each stage.  The copies keep more bytes in flight per SM than register
// loads can.  Every wait is bounded (never below OWN_WAIT_MIN hinted polls:
// they wait on the CTA's own copies); one that runs out marks the row as
// timed out, and the CTA waits for its copies still in flight before it
// leaves.
constexpr int VGB_NS = 4;
constexpr int VGB_STAGE = 16384;
template <class E, int DT>
__global__ void __launch_bounds__(DT) vg_bulk(const __grid_constant__ RowsParams P)
{
    constexpr int NW = DT / 32;
    constexpr int TPV = 16 / E::ES;                 // tokens per 16-byte vector
    constexpr int STOK = VGB_STAGE / E::ES;         // tokens per stage
    constexpr int VPT = VGB_STAGE / 16 / DT;        // vectors per thread per stage
    static_assert(VPT == 4, "a stage is four vectors per thread");
    extern __shared__ __align__(128) uint8_t vg_ring[];
    __shared__ unsigned long long full[VGB_NS];
    __shared__ float sm_v[NW];
    __shared__ int sm_i[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    const int K = P.K;
    const int r = (int)blockIdx.x;   // row r = b (K + 1) + i
    const int b = r / (K + 1), i = r - b * (K + 1);
    const uint8_t *row = static_cast<const uint8_t *>(P.target) + (size_t)r * (size_t)P.V * E::ES;
    const int V = P.V;
    const int nst = (V + STOK - 1) / STOK;
    if (tid == 0) {
        for (int q = 0; q < VGB_NS; ++q)
            mbar_init(&full[q], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int k = 0; k < VGB_NS && k < nst; ++k) {
            const uint32_t nb = (uint32_t)(min(STOK, V - k * STOK) * E::ES);
            mbar_arrive_tx(&full[k], nb);
            bulk_g2s(vg_ring + k * VGB_STAGE, row + (size_t)k * VGB_STAGE, nb, &full[k]);
        }
    }
    __syncthreads();
    float bv = -F_INF;
    int bi = -1, fl = 0;
    int k = 0;
    for (; k < nst; ++k) {
        const int q = k % VGB_NS;
        if (!__syncthreads_and(ring_wait(&full[q], (uint32_t)(k / VGB_NS) & 1u, P.spin_limit)))
            break;
        const int tok = k * STOK, n = min(STOK, V - tok);
        const uint4 *sv = reinterpret_cast<const uint4 *>(vg_ring + q * VGB_STAGE);
        uint4 v[VPT];
#pragma unroll
        for (int e = 0; e < VPT; ++e) {
            const int x = (e * DT + tid) * TPV;   // token within the stage
            v[e] = x < n ? sv[e * DT + tid] : E::neg_inf();
        }
        const float lm = E::quad_max(v);
        if (!(lm == lm) || lm == F_INF) {
            fl |= VR_BAD;
        } else if (lm > bv) {
            // the first of these tokens holding the new maximum
            int idx = -1;
#pragma unroll
            for (int e = VPT - 1; e >= 0; --e) {
                float f[TPV];
                E::unpack(v[e], f);
#pragma unroll
                for (int h = TPV - 1; h >= 0; --h)
                    if (f[h] == lm)
                        idx = tok + (e * DT + tid) * TPV + h;
            }
            bv = lm;
            bi = idx;
        }
        __syncthreads();   // every thread is done with slot q: refill it
        if (tid == 0 && k + VGB_NS < nst) {
            const int kk = k + VGB_NS;
            const uint32_t nb = (uint32_t)(min(STOK, V - kk * STOK) * E::ES);
            mbar_arrive_tx(&full[q], nb);
            bulk_g2s(vg_ring + q * VGB_STAGE, row + (size_t)kk * VGB_STAGE, nb, &full[q]);
        }
    }
    if (k < nst) {
        // a wait ran out: the copies still in flight land before the CTA leaves
        fl |= VG_TMO;
        if (tid == 0)
            for (int m = k; m < nst && m < k + VGB_NS; ++m)
                (void)mbar_wait(&full[m % VGB_NS], (uint32_t)(m / VGB_NS) & 1u, DRAIN_LIMIT, nullptr);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        argmax_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if (lane == 0) {
        sm_v[warp] = bv;
        sm_i[warp] = bi;
    }
    fl = __syncthreads_or(fl);
    if (warp != 0)
        return;
    vg_finish<NW>(P, b, i, 0, bv, bi, fl, sm_v, sm_i, lane);
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
    if (launches)
        *launches = 1;
    return launch_after(vg_argmax<E, DT, NSEG>, (int)grid, DT, 0, stream, P);
}

template <class E>
cudaError_t launch_greedy_bulk(RowsParams P, cudaStream_t stream, int *launches)
{
    constexpr int DT = 256;
    const int smem = VGB_NS * VGB_STAGE;
    static bool attr_set[kMaxDevicesGreedy] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevicesGreedy || !attr_set[dev]) {
        e = cudaFuncSetAttribute(vg_bulk<E, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDevicesGreedy)
            attr_set[dev] = true;
    }
    P.span = P.V;
    P.parts = 1;
    const long long rows = (long long)P.B * (P.K + 1);
    if (rows > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    if (launches)
        *launches = 1;
    return launch_after(vg_bulk<E, DT>, (int)rows, DT, smem, stream, P);
}

// Block size and segments in flight; SPECVERIFY_GREEDY_CFG = "threads,depth"
// picks another instantiation, for measurement.
template <class E>
cudaError_t launch_greedy_e(const RowsParams &P, cudaStream_t stream, int *launches)
{
    // rows that start 16-byte aligned: the bulk-copy kernel, unless a
    // register-load instantiation is asked for
    // many aligned rows of a full ring or more: the bulk-copy kernel, one CTA
    // per row (with fewer rows than two and a half per SM, the register-load
    // kernel's parts keep more of the GPU busy), unless an instantiation is
    // asked for
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    if (P.vec && (long long)P.V * E::ES >= (long long)VGB_NS * VGB_STAGE &&
        2LL * P.B * (P.K + 1) >= 5LL * sms && !std::getenv("SPECVERIFY_GREEDY_CFG"))
        return launch_greedy_bulk<E>(P, stream, launches);
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
