// api.cu -- the C ABI declared in include/specverify.h: argument checks,
// workspace layout, task geometry and kernel dispatch.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>

#include "specverify.h"
#include "sv_launch.h"
#include "sv_params.h"

namespace {

// kernels launched by this library in this process (every entry point)
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
constexpr int kStageBytes = 4096;    // bytes per ring stage (matches the kernel)
constexpr int kWorkersPerSM = 16;    // worker warps per CTA, one CTA per SM (matches the kernel)
constexpr uint32_t kDefaultSpin = 1u << 22;

// entry ids: 0..3 stoch (tdt*2 + probs), 4..5 greedy (tdt), 6..9 shortlist (tdt*2 + probs)
constexpr int kEntries = 10;

struct DeviceInfo {
    bool init = false;
    bool usable = false;
    int sms = 0;
    int occ[kEntries] = {};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

sv::KernelEntry entry_for(int mode, int tdt, bool probs, int *id)
{
    if (mode == sv::MODE_GREEDY) {
        *id = 4 + tdt;
        return sv::entry_greedy(tdt);
    }
    if (mode == sv::MODE_SHORT) {
        *id = 6 + tdt * 2 + (probs ? 1 : 0);
        return sv::entry_short(tdt, probs);
    }
    *id = tdt * 2 + (probs ? 1 : 0);
    return sv::entry_stoch(tdt, probs);
}

// Current device: must be compute capability 10.3 (the build targets sm_103a).
spec_status_t device_setup(int *sms, int mode, int tdt, bool probs, sv::KernelEntry *entry, int *occ)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return SPEC_ERR_UNSUPPORTED;
    int id = 0;
    *entry = entry_for(mode, tdt, probs, &id);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ERR_CUDA;
        d.usable = (major == 10 && minor == 3);
        d.sms = n;
        d.init = true;
    }
    if (!d.usable)
        return SPEC_ERR_UNSUPPORTED;
    if (d.occ[id] == 0) {
        int o = 0;
        if (entry->occupancy(&o) != cudaSuccess || o < 1)
            return SPEC_ERR_CUDA;
        d.occ[id] = o;
    }
    *sms = d.sms;
    *occ = d.occ[id];
    return SPEC_OK;
}


// Largest shared-memory footprint per CTA for the cluster kernel: three CTAs
// (three sequences in flight) per SM at V = 128256 bf16 with clusters of 8.
constexpr uint32_t kClusterSmemMax = 72 * 1024;

// Stochastic calls with at least this many logit rows (B (2K + 1)) go to the
// row-parallel kernels: measured faster than the cluster kernel
// from B = 32, K = 7 and B = 64, K = 4 up (B = 256, K = 4: 160 us against
// 202 us); smaller calls cannot fill the GPU with rows.
constexpr long long kRowsMinRows = 256;

// Kernel choice (SPECVERIFY_KERNEL), for measurement and tests.  By default
// the dispatch in run() picks the kernel; "cluster" and "rows" skip the other
// of those two; "general" forces the chunk-scheduled kernel.
enum KernelChoice { KC_AUTO = 0, KC_GENERAL = 2, KC_ROWS = 3, KC_CLUSTER = 4 };
KernelChoice kernel_choice()
{
    const char *s = std::getenv("SPECVERIFY_KERNEL");
    if (s && std::strcmp(s, "general") == 0)
        return KC_GENERAL;
    if (s && std::strcmp(s, "rows") == 0)
        return KC_ROWS;
    if (s && std::strcmp(s, "cluster") == 0)
        return KC_CLUSTER;
    return KC_AUTO;
}
bool cluster_disabled() { return kernel_choice() != KC_AUTO && kernel_choice() != KC_CLUSTER; }

// SPECVERIFY_DEBUG=1 prints each launch's geometry to stderr.
bool debug_enabled()
{
    const char *s = std::getenv("SPECVERIFY_DEBUG");
    return s && *s && std::strcmp(s, "0") != 0;
}

// Co-resident clusters for (kernel, cluster size, shared memory), per device.
std::map<std::tuple<int, int, int, uint32_t>, int> g_max_clusters;

uint32_t spin_limit()
{
    const char *s = std::getenv("SPECVERIFY_SPIN_LIMIT");
    if (s && *s) {
        const unsigned long v = std::strtoul(s, nullptr, 10);
        if (v > 0 && v < 0xffffffffUL)
            return (uint32_t)v;
    }
    return kDefaultSpin;
}

inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

bool sizes_ok(int B, int K, int V, int S)
{
    if (B < 1 || K < 1 || K > 31 || V < 1 || V > (1 << 30) || S < 0 || S > V)
        return false;
    // task counters are 32-bit: bound the worst-case number of tasks
    const long long rows = (long long)B * (2LL * K + 1);
    const long long chunks = (long long)(V / 1024 + 1);
    return rows * chunks < (1LL << 31);
}

// Row-parallel verification (k_rows.cu): logit draft rows (or greedy), no
// shortlist.  Serves the per-position outputs too (then every row is read).
// A shortlisted draft for run_rows: the list of (b, i) is the len[i] entries at
// idx + b seq + i pos (len: host array of K entries), draft rows [B][K][S].
struct RowsShortlist {
    const int32_t *idx = nullptr;
    long long seq = 0, pos = 0;
    const int32_t *len = nullptr;
    int S = 0;
};

spec_status_t run_rows(bool greedy, const void *target, spec_dtype_t tdt, const void *draft, const int32_t *tokens,
                       int B, int K, int V, float T, uint64_t seed, int32_t *out_tokens, int32_t *out_len,
                       void *workspace, const sv::WsLayout &L, const spec_aux_t *aux, void *stream,
                       const RowsShortlist &sl = RowsShortlist(), bool probs = false)
{
    if ((long long)B * (2 * K + 1) > INT32_MAX || (long long)B * sv::rows_chunks() > INT32_MAX)
        return SPEC_ERR_UNSUPPORTED;
    const int es = tdt == SPEC_F32 ? 4 : 2;
    char *w = static_cast<char *>(workspace);
    sv::RowsParams P{};
    P.target = target;
    P.draft = greedy ? nullptr : draft;
    P.tokens = tokens;
    P.out_tokens = out_tokens;
    P.out_len = out_len;
    if (aux) {
        P.aux_q = aux->q_draft;
        P.aux_p = aux->p_draft;
        P.aux_R = aux->residual_mass;
        P.aux_lse = aux->row_lse;
        P.aux_status = aux->device_status;
    }
    P.ctl = reinterpret_cast<uint32_t *>(w + L.ctl);
    P.stat = reinterpret_cast<sv::VrStat *>(w + L.vr_stat);
    P.pair = reinterpret_cast<uint32_t *>(w + L.vr_pair);
    P.rej = reinterpret_cast<uint32_t *>(w + L.vr_rej);
    P.errc = reinterpret_cast<int32_t *>(w + L.vr_errc);
    P.rowcnt = reinterpret_cast<uint32_t *>(w + L.vr_rowcnt);
    P.vpart = reinterpret_cast<sv::VrStat *>(w + L.vr_part);
    P.segm = reinterpret_cast<sv::VrSeg *>(w + L.vr_segm);
    P.vctl = reinterpret_cast<uint32_t *>(w + L.vr_ctl);
    P.dw = reinterpret_cast<unsigned long long *>(w + L.vr_dw);
    P.jobs = reinterpret_cast<sv::VrJob *>(w + L.vr_jobs);
    P.spin_limit = spin_limit();
    P.B = B;
    P.K = K;
    P.V = V;
    P.nseg = (V + sv::rows_segment_tokens() - 1) / sv::rows_segment_tokens();
    P.nch = sv::rows_chunks();
    P.greedy = greedy ? 1 : 0;
    P.skip = (P.aux_q || P.aux_p || P.aux_lse) ? 0 : 1;
    P.vec = ((long long)V * es) % 16 == 0 && reinterpret_cast<uintptr_t>(target) % 16 == 0 &&
            (greedy || reinterpret_cast<uintptr_t>(draft) % 16 == 0);
    if (probs && !greedy) {
        // float32 probability rows, read by the residual pass in 16-byte copies
        P.probs = 1;
        P.vec = P.vec && ((long long)V * 4) % 16 == 0;
    }
    if (sl.idx && !greedy) {
        P.sl = sl.idx;
        P.sl_seq = sl.seq;
        P.sl_pos = sl.pos;
        P.S = sl.S;
        for (int i = 0; i < K; ++i)
            P.sl_len[i] = sl.len ? sl.len[i] : sl.S;
        P.lb = reinterpret_cast<int32_t *>(w + L.vr_lb);
        P.vec = P.vec && ((long long)sl.S * es) % 16 == 0;
    }
    P.c = greedy ? 1.0f : (float)(1.4426950408889634 / (double)T);
    P.key0 = (uint32_t)(seed & 0xffffffffu);
    P.key1 = (uint32_t)(seed >> 32);
    if (debug_enabled())
        std::fprintf(stderr, "specverify: rows kernels %s %s B=%d K=%d V=%d skip=%d vec=%d\n",
                     greedy ? "greedy" : "stochastic", tdt == SPEC_BF16 ? "bf16" : "f32", B, K, V, P.skip, P.vec);
    int nl = 0;
    const cudaError_t le = sv::launch_rows(P, tdt == SPEC_BF16 ? 1 : 0, static_cast<cudaStream_t>(stream), &nl);
    if (le == cudaErrorNotSupported)
        return SPEC_ERR_UNSUPPORTED;
    if (le != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add((uint64_t)nl, std::memory_order_relaxed);
    return SPEC_OK;
}

// One sequence per cluster (sv_cluster.cuh).  Applies to stochastic
// verification with draft logits and to greedy verification, when no
// per-position output is requested, rows start 16-byte aligned and one CTA's
// slice of a position fits kClusterSmemMax.  Returns SPEC_ERR_UNSUPPORTED
// (without launching) when it does not apply.
spec_status_t run_cluster(bool greedy, const void *target, spec_dtype_t tdt, const void *draft,
                          const int32_t *tokens, int B, int K, int V, float T, uint64_t seed,
                          int32_t *out_tokens, int32_t *out_len, uint32_t *ctl, const spec_aux_t *aux,
                          void *stream, bool any_choice = false)
{
    if (!any_choice && cluster_disabled())
        return SPEC_ERR_UNSUPPORTED;
    if (aux && (aux->q_draft || aux->p_draft || aux->row_lse) && !greedy)
        return SPEC_ERR_UNSUPPORTED;
    const int es = tdt == SPEC_F32 ? 4 : 2;
    if (((long long)V * es) % 16 != 0 || reinterpret_cast<uintptr_t>(target) % 16 != 0 ||
        (!greedy && reinterpret_cast<uintptr_t>(draft) % 16 != 0))
        return SPEC_ERR_UNSUPPORTED;
    const int rows = greedy ? 1 : 2;
    const uint32_t hdr = sv::cluster_header_bytes();
    int csize = 0, chunk = 0;
    uint32_t smem = 0;
    for (int cs : {8, 16}) {
        const int ch = cdiv(cdiv(V, cs), 8) * 8;
        const long long bytes = (long long)hdr + (long long)ch * es * rows;
        if (bytes <= kClusterSmemMax) {
            csize = cs;
            chunk = ch;
            smem = (uint32_t)bytes;
            break;
        }
    }
    if (!csize)
        return SPEC_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SPEC_ERR_CUDA;
    const int tix = tdt == SPEC_BF16 ? 1 : 0;
    const sv::ClusterEntry entry = sv::entry_cluster(tix, greedy);
    int maxc = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        const auto key = std::make_tuple(dev, tix * 2 + (greedy ? 1 : 0), csize, smem);
        auto it = g_max_clusters.find(key);
        if (it == g_max_clusters.end()) {
            if (entry.max_clusters(csize, smem, &maxc) != cudaSuccess)
                return SPEC_ERR_CUDA;
            g_max_clusters[key] = maxc;
        } else {
            maxc = it->second;
        }
    }
    if (maxc < 1)
        return SPEC_ERR_UNSUPPORTED;
    sv::ClusterParams P{};
    P.target = target;
    P.draft = greedy ? nullptr : draft;
    P.tokens = tokens;
    P.out_tokens = out_tokens;
    P.out_len = out_len;
    if (aux) {
        P.aux_R = aux->residual_mass;
        P.aux_status = aux->device_status;
    }
    P.ctl = ctl;
    P.B = B;
    P.K = K;
    P.V = V;
    P.chunk = chunk;
    P.c = greedy ? 1.0f : (float)(1.4426950408889634 / (double)T);
    P.key0 = (uint32_t)(seed & 0xffffffffu);
    P.key1 = (uint32_t)(seed >> 32);
    P.spin_limit = spin_limit();
    const int clusters = std::min(maxc, B);
    if (debug_enabled())
        std::fprintf(stderr, "specverify: cluster kernel %s %s B=%d K=%d V=%d: cluster %d CTAs, chunk %d, "
                     "%u B shared memory, %d co-resident clusters, %d launched\n",
                     greedy ? "greedy" : "stochastic", tdt == SPEC_BF16 ? "bf16" : "f32", B, K, V, csize, chunk,
                     smem, maxc, clusters);
    if (entry.launch(P, clusters, csize, smem, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status_t run(int mode, const void *target, spec_dtype_t tdt, const void *draft, spec_dtype_t ddt,
                  int probs, const int32_t *shortlist, int S, const int32_t *tokens, int B, int K, int V,
                  float T, uint64_t seed, int32_t *out_tokens, int32_t *out_len, void *workspace,
                  size_t workspace_bytes, const spec_aux_t *aux, void *stream)
{
    // ---- synchronous argument checks (nothing touches the GPU before these pass)
    if (!sizes_ok(B, K, V, mode == sv::MODE_SHORT ? S : 0))
        return SPEC_ERR_INVALID_ARG;
    if (mode == sv::MODE_SHORT && S < 1)
        return SPEC_ERR_INVALID_ARG;
    if (!target || !tokens || !out_tokens || !out_len || !workspace)
        return SPEC_ERR_INVALID_ARG;
    if (tdt != SPEC_F32 && tdt != SPEC_BF16)
        return SPEC_ERR_INVALID_ARG;
    if (!std::isfinite(T) || T < 0.0f)
        return SPEC_ERR_INVALID_ARG;
    if (T == 0.0f)
        mode = sv::MODE_GREEDY;
    if (mode != sv::MODE_GREEDY) {
        if (!draft)
            return SPEC_ERR_INVALID_ARG;
        if (probs ? ddt != SPEC_F32 : ddt != tdt)
            return SPEC_ERR_INVALID_ARG;
        if (mode == sv::MODE_SHORT && !shortlist)
            return SPEC_ERR_INVALID_ARG;
        const double c = 1.4426950408889634 / (double)T;
        if (!std::isfinite((float)c))
            return SPEC_ERR_INVALID_ARG;
    }
    const int S_eff = mode == sv::MODE_SHORT ? S : 0;
    const sv::WsLayout L = sv::ws_layout(B, K, V, S_eff);
    if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return SPEC_ERR_INVALID_ARG;

    int sms = 0, occ = 0;
    sv::KernelEntry entry{};
    spec_status_t st = device_setup(&sms, mode, tdt == SPEC_BF16 ? 1 : 0, probs != 0, &entry, &occ);
    if (st != SPEC_OK)
        return st;

    // shortlisted draft logits with enough rows to fill the GPU: the row-parallel
    // kernels, every position using the sequence's list
    if (mode == sv::MODE_SHORT && !probs) {
        const KernelChoice kc = kernel_choice();
        if (kc == KC_ROWS || (kc == KC_AUTO && (long long)B * (2 * K + 1) >= kRowsMinRows)) {
            RowsShortlist sl;
            sl.idx = shortlist;
            sl.seq = S;
            sl.pos = 0;
            sl.S = S;
            const spec_status_t rs = run_rows(false, target, tdt, draft, tokens, B, K, V, T, seed, out_tokens,
                                              out_len, workspace, L, aux, stream, sl);
            if (rs != SPEC_ERR_UNSUPPORTED)
                return rs;
        }
    }
    // draft probabilities with the rows' layout the stream reads: the
    // row-parallel path streams the target rows alone (same size rule as logits)
    if (mode == sv::MODE_STOCH && probs) {
        const KernelChoice kc = kernel_choice();
        if (kc == KC_ROWS || (kc == KC_AUTO && ((long long)B * (2 * K + 1) >= kRowsMinRows || B <= 2 || K >= 6))) {
            const spec_status_t rs = run_rows(false, target, tdt, draft, tokens, B, K, V, T, seed, out_tokens,
                                              out_len, workspace, L, aux, stream, RowsShortlist(), true);
            if (rs != SPEC_ERR_UNSUPPORTED)
                return rs;
        }
    }
    if (mode == sv::MODE_GREEDY || (mode == sv::MODE_STOCH && !probs)) {
        const bool full = aux && (aux->q_draft || aux->p_draft || aux->row_lse);
        const KernelChoice kc = kernel_choice();
        // greedy: every target row's argmax in one launch (any batch, any row alignment)
        if (kc == KC_ROWS || (kc == KC_AUTO && mode == sv::MODE_GREEDY)) {
            const spec_status_t rs = run_rows(mode == sv::MODE_GREEDY, target, tdt, draft, tokens, B, K, V, T, seed,
                                              out_tokens, out_len, workspace, L, aux, stream);
            if (rs != SPEC_ERR_UNSUPPORTED)
                return rs;
        }
        // stochastic calls with enough rows to fill the GPU: the row-parallel
        // kernels (they also serve the per-position outputs); and the smallest
        // batches or long drafts, where reading every row at once beats the
        // cluster kernel's one position at a time (B = 1, K = 4 bf16: 39 us
        // against 53 us; B = 8, K = 8: 51 us against 64 us; B = 8, K = 4 stays
        // with the cluster kernel, 43 us against 45 us)
        // and small calls whose rows all fit the shared memory of the GPU's
        // resident CTAs
        const int es = tdt == SPEC_BF16 ? 2 : 4;
        const bool aligned = ((long long)V * es) % 16 == 0 && reinterpret_cast<uintptr_t>(target) % 16 == 0 &&
                             reinterpret_cast<uintptr_t>(draft) % 16 == 0;
        if (kc == KC_AUTO && mode == sv::MODE_STOCH &&
            ((long long)B * (2 * K + 1) >= kRowsMinRows || B <= 2 || K >= 6 ||
             (aligned && sv::rows_resident_fits(B, K, V, tdt == SPEC_BF16 ? 1 : 0)))) {
            const spec_status_t rs = run_rows(false, target, tdt, draft, tokens, B, K, V, T, seed, out_tokens,
                                              out_len, workspace, L, aux, stream);
            if (rs != SPEC_ERR_UNSUPPORTED)
                return rs;
        }
        if (!(full && mode != sv::MODE_GREEDY)) {
            uint32_t *ctl = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + L.ctl);
            const spec_status_t cs = run_cluster(mode == sv::MODE_GREEDY, target, tdt, draft, tokens, B, K, V, T,
                                                 seed, out_tokens, out_len, ctl, aux, stream);
            if (cs != SPEC_ERR_UNSUPPORTED)
                return cs;
        }
    }

    sv::Params P{};
    const bool greedy = mode == sv::MODE_GREEDY;
    const bool is_probs = !greedy && probs != 0;
    P.target = target;
    P.draft = greedy ? nullptr : draft;
    P.shortlist = mode == sv::MODE_SHORT ? shortlist : nullptr;
    P.tokens = tokens;
    P.B = B;
    P.K = K;
    P.V = V;
    P.S = S_eff;
    P.Vd = mode == sv::MODE_SHORT ? S : V;
    const double Tsafe = greedy ? 1.0 : (double)T;
    P.cd = 1.4426950408889634 / Tsafe;
    P.c = (float)P.cd;
    P.invT = 1.0 / Tsafe;
    P.key0 = (uint32_t)(seed & 0xffffffffu);
    P.key1 = (uint32_t)(seed >> 32);
    P.out_tokens = out_tokens;
    P.out_len = out_len;
    if (aux) {
        P.aux_q = greedy ? nullptr : aux->q_draft;
        P.aux_p = greedy ? nullptr : aux->p_draft;
        P.aux_R = aux->residual_mass;
        P.aux_lse = greedy ? nullptr : aux->row_lse;
        P.aux_status = aux->device_status;
    }
    P.full = (P.aux_q || P.aux_p || P.aux_lse) ? 1 : 0;

    char *w = static_cast<char *>(workspace);
    P.ctl = reinterpret_cast<uint32_t *>(w + L.ctl);
    P.state = reinterpret_cast<unsigned long long *>(w + L.state);
    P.res_rec = reinterpret_cast<sv::ResRec *>(w + L.res_rec);
    P.pair_cnt = reinterpret_cast<uint32_t *>(w + L.pair_cnt);
    P.res_cnt = reinterpret_cast<uint32_t *>(w + L.res_cnt);
    P.fin = reinterpret_cast<int32_t *>(w + L.fin);
    P.errres = reinterpret_cast<int32_t *>(w + L.errres);
    P.errcode = reinterpret_cast<int32_t *>(w + L.errcode);
    P.terminal = reinterpret_cast<int32_t *>(w + L.terminal);
    P.gtok = reinterpret_cast<int32_t *>(w + L.gtok);
    P.dec = reinterpret_cast<sv::Dec *>(w + L.dec);
    P.part = reinterpret_cast<sv::Partial *>(w + L.part);
    P.seg = reinterpret_cast<sv::SegMass *>(w + L.seg);
    P.sl_lb = reinterpret_cast<int32_t *>(w + L.sl_lb);

    // ---- task geometry
    P.es_t = tdt == SPEC_F32 ? 4 : 2;
    P.es_d = is_probs ? 4 : P.es_t;
    P.se_t = kStageBytes / P.es_t;
    P.se_d = kStageBytes / P.es_d;
    const bool draft_stats = !greedy && !is_probs;
    // stats units: one stage of one row each
    P.nct = cdiv(V, P.se_t);
    P.ncd = draft_stats ? cdiv(P.Vd, P.se_d) : 0;
    P.npt = P.nct + P.ncd;
    P.n_stats = (uint32_t)((long long)K * B * P.npt + (long long)B * P.nct);
    // a residual stage holds the same tokens of the target row and, at a
    // rejection over the full vocabulary, of the draft row
    const int res_es = P.es_t + ((mode == sv::MODE_STOCH) ? P.es_d : 0);
    P.rse = (kStageBytes / res_es) / 256 * 256;
    P.rd_off = P.rse * P.es_t;
    const long long grid_max = (long long)sms * occ;
    const long long grid =
        std::min<long long>(grid_max, std::max<long long>(1, cdiv(P.n_stats, 2 * kWorkersPerSM)));
    P.workers = (uint32_t)(grid * kWorkersPerSM);
    const long long res_stages = cdiv(V, P.rse);
    P.rspt = (int)std::max<long long>(1, std::min<long long>(3, (long long)B * res_stages / ((long long)P.workers * 4)));
    P.ncr = cdiv(V, (long long)P.rspt * P.rse);
    P.nseg = L.nseg;
    P.n_res = greedy ? 0u : (uint32_t)((long long)B * P.ncr);
    // first batches: about a sixth of the units, at most 16 per worker
    P.g0 = (uint32_t)std::max<long long>(1, std::min<long long>(16, (long long)P.n_stats / (6LL * P.workers)));
    P.first_units = std::min<uint32_t>(P.n_stats, P.g0 * P.workers);
    P.spin_limit = spin_limit();
    P.bulk_t = (reinterpret_cast<uintptr_t>(target) % 16 == 0) && ((long long)V * P.es_t) % 16 == 0;
    P.bulk_d = !greedy && (reinterpret_cast<uintptr_t>(draft) % 16 == 0) &&
               ((long long)P.Vd * P.es_d) % 16 == 0;

    if (entry.launch(P, (int)grid, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_workspace_bytes(int B, int K, int V, int S)
{
    if (!sizes_ok(B, K, V, S))
        return 0;
    return sv::ws_layout(B, K, V, S).total;
}

spec_status_t spec_verify(const void *target_logits, spec_dtype_t tdt, const void *draft, spec_dtype_t ddt,
                          int draft_is_probs, const int32_t *draft_tokens, int B, int K, int V, float T,
                          uint64_t seed, int32_t *out_tokens, int32_t *out_accept_len, void *workspace,
                          size_t workspace_bytes, const spec_aux_t *aux, void *stream)
{
    return run(sv::MODE_STOCH, target_logits, tdt, draft, ddt, draft_is_probs, nullptr, 0, draft_tokens, B, K,
               V, T, seed, out_tokens, out_accept_len, workspace, workspace_bytes, aux, stream);
}

spec_status_t spec_verify_greedy(const void *target_logits, spec_dtype_t tdt, const int32_t *draft_tokens,
                                 int B, int K, int V, int32_t *out_tokens, int32_t *out_accept_len,
                                 void *workspace, size_t workspace_bytes, const spec_aux_t *aux, void *stream)
{
    return run(sv::MODE_GREEDY, target_logits, tdt, nullptr, tdt, 0, nullptr, 0, draft_tokens, B, K, V, 0.0f,
               0, out_tokens, out_accept_len, workspace, workspace_bytes, aux, stream);
}

spec_status_t spec_verify_shortlist(const void *target_logits, spec_dtype_t tdt, const void *draft_sl,
                                    spec_dtype_t ddt, int draft_is_probs, const int32_t *shortlist_idx, int S,
                                    const int32_t *draft_tokens, int B, int K, int V, float T, uint64_t seed,
                                    int32_t *out_tokens, int32_t *out_accept_len, void *workspace,
                                    size_t workspace_bytes, const spec_aux_t *aux, void *stream)
{
    if (S < 1)
        return SPEC_ERR_INVALID_ARG;
    return run(sv::MODE_SHORT, target_logits, tdt, draft_sl, ddt, draft_is_probs, shortlist_idx, S,
               draft_tokens, B, K, V, T, seed, out_tokens, out_accept_len, workspace, workspace_bytes, aux,
               stream);
}

spec_status_t spec_verify_shortlist_pos(const void *target_logits, spec_dtype_t tdt, const void *draft_sl,
                                        spec_dtype_t ddt, const int32_t *shortlist_idx, long long sl_seq_stride,
                                        long long sl_pos_stride, const int32_t *shortlist_len, int S,
                                        const int32_t *draft_tokens, int B, int K, int V, float T, uint64_t seed,
                                        int32_t *out_tokens, int32_t *out_accept_len, void *workspace,
                                        size_t workspace_bytes, const spec_aux_t *aux, void *stream)
{
    if (!sizes_ok(B, K, V, S) || S < 1 || S > V || sl_seq_stride < 0 || sl_pos_stride < 0)
        return SPEC_ERR_INVALID_ARG;
    if (!target_logits || !draft_sl || !shortlist_idx || !draft_tokens || !out_tokens || !out_accept_len ||
        !workspace)
        return SPEC_ERR_INVALID_ARG;
    if ((tdt != SPEC_F32 && tdt != SPEC_BF16) || ddt != tdt || !std::isfinite(T) || T < 0.0f)
        return SPEC_ERR_INVALID_ARG;
    if (shortlist_len)
        for (int i = 0; i < K; ++i)
            if (shortlist_len[i] < 1 || shortlist_len[i] > S)
                return SPEC_ERR_INVALID_ARG;
    if (T == 0.0f)   // greedy: the draft is not read
        return run(sv::MODE_GREEDY, target_logits, tdt, nullptr, tdt, 0, nullptr, 0, draft_tokens, B, K, V, T,
                   seed, out_tokens, out_accept_len, workspace, workspace_bytes, aux, stream);
    if (!std::isfinite((float)(1.4426950408889634 / (double)T)))
        return SPEC_ERR_INVALID_ARG;
    const sv::WsLayout L = sv::ws_layout(B, K, V, S);
    if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return SPEC_ERR_INVALID_ARG;
    RowsShortlist sl;
    sl.idx = shortlist_idx;
    sl.seq = sl_seq_stride;
    sl.pos = sl_pos_stride;
    sl.len = shortlist_len;
    sl.S = S;
    return run_rows(false, target_logits, tdt, draft_sl, draft_tokens, B, K, V, T, seed, out_tokens,
                    out_accept_len, workspace, L, aux, stream, sl);
}

// Verification without a caller workspace.  Callers that cannot allocate, or
// cannot hold a workspace per call in flight, use it. Examples: code that
// runs where device allocation is not allowed, or that keeps a fixed memory
// plan.  Its scratch is the 256-byte static array in k_cluster.cu (the
// cluster kernel's control block), so calls share it and must not overlap on
// the GPU.  Only the cluster kernel's shapes are served; any other shape
// returns SPEC_ERR_UNSUPPORTED without launching.
spec_status_t spec_verify_static(const void *target_logits, spec_dtype_t tdt, const void *draft_logits,
                                 const int32_t *draft_tokens, int B, int K, int V, float T, uint64_t seed,
                                 int32_t *out_tokens, int32_t *out_accept_len, const spec_aux_t *aux,
                                 void *stream)
{
    if (!sizes_ok(B, K, V, 0) || !target_logits || !draft_tokens || !out_tokens || !out_accept_len)
        return SPEC_ERR_INVALID_ARG;
    if (tdt != SPEC_F32 && tdt != SPEC_BF16)
        return SPEC_ERR_INVALID_ARG;
    if (!std::isfinite(T) || T < 0.0f)
        return SPEC_ERR_INVALID_ARG;
    const bool greedy = T == 0.0f;
    if (!greedy) {
        if (!draft_logits)
            return SPEC_ERR_INVALID_ARG;
        const double c = 1.4426950408889634 / (double)T;
        if (!std::isfinite((float)c))
            return SPEC_ERR_INVALID_ARG;
    }
    if (aux && (aux->q_draft || aux->p_draft || aux->row_lse))
        return SPEC_ERR_UNSUPPORTED;   // per-position outputs need the chunk-scheduled kernel and its workspace
    int sms = 0, occ = 0;
    sv::KernelEntry entry{};
    spec_status_t st = device_setup(&sms, greedy ? sv::MODE_GREEDY : sv::MODE_STOCH,
                                    tdt == SPEC_BF16 ? 1 : 0, false, &entry, &occ);
    if (st != SPEC_OK)
        return st;
    // the scratch's device address on the current device, looked up on every
    // call: a host-side lookup, no stream operation, and never stale (a
    // cudaDeviceReset reloads the module at another address)
    uint32_t *ctl = nullptr;
    if (sv::static_scratch_address(&ctl) != cudaSuccess || !ctl)
        return SPEC_ERR_CUDA;
    return run_cluster(greedy, target_logits, tdt, draft_logits, draft_tokens, B, K, V, T, seed, out_tokens,
                       out_accept_len, ctl, aux, stream, true);
}

spec_status_t spec_philox_words(uint64_t seed, uint32_t tag, int B, int P, uint32_t *out, void *stream)
{
    if (B < 1 || P < 1 || !out || (long long)B * P > (1LL << 28))
        return SPEC_ERR_INVALID_ARG;
    if (sv::launch_philox_words((uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32), tag, B, P, out,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status_t spec_draft_sample(const void *draft_logits, spec_dtype_t ddt, int B, int K, int V, float T,
                                uint64_t seed, int32_t *out_tokens, float *out_prob, int32_t *device_status,
                                void *stream)
{
    if (!draft_logits || !out_tokens || B < 1 || K < 1 || V < 1 || (ddt != SPEC_F32 && ddt != SPEC_BF16))
        return SPEC_ERR_INVALID_ARG;
    if (!(T >= 0.0f) || !std::isfinite(T) || (long long)B * K > (1LL << 30))
        return SPEC_ERR_INVALID_ARG;
    if (V > sv::draft_max_v())
        return SPEC_ERR_UNSUPPORTED;
    if (sv::launch_draft_sample(draft_logits, ddt == SPEC_BF16 ? 1 : 0, B, K, V, T, seed, out_tokens, out_prob,
                                device_status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status_t spec_kv_commit(void *cache, const void *staged, int NL, int B, int K, int L, size_t entry_bytes,
                             const int32_t *accept_len, int32_t *seq_len, int32_t *device_status, void *stream)
{
    if (!cache || !accept_len || !seq_len || NL < 1 || B < 1 || K < 1 || L < 1 || entry_bytes < 1)
        return SPEC_ERR_INVALID_ARG;
    const unsigned long long W = entry_bytes;
    // the cache (NL B L W bytes) within 2^48 bytes, so every offset fits 64 bits
    if ((double)NL * (double)B * (double)L * (double)W > 281474976710656.0)
        return SPEC_ERR_INVALID_ARG;
    const unsigned long long per = 256ULL * 64ULL;
    if ((unsigned long long)NL * B * ((K * W + per - 1) / per) > 0x7fffffffULL)
        return SPEC_ERR_UNSUPPORTED;
    int launches = 0;
    if (sv::launch_kv_commit(cache, staged, NL, B, K, L, (long long)W, accept_len, seq_len, device_status,
                             static_cast<cudaStream_t>(stream), &launches) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add((uint64_t)launches, std::memory_order_relaxed);
    return SPEC_OK;
}

size_t spec_tree_workspace_bytes(int B, int N, int V)
{
    if (B < 1 || N < 1 || V < 1 || N > sv::tree_max_nodes() || (long long)B * N > (1LL << 30))
        return 0;
    return ((size_t)B * N * 4 + 255) & ~(size_t)255;
}

spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t tdt, const int32_t *tree_tokens,
                                      const int32_t *parent, int B, int N, int V, int32_t *out_tokens,
                                      int32_t *out_nodes, int32_t *out_accept_len, void *workspace,
                                      size_t workspace_bytes, int32_t *device_status, void *stream)
{
    if (!target_logits || !tree_tokens || !parent || !out_tokens || !out_nodes || !out_accept_len || !workspace)
        return SPEC_ERR_INVALID_ARG;
    if (tdt != SPEC_F32 && tdt != SPEC_BF16)
        return SPEC_ERR_INVALID_ARG;
    const size_t need = spec_tree_workspace_bytes(B, N, V);
    if (need == 0 || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return SPEC_ERR_INVALID_ARG;
    if (V > sv::draft_max_v())
        return SPEC_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (device_status && cudaMemsetAsync(device_status, 0, sizeof(int32_t), st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    int32_t *g = static_cast<int32_t *>(workspace);
    // the argmax of every node row: the draft sampler's greedy kernel over B * N rows
    if (sv::launch_draft_sample(target_logits, tdt == SPEC_BF16 ? 1 : 0, B, N, V, 0.0f, 0, g, nullptr, nullptr,
                                st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (sv::launch_tree_walk(tree_tokens, parent, g, B, N, V, out_tokens, out_nodes, out_accept_len, device_status,
                             st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status_t spec_tree_mask(const int32_t *parent, int B, int N, uint8_t *mask, int32_t *device_status,
                             void *stream)
{
    if (!parent || !mask || B < 1 || N < 1 || (long long)B * N > 0x7fffffffLL ||
        (double)B * (double)N * (double)N > 281474976710656.0)
        return SPEC_ERR_INVALID_ARG;
    if (sv::launch_tree_mask(parent, B, N, mask, device_status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

uint64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *spec_status_string(spec_status_t status)
{
    switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_NONFINITE: return "non-finite logit, all -inf row, or bad draft probability";
    case SPEC_ERR_TOKEN_RANGE: return "draft token outside [0, V)";
    case SPEC_ERR_SHORTLIST: return "shortlist not strictly ascending inside [0, V)";
    case SPEC_ERR_UNSUPPORTED: return "no usable sm_103a device";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_TIMEOUT: return "on-device wait ran out";
    }
    return "unknown status";
}

}  // extern "C"
