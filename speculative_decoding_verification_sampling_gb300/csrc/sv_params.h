// sv_params.h -- launch parameters shared by the host launcher and the
// verification kernels (plain C++ types only).
#pragma once
#include <cstddef>
#include <cstdint>

namespace sv {

enum Mode { MODE_STOCH = 0, MODE_GREEDY = 1, MODE_SHORT = 2 };

// Status codes; the same values as spec_status_t.
enum Status { ST_OK = 0, ST_NONFINITE = 2, ST_TOKEN = 3, ST_SHORTLIST = 4, ST_TIMEOUT = 7 };

// Words of the control block at the start of the workspace.
// Words 5..7 belong to the cluster kernel (next sequence to claim, CTAs that
// have finished, abort flag); both kernels leave every word zeroed.
enum Ctl { CTL_STATS_NEXT = 0, CTL_RES_TICKET = 1, CTL_RES_COUNT = 2, CTL_EXIT = 3, CTL_STATUS = 4,
           CTL_CL_NEXT = 5, CTL_CL_EXIT = 6, CTL_CL_ABORT = 7, CTL_WORDS = 8 };

// Partial result of one stats task (one chunk of one row):
//   logits: m = max raw logit of the chunk, s = sum 2^((x - m) * c) over the chunk;
//   greedy: m = max raw logit and its lowest index.
// flag bit 0: NaN or +inf seen; bit 1: shortlist entry out of range or out of order.
struct Partial {
    float m;
    int flag;
    float s_hi;   // s = s_hi + s_lo (a float pair; greedy: s_hi holds the index bits)
    float s_lo;
};

// Residual mass r and target mass q of one 256-token segment.
struct SegMass {
    float r, q;
};

// A sequence published for its residual pass: b1 = sequence + 1 (0 while the
// slot is unpublished), j = position of the emitted target token (-1 when the
// sequence ended with a data error), rc = its Dec.  Written before b1.
struct alignas(16) ResRec {
    int32_t b1, j, pad0, pad1;
    float rc[4];
};

// Per (sequence, position) quantities the residual pass needs, in float32:
// Mt = max target logit, Lt2 = log2 of the target sum, dL = log2(Z_draft / Z_target)
// split into a high and a low float.
struct Dec {
    float Mt, Lt2, dLhi, dLlo;
};

struct Params {
    // inputs (device)
    const void *target;        // [B][K+1][V]
    const void *draft;         // [B][K][Vd]  (Vd = V, or S with a shortlist)
    const int32_t *shortlist;  // [B][S] or nullptr
    const int32_t *tokens;     // [B][K]
    int B, K, V, Vd, S;
    float c;                   // log2(e) / T
    double cd;                 // log2(e) / T in float64
    double invT;               // 1 / T
    uint32_t key0, key1;       // Philox key (seed low, seed high)
    int full;                  // evaluate every position (per-position outputs requested)

    // outputs (device)
    int32_t *out_tokens;       // [B][K+1]
    int32_t *out_len;          // [B]
    float *aux_q, *aux_p, *aux_R, *aux_lse;
    int32_t *aux_status;

    // workspace (device)
    uint32_t *ctl;                 // [CTL_WORDS]
    unsigned long long *state;     // [B]  decided positions (low word) | accepted positions (high word)
    ResRec *res_rec;               // [B]  residual slots in publication order
    uint32_t *pair_cnt;            // [B][K+1] finished stats tasks per position
    uint32_t *res_cnt;             // [B]  finished residual tasks per sequence
    int32_t *fin;                  // [B]  1 once the sequence's outputs are written
    int32_t *errres;               // [B]  1 when the residual pass met a bad draft probability
    int32_t *errcode;              // [B][K+1] data error found at the position (0 = none)
    int32_t *terminal;             // [B]  position of the emitted target token (-1 on error)
    int32_t *gtok;                 // [B][K+1] greedy argmax per position
    Dec *dec;                      // [B][K+1]
    Partial *part;                 // [B][K+1][npt]
    SegMass *seg;                  // [B][nseg] residual mass and target mass per 256-token segment
    int32_t *sl_lb;                // [B][nseg+1] first shortlist entry at or after token 256*t

    // task geometry
    int es_t, es_d;                // element sizes of target and draft rows
    int se_t, se_d;                // elements per stats stage
    int nct, ncd, npt;             // stats units (stages) per target row, per draft row, per position
    int rse, rd_off;               // elements per residual stage; byte offset of its draft part
    int rspt, ncr;                 // stages per residual task, residual tasks per sequence
    int nseg;                      // 256-token segments per target row
    uint32_t n_stats, n_res;       // total stats units, total residual tasks
    uint32_t workers;              // worker warps in the grid
    uint32_t g0, first_units;      // units in each worker's first batch, and in all first batches
    uint32_t spin_limit;           // bound on every on-device wait loop
    int bulk_t, bulk_d;            // rows eligible for bulk copies (16-byte aligned)
};

// Launch parameters of the cluster kernel (one sequence per thread-block
// cluster; CTA r of a cluster owns tokens [r*chunk, (r+1)*chunk) of every row).
struct ClusterParams {
    const void *target;        // [B][K+1][V]
    const void *draft;         // [B][K][V] draft logits; nullptr for greedy
    const int32_t *tokens;     // [B][K]
    int32_t *out_tokens;       // [B][K+1]
    int32_t *out_len;          // [B]
    float *aux_R;              // [B] or nullptr
    int32_t *aux_status;       // [1] or nullptr
    uint32_t *ctl;             // [CTL_WORDS] at the start of the workspace
    int B, K, V;
    int chunk;                 // tokens of a row per CTA (a multiple of 8)
    float c;                   // log2(e) / T
    uint32_t key0, key1;       // Philox key (seed low, seed high)
    uint32_t spin_limit;       // bound on every on-device wait loop
};


// Workspace layout for (B, K, V, S); every array starts 256-byte aligned.
// Row-parallel verification (k_rows.cu): the statistics of one logit row.
//   m        reference floor(max * c) in log2 units (greedy: the maximum)
//   s_hi/lo  sum of 2^(x c - m) as a float pair (greedy: s_hi holds the
//            argmax index's bits)
//   flags    VR_BAD (NaN or +inf seen), VR_SKIP (not computed: not needed)
//   zd       the logit at the drafted token of the row's position
struct alignas(16) VrStat {
    float m, s_hi, s_lo;
    int flags;
    float zd;
    int pad0, pad1, pad2;
};
enum { VR_BAD = 1, VR_SKIP = 2, VR_HASD = 4, VR_SLBAD = 8 };
// The row-parallel call's counters (words VC_* * VC_LINE of vctl): parts
// claimed by vr_stream, timeout (a bounded wait ran out), vr_sample CTAs done
// (the last one zeroes the counters), residual jobs posted, residual chunks
// claimed, sequences ended.
enum { VC_CLAIM = 0, VC_TIMEOUT = 1, VC_SDONE = 2, VC_JOBS = 3, VC_TICKETS = 4, VC_ENDED = 5, VC_N = 6 };
constexpr int VC_LINE = 32;
constexpr int VR_SMAX = 16;   // most parts a row is split into
struct VrSeg {
    float r, q;   // residual and target masses of one 256-token segment, relative to 2^Mt
};
// A residual job of vr_stream: sequence b (stored as b + 1, 0 until written)
// ended at position j; the coefficients of its row pair j.
struct alignas(16) VrJob {
    int b1, j;
    float Mt, dLhi, dLlo;
    int pad0, pad1, pad2;
};

struct RowsParams {
    const void *target;        // [B][K+1][V]
    const void *draft;         // [B][K][V] logits; nullptr for greedy
    const int32_t *tokens;     // [B][K]
    int32_t *out_tokens;       // [B][K+1]
    int32_t *out_len;          // [B]
    float *aux_q, *aux_p, *aux_R, *aux_lse;
    int32_t *aux_status;
    uint32_t *ctl;             // control words (status)
    VrStat *stat;              // [B][2K+1]: target rows 0..K, then draft rows 0..K-1
    uint32_t *pair;            // [B][K+1] rows of a position done
    uint32_t *rowcnt;          // [B][2K+1] parts of a row done
    VrStat *vpart;             // [B][2K+1][VR_SMAX] statistics of the parts of a row
    uint32_t *rej;             // [B] bit i: position i decided against (or in error)
    int32_t *errc;             // [B][K+1] status of a decision in error (valid where rej is set)
    VrSeg *segm;             // [B][nseg]
    int B, K, V, nseg, nch;
    int pos, npos;             // vr_stats: the positions [pos, pos + npos) this launch streams
    // shortlisted draft (sl != nullptr): the draft row of (b, i) holds sl_len[i]
    // logits for the tokens sl[b sl_seq + i sl_pos + s] (ascending); draft rows
    // are [B][K][S]; lb[(b K + i)][t] is the first list entry >= 256 t
    const int32_t *sl;
    long long sl_seq, sl_pos;
    int S;
    int sl_len[32];
    int32_t *lb;               // [B][K][nseg + 1]
    int parts, span;           // vr_stats: parts per row, tokens per part (a multiple of 8)
    int greedy, skip, vec;
    // draft probabilities (float32 [B][K][V], probs != 0): only target rows
    // are streamed; p_i(d_i) is read where a position is decided, the row p_j
    // by the residual pass
    int probs;
    float c;
    uint32_t key0, key1;
    // the call's counters, each on its own 128-byte line (index VC_* * 32)
    uint32_t *vctl;
    uint32_t spin_limit;
    // vr_stream's residual pass (fused != 0): per sequence the decided
    // positions (low 32 bits) and the positions that end it (high 32 bits);
    // the posted jobs; chunks per sequence and stages per chunk
    unsigned long long *dw;
    VrJob *jobs;
    int fused, rnch, rcs;
};

struct WsLayout {
    size_t ctl, state, res_rec, pair_cnt, res_cnt, fin, errres,
        vr_pair, vr_rej, vr_rowcnt, vr_ctl, vr_dw, vr_jobs, errcode, terminal, gtok, dec, part, seg, sl_lb,
        vr_stat, vr_errc, vr_part, vr_segm, vr_lb, total;
    size_t reset_end;   // [ctl, reset_end) holds what a call must find zeroed
    int npt_max, nseg;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Stats chunks are at least 1024 elements (one 4 KB stage of float32), so this
// bounds the number of partials any chunking chooses.
inline WsLayout ws_layout(int B, int K, int V, int S)
{
    WsLayout w{};
    const size_t Bz = (size_t)B, P = (size_t)K + 1;
    const int Vd = S > 0 ? S : V;
    w.nseg = (V + 255) / 256;
    w.npt_max = (V + 1023) / 1024 + (Vd + 1023) / 1024;
    size_t o = 0;
    w.ctl = o;      o = align256(o + 8 * sizeof(uint32_t));
    w.state = o;    o = align256(o + Bz * 8);
    w.res_rec = o;  o = align256(o + Bz * sizeof(ResRec));
    w.pair_cnt = o; o = align256(o + Bz * P * 4);
    w.res_cnt = o;  o = align256(o + Bz * 4);
    w.fin = o;      o = align256(o + Bz * 4);
    w.errres = o;   o = align256(o + Bz * 4);
    w.vr_pair = o;  o = align256(o + Bz * P * 4);
    w.vr_rej = o;   o = align256(o + Bz * 4);
    w.vr_rowcnt = o; o = align256(o + Bz * (2 * P - 1) * 4);
    w.vr_ctl = o;   o = align256(o + VC_N * VC_LINE * 4);
    w.vr_dw = o;    o = align256(o + Bz * 8);
    w.vr_jobs = o;  o = align256(o + Bz * sizeof(VrJob));
    w.reset_end = o;
    w.errcode = o;  o = align256(o + Bz * P * 4);
    w.terminal = o; o = align256(o + Bz * 4);
    w.gtok = o;     o = align256(o + Bz * P * 4);
    w.dec = o;      o = align256(o + Bz * P * sizeof(Dec));
    w.part = o;     o = align256(o + Bz * P * (size_t)w.npt_max * sizeof(Partial));
    w.seg = o;      o = align256(o + Bz * (size_t)w.nseg * sizeof(SegMass));
    w.sl_lb = o;    o = align256(o + (S > 0 ? Bz * (size_t)(w.nseg + 1) * 4 : 0));
    w.vr_stat = o;  o = align256(o + Bz * (2 * P - 1) * sizeof(VrStat));
    w.vr_errc = o;  o = align256(o + Bz * P * 4);
    w.vr_part = o;  o = align256(o + Bz * (2 * P - 1) * (size_t)VR_SMAX * sizeof(VrStat));
    w.vr_segm = o;  o = align256(o + Bz * (size_t)w.nseg * sizeof(VrSeg));
    w.vr_lb = o;    o = align256(o + (S > 0 ? Bz * (P - 1) * (size_t)(w.nseg + 1) * 4 : 0));
    w.total = o;
    return w;
}

}  // namespace sv
