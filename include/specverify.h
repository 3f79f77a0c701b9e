/*
 * specverify.h -- C ABI of the batched speculative-decoding verification
 * library (libspecverify.so, CUDA kernels for sm_103a).
 *
 * The operation (one verification round per sequence) is the rule stated in
 *   - nextadmin.net lesson "Speculative Decoding (دیکودینگ گمانه‌زن)",
 *     § Core algorithm, steps 4-6, and § Step 1 (accept/reject), § Step 2
 *     (residual distribution), § Step 3 (one speculative step);
 *   - aiengineeringfromscratch.com Phase 10 lesson 25 "Speculative Decoding",
 *     § The exact rule and § Greedy case;
 *   - runelab.ai "Küçük bir model büyük olanı nasıl hızlandırır?", § the
 *     exact rule (points 1-3 and the bonus token);
 *   - for the shortlisted draft, the DynaSpec summary (lowest.today, "DynaSpec:
 *     Context-aware Dynamic Speculative Sampling for Large-Vocabulary Language
 *     Models"), § Abstract and § Method 3: the drafter works on a
 *     per-context shortlist, verification keeps the full vocabulary.
 * Notation: q = target distribution, p = draft distribution, d_i = drafted
 * tokens (i = 1..K), V = vocabulary size, T = temperature.
 *
 * For each sequence b, with q_i = softmax(target[b][i-1] / T) and
 * p_i = softmax(draft[b][i-1] / T) (or the given draft probabilities):
 *   for i = 1..K, left to right, accept d_i iff u_i < min(1, q_i(d_i)/p_i(d_i))
 *   (always when p_i(d_i) == 0); at the first rejection j emit a token drawn
 *   from (q_j - p_j)_+ / R_j (R_j its total; q_j itself when R_j == 0) and stop;
 *   if all K are accepted emit a bonus token drawn from q_{K+1}.
 *   T == 0 is greedy: accept d_i while d_i == argmax q_i (lowest index on
 *   ties), then emit argmax q_j at the first mismatch (argmax q_{K+1} if none).
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11) with counter
 *   (position i-1, sequence b, 0, 0) and key (seed & 0xffffffff, seed >> 32);
 *   word 0 gives u_i, word 1 gives the sampling uniform v; a word w maps to
 *   ((w >> 8) + 0.5) * 2^-24.  Sampling is inverse-CDF in ascending token
 *   order: the smallest x with sum_{y<=x} r(y) > v * R.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; rows are
 *     contiguous and row-major.  Rows whose start is 16-byte aligned (row
 *     length times element size a multiple of 16 and a 16-byte aligned base)
 *     take the bulk-copy path; other shapes are correct but slower.
 *   - `workspace` is caller-owned device scratch of at least
 *     spec_workspace_bytes(B, K, V, S) bytes.  It must be zero-filled before
 *     its first use with given sizes (B, K, V, S); a call that returns SPEC_OK
 *     leaves it ready for the next call with the same sizes.  Before reusing it
 *     with other sizes, zero-fill it again: its control words sit at offsets
 *     that depend on the sizes.  One workspace per call in flight: two calls
 *     that overlap on the GPU must not share one.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Argument errors are returned synchronously, before
 *     anything is launched.  Data errors are found on the device, in the rows
 *     the left-to-right rule examines: that sequence gets out_accept_len[b] =
 *     -code and out_tokens[b][*] = -1, and aux->device_status (if given)
 *     receives the code of one failing sequence after the kernel ends.  The
 *     device never traps.
 *   - out_tokens[b] holds the accepted draft tokens followed by one target
 *     token; out_accept_len[b] is the number of accepted draft tokens (0..K),
 *     so out_accept_len[b] + 1 tokens are emitted; unused slots are -1.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,  /* bad size, pointer, dtype, temperature or workspace size */
    SPEC_ERR_NONFINITE = 2,    /* NaN / +inf logit, all -inf row, or bad draft probability */
    SPEC_ERR_TOKEN_RANGE = 3,  /* a drafted token outside [0, V) */
    SPEC_ERR_SHORTLIST = 4,    /* shortlist not ascending and unique inside [0, V) */
    SPEC_ERR_UNSUPPORTED = 5,  /* no usable sm_103a device, or a shape the entry point does not take */
    SPEC_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed */
    SPEC_ERR_TIMEOUT = 7       /* a bounded on-device wait ran out (the kernel gave up) */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Optional per-call outputs.  Any NULL member is not written.  Asking for
 * q_draft, p_draft or row_lse makes the call evaluate every position (it then
 * reads every row), not only the positions up to the first rejection.
 * All pointers are device pointers.                                          */
typedef struct {
    float *q_draft;          /* [B][K]     q_i(d_i); NaN where row or token is invalid   */
    float *p_draft;          /* [B][K]     p_i(d_i); NaN where row or token is invalid   */
    float *residual_mass;    /* [B]        total R of the distribution the last token was
                                           drawn from (residual, or q_{K+1} for a bonus) */
    float *row_lse;          /* [B][2K+1]  log sum exp(z / T): target rows 0..K, then draft
                                           rows 0..K-1 (NaN for draft probabilities)      */
    int32_t *device_status;  /* [1]        0, or the code of one failing sequence         */
} spec_aux_t;

/* Bytes of device workspace a call with these sizes needs (S = 0 without a
 * shortlist).  Returns 0 for sizes the library rejects.                      */
size_t spec_workspace_bytes(int B, int K, int V, int S);

/* Stochastic verification; T == 0 runs the greedy rule.
 *   target_logits  [B][K+1][V]  dtype `tdt`
 *   draft          [B][K][V]    logits of dtype `tdt`, or float32 probabilities
 *                               when draft_is_probs != 0 (ddt must then be SPEC_F32)
 *   draft_tokens   [B][K]       int32
 *   out_tokens     [B][K+1]     int32;  out_accept_len [B] int32
 * Limits: B >= 1, 1 <= K <= 31, V >= 1, T finite and >= 0.                     */
spec_status_t spec_verify(const void *target_logits, spec_dtype_t tdt,
                          const void *draft, spec_dtype_t ddt, int draft_is_probs,
                          const int32_t *draft_tokens,
                          int B, int K, int V, float T, uint64_t seed,
                          int32_t *out_tokens, int32_t *out_accept_len,
                          void *workspace, size_t workspace_bytes,
                          const spec_aux_t *aux, void *stream);

/* Greedy verification (aiengineeringfromscratch.com lesson 25, § Greedy case):
 * only the target logits are read. */
spec_status_t spec_verify_greedy(const void *target_logits, spec_dtype_t tdt,
                                 const int32_t *draft_tokens, int B, int K, int V,
                                 int32_t *out_tokens, int32_t *out_accept_len,
                                 void *workspace, size_t workspace_bytes,
                                 const spec_aux_t *aux, void *stream);

/* Verification with a draft defined on a per-sequence shortlist (DynaSpec):
 *   draft_sl       [B][K][S]  logits (dtype `tdt`) or float32 probabilities over
 *                             the shortlisted tokens; p is 0 off the shortlist
 *   shortlist_idx  [B][S]     int32, strictly ascending, each in [0, V)
 * The target distribution and the residual stay over the full vocabulary.
 * A drafted token outside its shortlist has p_i(d_i) = 0 and is accepted.    */
spec_status_t spec_verify_shortlist(const void *target_logits, spec_dtype_t tdt,
                                    const void *draft_sl, spec_dtype_t ddt, int draft_is_probs,
                                    const int32_t *shortlist_idx, int S,
                                    const int32_t *draft_tokens,
                                    int B, int K, int V, float T, uint64_t seed,
                                    int32_t *out_tokens, int32_t *out_accept_len,
                                    void *workspace, size_t workspace_bytes,
                                    const spec_aux_t *aux, void *stream);

/* Verification with a shortlisted draft whose list may depend on the position
 * (DynaSpec summary, § Method 3: the position-aware budget k_c(t) sets how
 * many clusters, hence tokens, the drafter uses at draft step t; a static
 * list shared by every sequence and position, as in FR-Spec, is the same
 * layout with both strides 0).
 *   draft_sl       [B][K][S]  draft logits of dtype `tdt` (ddt == tdt); row (b, i)
 *                             holds shortlist_len[i] logits, for the tokens of
 *                             list (b, i)
 *   shortlist_idx  list (b, i) starts at shortlist_idx + b * sl_seq_stride +
 *                  i * sl_pos_stride (entries): strictly ascending, each in [0, V)
 *                  (per position: strides K*S and S; per sequence: S and 0;
 *                  shared: 0 and 0)
 *   shortlist_len  HOST array of K entry counts, each in [1, S], or NULL (all S)
 * p_i is 0 off list (b, i); the target and the residual stay over the full
 * vocabulary; a drafted token off its list has p_i(d_i) = 0 and is accepted.
 * A list that is not strictly ascending inside [0, V) is an error
 * (SPEC_ERR_SHORTLIST) at the position that uses it, found only if the rule
 * reaches that position.  Draft probabilities are not accepted here.
 * The workspace is spec_workspace_bytes(B, K, V, S).  T == 0 runs the greedy
 * rule (the draft is not read).  Served by the row-parallel kernels.         */
spec_status_t spec_verify_shortlist_pos(const void *target_logits, spec_dtype_t tdt, const void *draft_sl,
                                        spec_dtype_t ddt, const int32_t *shortlist_idx, long long sl_seq_stride,
                                        long long sl_pos_stride, const int32_t *shortlist_len, int S,
                                        const int32_t *draft_tokens, int B, int K, int V, float T, uint64_t seed,
                                        int32_t *out_tokens, int32_t *out_accept_len, void *workspace,
                                        size_t workspace_bytes, const spec_aux_t *aux, void *stream);

/* Verification with no caller workspace (the pages have no counterpart: this
 * is an interface for callers that cannot allocate device memory, or cannot
 * hold a workspace per call, e.g. code with a fixed memory plan).  Arguments
 * and results are those of spec_verify (T == 0: greedy, draft_logits may be
 * NULL) with draft logits only.
 *   Scratch: a 256-byte device array inside the library holds the kernel's
 *   control words.  It is zero when the library loads, and every call that
 *   completes leaves it zero.  The call allocates nothing; it is served by
 *   the cluster kernel alone.
 *   Limits: rows 16-byte aligned (V * element size a multiple of 16, aligned
 *   bases), one CTA's slice of a position within that kernel's shared-memory
 *   budget (about V <= 289280 bfloat16 / 144640 float32 logits with draft
 *   rows, twice that for greedy), and no q_draft / p_draft / row_lse outputs.
 *   Any other call returns SPEC_ERR_UNSUPPORTED without launching;
 *   spec_verify serves it.
 *   Overlapping calls race: all calls on a device share the scratch, so they
 *   must be ordered on the GPU (one stream, or events between streams).
 *   Every call looks up the scratch's device address with a CUDA runtime
 *   call (a host-side lookup, not a stream operation), so the address stays
 *   right after a cudaDeviceReset.  The first call on a device also loads the
 *   library's kernels there; make that first call outside any stream capture. */
spec_status_t spec_verify_static(const void *target_logits, spec_dtype_t tdt, const void *draft_logits,
                                 const int32_t *draft_tokens, int B, int K, int V, float T, uint64_t seed,
                                 int32_t *out_tokens, int32_t *out_accept_len, const spec_aux_t *aux,
                                 void *stream);

/* Fused draft-token sampler: the drafting step that precedes verification
 * (nextadmin.net lesson "Speculative Decoding", § Core algorithm step 2 and
 * § Build it, spec_step: each drafted token is drawn from the draft
 * distribution and its probability p_dist[d] is kept for the acceptance test;
 * aiengineeringfromscratch.com lesson 25, § Build it: softmax of the logits
 * divided by the temperature).
 *   draft_logits  [B][K][V]  dtype `ddt`; row (b, i) is the drafter's output at
 *                            position i of sequence b (already conditioned on
 *                            the earlier drafts)
 *   out_tokens    [B][K]     int32: d_i = the smallest x whose running sum of
 *                            softmax(z / T) in ascending token order exceeds
 *                            v * R (R the total), v = word 0 of Philox4x32-10
 *                            with counter (i, b, 1, 0) and key (seed low, seed
 *                            high), mapped by ((w >> 8) + 0.5) * 2^-24
 *   out_prob      [B][K]     float: p_i(d_i) (may be NULL)
 *   device_status [1]        set to 0, or SPEC_ERR_NONFINITE when some row has a
 *                            NaN or +inf logit or is -inf everywhere (that row
 *                            gets token -1 and probability NaN); may be NULL
 * T == 0 drafts greedily: the first index of the largest logit, probability 1.
 * Limits: B, K, V >= 1, B * K <= 2^30, V <= 2093056, T finite and >= 0.
 * No workspace; the call is asynchronous on `stream`.                         */
spec_status_t spec_draft_sample(const void *draft_logits, spec_dtype_t ddt, int B, int K, int V, float T,
                                uint64_t seed, int32_t *out_tokens, float *out_prob, int32_t *device_status,
                                void *stream);

/* KV-cache commit (and rollback) after verification (nextadmin.net lesson
 * "Speculative Decoding", § KV cache management: the verification pass
 * appends the K drafts' entries; when drafts are rejected the cache returns
 * to the accepted prefix, production systems staging the K entries and
 * committing the accepted ones; § Exercises item 4 fixes the outcome).
 *   cache       [NL][B][L][entry_bytes]  the KV cache: NL layers, capacity L
 *                                        entries per sequence, entry_bytes
 *                                        bytes per entry and layer (keys and
 *                                        values of all heads, any dtype)
 *   staged      [NL][B][K][entry_bytes]  the K new entries of the verification
 *                                        pass, or NULL when they were written in
 *                                        place at [seq_len[b], seq_len[b] + K)
 *   accept_len  [B]   spec_verify's out_accept_len (accepted drafts, or < 0
 *                     for a sequence in error)
 *   seq_len     [B]   in/out: cache lengths
 * For a = accept_len[b] >= 0: entries 0..a-1 of staged[l][b] are copied to
 * cache[l][b][seq_len[b]..] for every layer and seq_len[b] += a; the drafts'
 * other entries are dropped (rolled back).  a < 0 changes nothing.  a > K, or
 * seq_len[b] + a > L, changes nothing and sets *device_status to
 * SPEC_ERR_INVALID_ARG (device_status is set to 0 first; it may be NULL).
 * Device pointers; staged must not overlap cache.  16-byte aligned buffers
 * with entry_bytes a multiple of 16 take the vector path.  Asynchronous on
 * `stream`; two launches (one in place).  The token emitted at the rejection
 * (or the bonus token) has no entry yet: it is the next round's input.       */
spec_status_t spec_kv_commit(void *cache, const void *staged, int NL, int B, int K, int L, size_t entry_bytes,
                             const int32_t *accept_len, int32_t *seq_len, int32_t *device_status,
                             void *stream);

/* Greedy tree verification (aiengineeringfromscratch.com Phase 10 lesson 25,
 * § Tree attention verification: one target pass over a draft tree under a
 * mask where each token sees only its ancestors; the output is the longest
 * accepted prefix along any path; § Greedy case: a draft is accepted when it
 * is the target's argmax).  The stochastic multi-branch rule is not on the
 * pages and is not offered.
 *   target_logits  [B][N][V]  dtype `tdt`; row n: the target's prediction after
 *                             node n's token
 *   tree_tokens    [B][N]     int32: node n's drafted token (node 0, the root,
 *                             is the last accepted token and is not read)
 *   parent         [B][N]     int32: parent[0] == -1, parent[n] in [0, n)
 *   out_tokens     [B][N]     int32: the accepted path's drafts, then the
 *                             argmax of its last node's row; -1 after
 *   out_nodes      [B][N]     int32: the path's node indices (root excluded); -1 after
 *   out_accept_len [B]        int32: accepted drafts (the path's depth), or
 *                             -code on a data error in an examined place:
 *                             1 malformed parent array, 2 NaN / +inf / all -inf
 *                             row of an accepted node, 3 token outside [0, V)
 *                             at a child of an accepted node
 * A child is accepted iff its parent is accepted and its token equals the
 * first index of the maximum of the parent's row.  The path ends at the
 * deepest accepted node, the lowest node index among equally deep ones.
 *   workspace      device scratch of spec_tree_workspace_bytes(B, N, V) bytes
 *                  (no zero-fill needed), 16-byte aligned
 *   device_status  [1] set to 0, or the code of one failing sequence; may be NULL
 * Limits: B, N, V >= 1, N <= 2048, B * N <= 2^30, V <= 2093056.  Two launches,
 * asynchronous on `stream`.                                                   */
size_t spec_tree_workspace_bytes(int B, int N, int V);
spec_status_t spec_verify_tree_greedy(const void *target_logits, spec_dtype_t tdt, const int32_t *tree_tokens,
                                      const int32_t *parent, int B, int N, int V, int32_t *out_tokens,
                                      int32_t *out_nodes, int32_t *out_accept_len, void *workspace,
                                      size_t workspace_bytes, int32_t *device_status, void *stream);

/* Tree attention mask (the same section): mask[b][i][j] = 1 iff node j is
 * node i or one of its ancestors, else 0; uint8 [B][N][N], device pointers.
 * A malformed parent array sets *device_status to 1 (it is set to 0 first;
 * may be NULL) and leaves that row's walk cut short.  One launch.            */
spec_status_t spec_tree_mask(const int32_t *parent, int B, int N, uint8_t *mask, int32_t *device_status,
                             void *stream);

/* Philox4x32-10 words as the verification kernels draw them, for checking:
 * out[(b * P + pos) * 4 + w] = word w of Philox(counter (pos, b, tag, 0),
 * key (seed low, seed high)) for b < B, pos < P.  `out` is a device pointer of
 * B * P * 4 uint32 entries.                                                   */
spec_status_t spec_philox_words(uint64_t seed, uint32_t tag, int B, int P, uint32_t *out,
                                void *stream);

/* Number of kernels this library has launched in this process, over every
 * entry point and device: a successful spec_verify* call launches one kernel,
 * or two to four when the row-parallel kernels serve it (large stochastic
 * batches: two from 1024 rows with aligned rows, where the residual pass runs
 * inside the statistics stream); spec_draft_sample and spec_philox_words
 * launch one each, spec_kv_commit two (one in place).  For accounting;
 * thread-safe.                                                               */
uint64_t spec_launch_count(void);

/* A static description of a status code. */
const char *spec_status_string(spec_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
