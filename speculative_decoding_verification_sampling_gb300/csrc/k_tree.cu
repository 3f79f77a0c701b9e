// k_tree.cu -- greedy tree verification and the tree attention mask.
//
// aiengineeringfromscratch.com Phase 10 lesson 25 "Speculative Decoding",
// § Tree attention verification: a draft tree is verified by one target
// forward pass under a mask that lets each token attend only to its
// ancestors, and the output is the longest accepted prefix along any path;
// § Greedy case: a drafted token is accepted when it is the target's argmax.
//
// Tree layout per sequence: N nodes, parents before children; node 0 is the
// root (the last accepted token, parent -1); node n >= 1 holds a drafted
// token and parent[n] in [0, n).  Target row n is the prediction after node n.
//
// Verification is two launches: the argmax of every node row (the draft
// sampler's greedy kernel, one CTA per row, into the workspace), then one CTA
// per sequence that applies, to every node at once, the walk in node order:
//   a child of an accepted node is accepted iff its token equals the parent
//   row's argmax; the longest accepted path ends at the deepest accepted node
//   (lowest index among equally deep ones); the emitted tokens are the path's
//   drafts and then the argmax of its last node's row.
// Only accepted nodes' rows are examined: a NaN / +inf / all -inf row there is
// an error (2), as is a token outside [0, V) at a child of an accepted node
// (3); a malformed parent array is an error (1).
#include <cstdint>
#include <cuda_runtime.h>

#include "sv_params.h"
#include "sv_launch.h"

namespace sv {
namespace {

constexpr int TW = 128;         // threads of a walk CTA
constexpr int TREE_NMAX = 2048; // nodes per tree
constexpr int TREE_KEY = 4096;  // (depth, -index) keys: depth * TREE_KEY + TREE_KEY - 1 - index

struct TreeParams {
    const int32_t *tokens;   // [B][N]
    const int32_t *parent;   // [B][N]
    const int32_t *g;        // [B][N] argmax of each node row (-1: row in error)
    int32_t *out_tokens;     // [B][N]
    int32_t *out_nodes;      // [B][N]
    int32_t *out_len;        // [B]
    int32_t *status;         // [1] or nullptr
    int B, N, V;
};

// One CTA per tree, every node at once.  A node is accepted iff every link on
// its path to the root holds (a link: the node's token lies in [0, V) and
// equals the argmax of its parent's row); a node's depth is the number of
// links on that path.  Both come from pointer jumping over the parent array
// (ceil(log2 N) rounds, double-buffered in shared memory).  The walk in node
// order that the rule describes stops at the first node in error, so the
// status is that of the lowest-numbered one:
//   - a child of an accepted node whose token lies outside [0, V) (3);
//   - an accepted node whose row is in error (2).
// The deepest accepted node (the lowest index among equally deep ones) comes
// from one atomicMax over (depth, -index), and its path is written back.
__global__ void __launch_bounds__(TW) tree_walk(const __grid_constant__ TreeParams P)
{
    __shared__ int32_t s_par[TREE_NMAX], s_tok[TREE_NMAX], s_g[TREE_NMAX];
    __shared__ int16_t s_anc[2][TREE_NMAX], s_dep[2][TREE_NMAX];
    __shared__ uint8_t s_ok[2][TREE_NMAX];
    __shared__ int s_bad, s_err, s_best;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the argmax launch's results
    const int b = blockIdx.x, N = P.N, tid = threadIdx.x;
    const size_t o = (size_t)b * N;
    if (tid == 0) {
        s_bad = 0;
        s_err = 0x7fffffff;
        s_best = TREE_KEY - 1;   // node 0 at depth 0
    }
    __syncthreads();
    for (int n = tid; n < N; n += TW) {
        const int p = __ldg(P.parent + o + n);
        s_par[n] = p;
        s_tok[n] = __ldg(P.tokens + o + n);
        s_g[n] = __ldg(P.g + o + n);
        if (n == 0 ? p != -1 : (p < 0 || p >= n))
            s_bad = 1;
        P.out_tokens[o + n] = -1;
        P.out_nodes[o + n] = -1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            P.out_len[b] = -1;
            if (P.status)
                atomicCAS(P.status, 0, 1);
        }
        return;
    }
    // round 0: each node's own link, one level up
    for (int n = tid; n < N; n += TW) {
        const int t = s_tok[n];
        s_anc[0][n] = (int16_t)(n == 0 ? 0 : s_par[n]);
        s_dep[0][n] = (int16_t)(n == 0 ? 0 : 1);
        s_ok[0][n] = n == 0 || (t >= 0 && t < P.V && t == s_g[s_par[n]]);
    }
    __syncthreads();
    int cur = 0;
    for (int step = 1; step < N; step <<= 1) {
        for (int n = tid; n < N; n += TW) {
            const int a = s_anc[cur][n];
            s_ok[cur ^ 1][n] = s_ok[cur][n] & s_ok[cur][a];
            s_dep[cur ^ 1][n] = (int16_t)(s_dep[cur][n] + s_dep[cur][a]);
            s_anc[cur ^ 1][n] = s_anc[cur][a];
        }
        __syncthreads();
        cur ^= 1;
    }
    // the first node in error, and the deepest accepted node
    int err = 0x7fffffff, best = TREE_KEY - 1;
    for (int n = tid; n < N; n += TW) {
        const bool acc = s_ok[cur][n];
        const int t = s_tok[n];
        if (n > 0 && s_ok[cur][s_par[n]] && !(t >= 0 && t < P.V))
            err = min(err, n * 4 + ST_TOKEN);
        else if (acc && s_g[n] < 0)
            err = min(err, n * 4 + ST_NONFINITE);
        if (acc)
            best = max(best, s_dep[cur][n] * TREE_KEY + (TREE_KEY - 1 - n));
    }
    if (err != 0x7fffffff)
        atomicMin(&s_err, err);
    atomicMax(&s_best, best);
    __syncthreads();
    if (tid != 0)
        return;
    if (s_err != 0x7fffffff) {
        const int code = s_err & 3;
        P.out_len[b] = -code;
        if (P.status)
            atomicCAS(P.status, 0, code);
        return;
    }
    const int bn = TREE_KEY - 1 - (s_best % TREE_KEY), d = s_best / TREE_KEY;
    for (int n = bn, k = d - 1; n > 0; n = s_par[n], --k) {
        P.out_tokens[o + k] = s_tok[n];
        P.out_nodes[o + k] = n;
    }
    P.out_tokens[o + d] = s_g[bn];
    P.out_len[b] = d;
}

// One CTA per mask row (b, i): zeros, then ones on the ancestors of i.
__global__ void __launch_bounds__(128) tree_mask_kernel(const int32_t *parent, int B, int N, uint8_t *mask,
                                                         int32_t *status)
{
    const size_t bi = blockIdx.x;
    const int b = (int)(bi / N), i = (int)(bi % N);
    uint8_t *row = mask + bi * N;
    for (int j = threadIdx.x; j < N; j += blockDim.x)
        row[j] = 0;
    __syncthreads();
    if (threadIdx.x != 0)
        return;
    const int32_t *par = parent + (size_t)b * N;
    // parents precede their children, so the walk ends within i + 1 steps
    int j = i;
    for (int steps = 0; steps <= i; ++steps) {
        row[j] = 1;
        if (j == 0) {
            if (__ldg(par) != -1 && status)
                atomicCAS(status, 0, 1);
            return;
        }
        const int p = __ldg(par + j);
        if (p < 0 || p >= j) {
            if (status)
                atomicCAS(status, 0, 1);
            return;
        }
        j = p;
    }
}

}  // namespace

int tree_max_nodes() { return TREE_NMAX; }

cudaError_t launch_tree_walk(const int32_t *tokens, const int32_t *parent, const int32_t *g, int B, int N, int V,
                             int32_t *out_tokens, int32_t *out_nodes, int32_t *out_len, int32_t *status,
                             cudaStream_t stream)
{
    TreeParams P{tokens, parent, g, out_tokens, out_nodes, out_len, status, B, N, V};
    // launched so that it may start while the argmax launch finishes (it waits
    // for that launch's results first)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(TW);
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_walk, P);
}

cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint8_t *mask, int32_t *status, cudaStream_t stream)
{
    if (status) {
        cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return e;
    }
    tree_mask_kernel<<<(unsigned)((long long)B * N), 128, 0, stream>>>(parent, B, N, mask, status);
    return cudaGetLastError();
}

}  // namespace sv
