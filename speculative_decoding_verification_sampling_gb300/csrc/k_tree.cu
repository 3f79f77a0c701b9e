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
// per sequence that walks the nodes in order:
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

__global__ void __launch_bounds__(TW) tree_walk(const __grid_constant__ TreeParams P)
{
    __shared__ int32_t s_par[TREE_NMAX], s_tok[TREE_NMAX], s_g[TREE_NMAX];
    __shared__ uint8_t s_acc[TREE_NMAX];
    __shared__ int16_t s_depth[TREE_NMAX];
    __shared__ int s_bad;
    const int b = blockIdx.x, N = P.N;
    const size_t o = (size_t)b * N;
    if (threadIdx.x == 0)
        s_bad = 0;
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += TW) {
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
    if (threadIdx.x != 0)
        return;
    int code = s_bad ? 1 : 0;
    if (!code) {
        s_acc[0] = 1;
        s_depth[0] = 0;
        for (int n = 0; n < N; ++n) {
            if (n > 0) {
                const int p = s_par[n];
                s_depth[n] = (int16_t)(s_depth[p] + 1);
                s_acc[n] = 0;
                if (!s_acc[p])
                    continue;
                const int t = s_tok[n];
                if (t < 0 || t >= P.V) {
                    code = ST_TOKEN;
                    break;
                }
                if (t != s_g[p])
                    continue;
                s_acc[n] = 1;
            }
            if (s_g[n] < 0) {
                code = ST_NONFINITE;
                break;
            }
        }
    }
    if (code) {
        P.out_len[b] = -code;
        if (P.status)
            atomicCAS(P.status, 0, code);
        return;
    }
    int best = 0;
    for (int n = 1; n < N; ++n)
        if (s_acc[n] && s_depth[n] > s_depth[best])
            best = n;
    const int d = s_depth[best];
    for (int n = best, k = d - 1; n > 0; n = s_par[n], --k) {
        P.out_tokens[o + k] = s_tok[n];
        P.out_nodes[o + k] = n;
    }
    P.out_tokens[o + d] = s_g[best];
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
    tree_walk<<<B, TW, 0, stream>>>(P);
    return cudaGetLastError();
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
