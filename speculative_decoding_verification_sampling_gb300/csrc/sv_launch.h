// sv_launch.h -- host-side entry points of the kernel instantiations.
#pragma once
#include <cuda_runtime.h>

#include "sv_params.h"

namespace sv {

// Launch kern(P) with programmatic dependent launch: it may begin while the
// previous kernel in the stream finishes, and waits for that kernel's results
// itself (griddepcontrol.wait before its first access to global memory).
template <class Kern, class Par>
cudaError_t launch_after(Kern kern, int grid, int block, int smem, cudaStream_t stream, const Par &P)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

struct KernelEntry {
    cudaError_t (*launch)(const Params &P, int grid, cudaStream_t stream);
    cudaError_t (*occupancy)(int *ctas_per_sm);
};

// tdt: 0 = float32, 1 = bfloat16 target (and draft logit) elements.
KernelEntry entry_stoch(int tdt, bool probs);
KernelEntry entry_greedy(int tdt);
KernelEntry entry_short(int tdt, bool probs);

// The cluster kernel: one sequence per cluster of `csize` CTAs.
struct ClusterEntry {
    cudaError_t (*launch)(const ClusterParams &P, int clusters, int csize, uint32_t smem, cudaStream_t stream);
    cudaError_t (*max_clusters)(int csize, uint32_t smem, int *clusters);
};
ClusterEntry entry_cluster(int tdt, bool greedy);
uint32_t cluster_header_bytes();   // shared memory ahead of the row slices

// Device scratch that needs no caller workspace: 64 words (256 bytes), of
// which the cluster kernel uses the CTL_WORDS control words.
constexpr int STATIC_SCRATCH_WORDS = 64;
cudaError_t static_scratch_address(uint32_t **addr);   // current device

// Row-parallel verification (k_rows.cu): statistics per row, residual masses
// per sequence chunk, then sampling per sequence (greedy: no residual kernel).
int rows_chunks();
// Whether a stochastic call with aligned rows of draft logits fits the
// resident path (every row of the call held in the shared memory of CTAs
// resident at once).
bool rows_resident_fits(int B, int K, int V, int tdt);
int rows_segment_tokens();
// *launches: the kernels the call launched
cudaError_t launch_rows(const RowsParams &P, int tdt, cudaStream_t stream, int *launches);
// Greedy verification in one launch (k_greedy_rows.cu): the argmax of every
// target row in parts; the last row of a sequence walks the rule.
cudaError_t launch_greedy_rows(const RowsParams &P, int tdt, cudaStream_t stream, int *launches);

// KV-cache commit after verification (k_kv.cu): copy, then the length update.
cudaError_t launch_kv_commit(void *cache, const void *staged, int NL, int B, int K, int L, long long W,
                             const int32_t *acc, int32_t *len, int32_t *status, cudaStream_t stream, int *launches);

// Greedy tree verification and the tree mask (k_tree.cu).
int tree_max_nodes();
cudaError_t launch_tree_walk(const int32_t *tokens, const int32_t *parent, const int32_t *g, int B, int N, int V,
                             int32_t *out_tokens, int32_t *out_nodes, int32_t *out_len, int32_t *status,
                             cudaStream_t stream);
cudaError_t launch_tree_mask(const int32_t *parent, int B, int N, uint8_t *mask, int32_t *status, cudaStream_t stream);

// The fused draft-token sampler (k_draft.cu): one CTA per row of draft logits.
int draft_max_v();
cudaError_t launch_draft_sample(const void *draft, int tdt, int B, int K, int V, float T, uint64_t seed,
                                int32_t *out_tokens, float *out_prob, int32_t *status, cudaStream_t stream);

cudaError_t launch_philox_words(uint32_t k0, uint32_t k1, uint32_t tag, int B, int P, uint32_t *out,
                                cudaStream_t stream);

}  // namespace sv
