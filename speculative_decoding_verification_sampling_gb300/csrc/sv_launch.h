// sv_launch.h -- host-side entry points of the kernel instantiations.
#pragma once
#include <cuda_runtime.h>

#include "sv_params.h"

namespace sv {

struct KernelEntry {
    cudaError_t (*launch)(const Params &P, int grid, cudaStream_t stream);
    cudaError_t (*occupancy)(int *ctas_per_sm);
};

// tdt: 0 = float32, 1 = bfloat16 target (and draft logit) elements.
KernelEntry entry_stoch(int tdt, bool probs);
KernelEntry entry_greedy(int tdt);
KernelEntry entry_short(int tdt, bool probs);

cudaError_t launch_philox_words(uint32_t k0, uint32_t k1, uint32_t tag, int B, int P, uint32_t *out,
                                cudaStream_t stream);

}  // namespace sv
