// Stochastic verification over the full vocabulary (draft logits or probabilities).
#include "sv_instantiate.cuh"

namespace sv {

// Philox words as the decisions draw them (for checking).
__global__ void philox_words_kernel(uint32_t k0, uint32_t k1, uint32_t tag, int B, int Pn, uint32_t *out)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * Pn)
        return;
    const int b = i / Pn, pos = i % Pn;
    const uint4 w = philox10((uint32_t)pos, (uint32_t)b, tag, 0u, k0, k1);
    reinterpret_cast<uint4 *>(out)[i] = w;
}

KernelEntry entry_stoch(int tdt, bool probs)
{
    if (tdt == 0)
        return probs ? make_entry<F32, MODE_STOCH, true>() : make_entry<F32, MODE_STOCH, false>();
    return probs ? make_entry<BF16, MODE_STOCH, true>() : make_entry<BF16, MODE_STOCH, false>();
}

cudaError_t launch_philox_words(uint32_t k0, uint32_t k1, uint32_t tag, int B, int P, uint32_t *out,
                                cudaStream_t stream)
{
    const int n = B * P;
    philox_words_kernel<<<(n + 255) / 256, 256, 0, stream>>>(k0, k1, tag, B, P, out);
    return cudaGetLastError();
}

}  // namespace sv
