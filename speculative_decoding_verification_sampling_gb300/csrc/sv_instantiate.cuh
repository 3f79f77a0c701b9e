// sv_instantiate.cuh -- launch and occupancy wrappers around verify_kernel.
#pragma once
#include "sv_kernel.cuh"
#include "sv_launch.h"

namespace sv {

template <class E, int MODE, bool PROBS>
cudaError_t launch_verify(const Params &P, int grid, cudaStream_t stream)
{
    auto kern = verify_kernel<E, MODE, PROBS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, NTHREADS, SMEM_BYTES, stream>>>(P);
    return cudaGetLastError();
}

template <class E, int MODE, bool PROBS>
cudaError_t occupancy_verify(int *ctas_per_sm)
{
    auto kern = verify_kernel<E, MODE, PROBS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kern, NTHREADS, SMEM_BYTES);
}

template <class E, int MODE, bool PROBS>
KernelEntry make_entry()
{
    return KernelEntry{&launch_verify<E, MODE, PROBS>, &occupancy_verify<E, MODE, PROBS>};
}

}  // namespace sv
