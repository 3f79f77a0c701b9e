// Sweep kernel instantiations (float32 and bfloat16; greedy is a parameter).
#include "sv_sweep.cuh"
#include "sv_launch.h"

namespace sv {

namespace {

template <class E>
cudaError_t set_attrs()
{
    auto kern = sweep_kernel<E>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SW_SMEM);
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

template <class E>
cudaError_t launch_sweep(const SweepParams &P, int grid, cudaStream_t stream)
{
    cudaError_t e = set_attrs<E>();
    if (e != cudaSuccess)
        return e;
    sweep_kernel<E><<<grid, WTHREADS, SW_SMEM, stream>>>(P);
    return cudaGetLastError();
}

template <class E>
cudaError_t occupancy_sweep(int *ctas_per_sm)
{
    cudaError_t e = set_attrs<E>();
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, sweep_kernel<E>, WTHREADS, SW_SMEM);
}

}  // namespace

SweepEntry entry_sweep(int tdt)
{
    if (tdt == 0)
        return SweepEntry{&launch_sweep<F32>, &occupancy_sweep<F32>, WSBH / 4 * SW_MAXST};
    return SweepEntry{&launch_sweep<BF16>, &occupancy_sweep<BF16>, WSBH / 2 * SW_MAXST};
}

}  // namespace sv
