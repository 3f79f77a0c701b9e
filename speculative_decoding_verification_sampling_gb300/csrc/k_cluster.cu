// Cluster kernel instantiations: stochastic (draft logits) and greedy, float32 and bfloat16.
#include "sv_cluster.cuh"
#include "sv_launch.h"

namespace sv {

namespace {

template <class E, int MODE>
cudaError_t launch_cluster(const ClusterParams &P, int clusters, int csize, uint32_t smem, cudaStream_t stream)
{
    auto kern = cluster_kernel<E, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    // all of the unified L1 / shared memory as shared memory: three CTAs per SM
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100)) != cudaSuccess)
        return e;
    if (csize > 8 &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(clusters * csize), 1, 1);
    cfg.blockDim = dim3(CL_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, P);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <class E, int MODE>
cudaError_t max_clusters_cluster(int csize, uint32_t smem, int *clusters)
{
    auto kern = cluster_kernel<E, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    // all of the unified L1 / shared memory as shared memory: three CTAs per SM
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100)) != cudaSuccess)
        return e;
    if (csize > 8 &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(csize * 1024), 1, 1);
    cfg.blockDim = dim3(CL_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

template <class E, int MODE>
ClusterEntry make_cluster_entry()
{
    return ClusterEntry{&launch_cluster<E, MODE>, &max_clusters_cluster<E, MODE>};
}

}  // namespace

uint32_t cluster_header_bytes() { return CL_HDR; }

// Scratch of spec_verify_static: the cluster kernel's control block lives in
// this module-scope array instead of a caller workspace.  Zero at load, and
// left zero by every call that completes.
static __device__ __align__(256) uint32_t g_static_scratch[STATIC_SCRATCH_WORDS];
static_assert(STATIC_SCRATCH_WORDS >= CTL_WORDS, "the control block must fit the static scratch");

cudaError_t static_scratch_address(uint32_t **addr)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    *addr = static_cast<uint32_t *>(p);
    return e;
}

ClusterEntry entry_cluster(int tdt, bool greedy)
{
    if (tdt == 0)
        return greedy ? make_cluster_entry<F32, MODE_GREEDY>() : make_cluster_entry<F32, MODE_STOCH>();
    return greedy ? make_cluster_entry<BF16, MODE_GREEDY>() : make_cluster_entry<BF16, MODE_STOCH>();
}

}  // namespace sv
