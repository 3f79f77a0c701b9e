// k_kv.cu -- KV-cache commit (and rollback) after verification.
//
// nextadmin.net lesson "Speculative Decoding", § KV cache management: the
// verification pass appends K entries to the target's KV cache; after the
// left-to-right rule, only the accepted drafts' entries may stay.  With a
// staging buffer the K entries are written there first and the accepted ones
// are committed; written in place, the rejected ones are rolled back by
// truncating the length.  For sequence b with a = accept_len[b] >= 0:
//   cache[l][b][len_b + t] = staged[l][b][t] for t < a and every layer l,
//   len_b += a;
// a < 0 (a sequence in error) commits nothing; a > K or len_b + a > L commits
// nothing and is reported.
//
// Two kernels in stream order: the copy (one CTA per (layer, sequence,
// chunk): the a committed entries of a layer are contiguous in both buffers,
// so each is one contiguous copy of a * W bytes, 16-byte vectors with four in
// flight per thread), then the length update (one thread per sequence),
// launched behind the copy with programmatic dependent launch.
#include <cstdint>
#include <cuda_runtime.h>

#include "sv_params.h"
#include "sv_launch.h"

namespace sv {
namespace {

constexpr int KT = 256;   // threads of a copy CTA

struct KvParams {
    uint8_t *cache;          // [NL][B][L][W]
    const uint8_t *staged;   // [NL][B][K][W], or nullptr (entries written in place)
    const int32_t *acc;      // [B]
    int32_t *len;            // [B]
    int32_t *status;         // [1] or nullptr
    int NL, B, K, L, nch;
    long long W;             // bytes per entry and layer
    long long chunk;         // bytes per copy CTA (a multiple of 16)
    int vec;                 // W and both bases 16-byte aligned
};

__device__ __forceinline__ bool kv_ok(const KvParams &P, int a, int n)
{
    return a >= 0 && a <= P.K && n >= 0 && (long long)n + a <= P.L;
}

__global__ void __launch_bounds__(KT) kv_copy(const __grid_constant__ KvParams P)
{
    // the length update may start launching; it waits for this launch's end
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0 && P.status)
        *P.status = 0;   // only the length update, after this launch, reports
    const int ch = blockIdx.x % P.nch;
    const long long lb = blockIdx.x / P.nch;   // layer * B + b
    const int b = (int)(lb % P.B);
    const int a = __ldg(P.acc + b), n = __ldg(P.len + b);
    if (!kv_ok(P, a, n))
        return;
    const long long bytes = (long long)a * P.W;
    const long long lo = ch * P.chunk, hi = bytes < lo + P.chunk ? bytes : lo + P.chunk;
    if (lo >= hi)
        return;
    const uint8_t *src = P.staged + lb * P.K * P.W;
    uint8_t *dst = P.cache + (lb * P.L + n) * P.W;
    if (P.vec) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        const long long v0 = lo / 16, v1 = hi / 16;
        long long v = v0 + threadIdx.x;
        for (; v + 3 * KT < v1; v += 4 * KT) {
            uint4 r[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                r[k] = __ldg(s4 + v + k * KT);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                d4[v + k * KT] = r[k];
        }
        for (; v < v1; v += KT)
            d4[v] = __ldg(s4 + v);
    } else {
        for (long long i = lo + threadIdx.x; i < hi; i += KT)
            dst[i] = src[i];
    }
}

__global__ void kv_len(const __grid_constant__ KvParams P)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");   // every copy has read the old lengths
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= P.B)
        return;
    const int a = P.acc[b], n = P.len[b];
    if (kv_ok(P, a, n))
        P.len[b] = n + a;
    else if (a >= 0 && P.status)
        atomicCAS(P.status, 0, 1);   // a commit past the capacity, or above K
}

}  // namespace

cudaError_t launch_kv_commit(void *cache, const void *staged, int NL, int B, int K, int L, long long W,
                             const int32_t *acc, int32_t *len, int32_t *status, cudaStream_t stream, int *launches)
{
    KvParams P{};
    P.cache = static_cast<uint8_t *>(cache);
    P.staged = static_cast<const uint8_t *>(staged);
    P.acc = acc;
    P.len = len;
    P.status = status;
    P.NL = NL;
    P.B = B;
    P.K = K;
    P.L = L;
    P.W = W;
    P.vec = W % 16 == 0 && reinterpret_cast<uintptr_t>(cache) % 16 == 0 &&
            (!staged || reinterpret_cast<uintptr_t>(staged) % 16 == 0);
    // about 64 bytes per thread per copy CTA
    const long long per = (long long)KT * 64;
    const long long most = (long long)K * W;
    P.nch = (int)((most + per - 1) / per);
    if (P.nch < 1)
        P.nch = 1;
    P.chunk = ((most + P.nch - 1) / P.nch + 15) / 16 * 16;
    *launches = 0;
    if (staged) {
        // the copy zeroes the status word; the length update is launched
        // behind it with programmatic dependent launch
        kv_copy<<<(unsigned)((long long)NL * B * P.nch), KT, 0, stream>>>(P);
        ++*launches;
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)((B + 255) / 256));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        ++*launches;
        return cudaLaunchKernelEx(&cfg, kv_len, P);
    }
    if (status) {
        cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), stream);
        if (e != cudaSuccess)
            return e;
    }
    kv_len<<<(B + 255) / 256, 256, 0, stream>>>(P);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace sv
