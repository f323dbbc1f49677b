// stage.cu - the residency split's staging copies (#363 "experts: smaller and fewer launches for the
// verify window's PCIe call", "What changes": the experts that live in host memory come over the
// CPU-GPU link for the layer's second call). One kernel copies a call's host-resident blobs into
// their device staging slots: it reads pinned host memory through unified addressing, 16 bytes
// at a time with four reads in flight per thread, so the bytes cross the link at the link's rate
// without a copy-engine node per blob between the kernels of a graph, and the expert call that
// follows can be launched with programmatic dependent launch (it waits for this grid to complete
// before reading the slots).
#include "common.cuh"
#include "internal.h"

namespace moe {

struct StageBatch {
    const uint4* src[kStageMax];
    uint4* dst[kStageMax];
    long long n16[kStageMax];
};

__global__ void __launch_bounds__(256) stage_kernel(const StageBatch b) {
    pdl_trigger();  // the call that reads the slots may launch and run its prologue meanwhile
    const int blob = blockIdx.y;
    const uint4* __restrict__ src = b.src[blob];
    uint4* __restrict__ dst = b.dst[blob];
    const long long n = b.n16[blob];
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 v0 = src[i], v1 = src[i + stride], v2 = src[i + 2 * stride], v3 = src[i + 3 * stride];
        dst[i] = v0;
        dst[i + stride] = v1;
        dst[i + 2 * stride] = v2;
        dst[i + 3 * stride] = v3;
    }
    for (; i < n; i += stride) dst[i] = src[i];
}

cudaError_t launch_stage_blobs(const void* const* src, void* const* dst, const int64_t* bytes, int n, cudaStream_t s) {
    for (int i0 = 0; i0 < n; i0 += kStageMax) {
        const int m = n - i0 < kStageMax ? n - i0 : kStageMax;
        StageBatch b{};
        long long most = 0;
        for (int k = 0; k < m; ++k) {
            b.src[k] = static_cast<const uint4*>(src[i0 + k]);
            b.dst[k] = static_cast<uint4*>(dst[i0 + k]);
            b.n16[k] = bytes[i0 + k] / 16;
            most = b.n16[k] > most ? b.n16[k] : most;
        }
        long long gx = (most + 4 * 256 - 1) / (4 * 256);  // four 16-byte words per thread per pass
        gx = gx < 1 ? 1 : gx > 152 ? 152 : gx;
        stage_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(m)), 256, 0, s>>>(b);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
