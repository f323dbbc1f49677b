// swiglu_q8_1.cu - the activation q8_1 quantizer and the fused SwiGLU + q8_1 kernel.
//
// Fused kernel: #363 "experts: smaller and fewer launches for the verify window's PCIe call",
// "What changes": one kernel over the call's own entries [grp_start[0], grp_start[n_groups]);
// the SwiGLU product is rounded on its own before the q8_1 block sums. One warp per q8_1 block
// (32 consecutive h values of one entry); the grid is sized from cap_entries and every warp
// reads the device-side entry range, so an empty call returns at once.
#include "internal.h"
#include "q8_1.cuh"

namespace moe {

__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float* __restrict__ x, int64_t nblocks,
                                                            moe_q8_1* __restrict__ xq) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += warps)
        warp_q8_1(x[b * 32 + lane], xq + b, lane);
}

__global__ void __launch_bounds__(256) swiglu_q8_1_kernel(const float* __restrict__ gu, int n_ff,
                                                          const int32_t* __restrict__ grp_start,
                                                          const int32_t* __restrict__ n_groups, int cap_groups,
                                                          int cap_entries, moe_q8_1* __restrict__ hq,
                                                          int32_t* err) {
    pdl_wait();
    pdl_trigger();
    int G = *n_groups;
    if (G < 0 || G > cap_groups) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, MOE_ERR_NGROUPS);
        G = G < 0 ? 0 : cap_groups;
    }
    if (G == 0) return;
    const int e0 = grp_start[0], e1 = grp_start[G];
    if (e0 < 0 || e1 < e0 || e1 > cap_entries) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_err(err, MOE_ERR_START);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int bpe = n_ff / 32;
    const int64_t total = (int64_t)(e1 - e0) * bpe;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += warps) {
        const int e = e0 + static_cast<int>(w / bpe), b = static_cast<int>(w % bpe);
        const float* row = gu + (int64_t)e * 2 * n_ff;
        const int j = b * 32 + lane;
        warp_q8_1(swiglu_rn(row[j], row[n_ff + j]), hq + (int64_t)e * bpe + b, lane);
    }
}

cudaError_t launch_quantize_q8_1(const float* x, int64_t rows, int64_t cols, moe_q8_1* xq, cudaStream_t s,
                                 bool pdl) {
    const int64_t nblocks = rows * (cols / 32);
    if (nblocks == 0) return cudaSuccess;
    int grid = static_cast<int>((nblocks + 7) / 8);
    if (grid > 152 * 16) grid = 152 * 16;
    return launch_kernel(quantize_q8_1_kernel, dim3(grid), dim3(256), 0, s, pdl, x, nblocks, xq);
}

cudaError_t launch_swiglu_q8_1(const float* gu, int n_ff, const int32_t* grp_start, const int32_t* n_groups,
                               int cap_groups, int cap_entries, moe_q8_1* hq, int32_t* err, cudaStream_t s,
                               bool pdl) {
    const int64_t warps = (int64_t)cap_entries * (n_ff / 32);
    int grid = static_cast<int>((warps + 7) / 8);
    if (grid > 152 * 16) grid = 152 * 16;
    if (grid < 1) grid = 1;
    return launch_kernel(swiglu_q8_1_kernel, dim3(grid), dim3(256), 0, s, pdl, gu, n_ff, grp_start, n_groups,
                         cap_groups, cap_entries, hq, err);
}

}  // namespace moe
