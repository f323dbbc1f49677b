// router_combine.cu - the steps either side of the grouped call: the router's top-k expert ids
// with softmax weights over the selected logits, and the per-token weighted combine of the k
// entry rows ("the combined output" that #3455 "GP100 (sm_60): 4-bit slots for resident IQ2_S /
// IQ3_XXS / IQ3_S gate/up experts" checks in "Passed"). The pages do not define the router; the
// plainest reading is used: the k largest logits (ties: the lower expert id first), in
// descending order, weights e^(l_j) / sum of e^(l_i) over the k selected.
#include "common.cuh"
#include "internal.h"
#include "q8_1.cuh"

namespace moe {

// One warp per token. k rounds of a warp-wide arg-max over the experts not yet taken (larger
// logit first, then the lower id); lane i scans experts i, i + 32, ... and keeps its taken ones
// in a bit mask (E <= 1024). Lane j then holds slot j; the weights use the largest logit as the
// shift: e_j = exp(l_j - l_0) (this library's exp), summed in slot order, divided (IEEE).
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                          int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;  // warp-uniform
    const float* l = logits + static_cast<int64_t>(t) * E;
    uint32_t taken = 0;
    float selv = 0.0f;
    int seli = 0;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int bi = 0;
        bool has = false;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if ((taken >> i) & 1u) continue;
            const float v = __ldg(l + e);
            if (!has || v > bv) {  // experts in ascending order: a tie keeps the lower id
                bv = v;
                bi = e;
                has = true;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            const bool oh = __shfl_xor_sync(0xffffffffu, has ? 1 : 0, o) != 0;
            if (oh && (!has || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
                has = true;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            selv = bv;
            seli = bi;
        }
    }
    const float m = __shfl_sync(0xffffffffu, selv, 0);
    const float ex = lane < k ? exp_cw(__fsub_rn(selv, m)) : 0.0f;
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, ex, j));
    if (lane < k) {
        ids[static_cast<int64_t>(t) * k + lane] = seli;
        w[static_cast<int64_t>(t) * k + lane] = __fdiv_rn(ex, s);
    }
}

// y[t][n] = sum over the slots j < k in order, skipping ids outside [0, E), of w[t][j] *
// out[t*k + j][n], as fp32 fused multiply-adds from zero. One thread per (token, column).
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ out, int64_t os,
                                                      const int32_t* __restrict__ ids, const float* __restrict__ w,
                                                      int k, int E, int N, float* __restrict__ y, int64_t ys) {
    const int t = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int x = __ldg(ids + static_cast<int64_t>(t) * k + j);
        if (x < 0 || x >= E) continue;
        acc = fmaf(__ldg(w + static_cast<int64_t>(t) * k + j), __ldg(out + (static_cast<int64_t>(t) * k + j) * os + n),
                   acc);
    }
    y[static_cast<int64_t>(t) * ys + n] = acc;
}

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
    const int per_block = 8;  // tokens (warps) per 256-thread block
    return launch_kernel(router_topk_kernel, dim3((T + per_block - 1) / per_block), dim3(32 * per_block), 0, s, false,
                         logits, T, E, k, ids, w);
}

cudaError_t launch_combine(const float* out, int64_t os, const int32_t* ids, const float* w, int T, int k, int E, int N,
                           float* y, int64_t ys, cudaStream_t s) {
    return launch_kernel(combine_kernel, dim3((N + 255) / 256, T), dim3(256), 0, s, false, out, os, ids, w, k, E, N, y,
                         ys);
}

}  // namespace moe
