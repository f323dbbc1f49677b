// route.cu - routing/grouping of a window's top-k expert ids into expert groups (a0).
//
// The groups that #363 "experts: smaller and fewer launches for the verify window's PCIe call"
// ("What changes") passes to each call: one group per distinct expert, groups by ascending
// expert id, entries of a group by ascending (token, slot). One CTA, one thread per (t, slot);
// every thread ranks itself against all others (T*k <= 1024), so the result is deterministic.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(1024) route_group_kernel(const int32_t* __restrict__ ids, int T, int k, int n_experts,
                                                           int entry_base, int32_t* grp_expert, int32_t* grp_start,
                                                           int32_t* n_groups, int32_t* ent_src, int32_t* ent_dst,
                                                           int32_t* err) {
    __shared__ int sid[1024];
    __shared__ int sfirst[1024];
    __shared__ int scount[2];
    pdl_wait();
    pdl_trigger();
    const int n = T * k, i = threadIdx.x;
    int my = -1;
    if (i < n) {
        const int v = ids[i];
        my = (v >= 0 && v < n_experts) ? v : -1;
        if (my < 0) set_err(err, MOE_ERR_ROUTE);
        sid[i] = my;
    }
    if (i < 2) scount[i] = 0;
    __syncthreads();
    bool first = false;
    if (my >= 0) {
        first = true;
        for (int j = 0; j < i; ++j)
            if (sid[j] == my) { first = false; break; }
        sfirst[i] = first;
        atomicAdd(&scount[0], 1);
        if (first) atomicAdd(&scount[1], 1);
    } else if (i < n) {
        sfirst[i] = 0;
    }
    __syncthreads();
    if (my >= 0) {
        int rank = 0, grp = 0;
        for (int j = 0; j < n; ++j) {
            const int v = sid[j];
            if (v < 0) continue;
            if (v < my || (v == my && j < i)) ++rank;
            if (v < my && sfirst[j]) ++grp;
        }
        const int e = entry_base + rank;
        ent_src[e] = i / k;
        ent_dst[e] = i;
        if (first) {
            grp_expert[grp] = my;
            grp_start[grp] = e;
        }
    }
    if (i == 0) {
        grp_start[scount[1]] = entry_base + scount[0];
        *n_groups = scount[1];
    }
}

cudaError_t launch_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base,
                               int32_t* grp_expert, int32_t* grp_start, int32_t* n_groups, int32_t* ent_src,
                               int32_t* ent_dst, int32_t* err, cudaStream_t s) {
    const int n = T * k;
    const int threads = ((n + 31) / 32) * 32;
    return launch_kernel(route_group_kernel, dim3(1), dim3(threads), 0, s, false, topk_ids, T, k, n_experts,
                         entry_base, grp_expert, grp_start, n_groups, ent_src, ent_dst, err);
}

}  // namespace moe
