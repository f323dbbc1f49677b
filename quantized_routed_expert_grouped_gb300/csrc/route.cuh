// route.cuh - routing/grouping of a window's top-k expert ids by one CTA (a0).
//
// The groups that #363 "experts: smaller and fewer launches for the verify window's PCIe call"
// ("What changes") passes to each call: one group per distinct expert, groups by ascending expert
// id, entries of a group by ascending (token, slot). Thread i < n owns id i (n = T*k <= blockDim)
// and ranks itself against all others, so the result does not depend on scheduling.
#pragma once

#include "common.cuh"

namespace moe {

// Every thread of the CTA must call this (it holds two CTA barriers). sid, sfirst: n ints of
// shared scratch; scount: 2 ints of shared scratch. Outputs go through generic pointers (global
// or shared memory): grp_expert[G], grp_start[G+1], *n_groups, and for each entry e (numbered
// from entry_base) ent_src[e] = t, ent_dst[e] = t*k + slot. Ids outside [0, n_experts) are
// dropped; `report` threads set MOE_ERR_ROUTE for them.
__device__ __forceinline__ void route_cta(const int32_t* ids, int n, int k, int n_experts, int entry_base, int* sid,
                                          int* sfirst, int* scount, int32_t* grp_expert, int32_t* grp_start,
                                          int32_t* n_groups, int32_t* ent_src, int32_t* ent_dst, int32_t* err,
                                          bool report) {
    const int i = threadIdx.x;
    int my = -1;
    if (i < n) {
        const int v = ids[i];
        my = (v >= 0 && v < n_experts) ? v : -1;
        if (my < 0 && report) set_err(err, MOE_ERR_ROUTE);
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

}  // namespace moe
