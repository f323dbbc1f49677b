// route.cu - the routing/grouping kernel (a0): one CTA, one thread per (t, slot); the grouping
// itself is route_cta (route.cuh), shared with the fused layer kernel.
#include "internal.h"
#include "route.cuh"

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
    route_cta(ids, T * k, k, n_experts, entry_base, sid, sfirst, scount, grp_expert, grp_start, n_groups, ent_src,
              ent_dst, err, true);
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
