// internal.h - launchers and launch geometry shared by the C-ABI layer and the kernel files.
// Internal header (not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "moe_grouped.h"

namespace moe {

// Launch `kern` with an optional programmatic-dependent-launch edge to the previous work on the
// stream (the kernel itself calls griddepcontrol.wait before reading dependent data).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Arguments of one grouped GEMV launch (gate/up or down).
struct GemvArgs {
    const void* const* w;  // [n_experts] blob pointers
    int n_experts;
    int K;            // weights per row
    int rows;         // rows per expert
    int row_bytes;    // bytes per row
    int nch;          // 256-weight chunks per row
    int CPW;          // chunks per consumer warp and tile
    int WPS;          // consumer warps per warp-set (one tile per set at a time) = ceil(nch / CPW)
    int TP;           // warp-sets per CTA (tiles in flight in compute)
    int CW;           // consumer warps per CTA = WPS * TP (plus one producer warp)
    int RT;           // rows per tile (32, or 16 for very long rows): lane = row
    int stages;       // staging ring depth
    int stage_bytes;  // bytes per ring slot (tile + slack, multiple of 128)
    int alpha;        // decode cost of a row relative to one entry's dot products (balancing)
    const int32_t* grp_expert;
    const int32_t* grp_start;
    const int32_t* n_groups;
    int cap_groups;
    int cap_entries;
    const moe_q8_1* act;  // activation rows
    int n_act_rows;
    const int32_t* ent_in;   // entry -> activation row (nullptr: the entry itself)
    const int32_t* ent_out;  // entry -> output row (nullptr: the entry itself)
    float* out;
    int64_t out_rows;
    int64_t out_stride;
    int32_t* err;
    const int8_t* codebook;
    int prefetch_before_wait;  // weight tiles may be requested before griddepcontrol.wait
    // dynamic shared-memory layout (byte offsets; a CB codebook, when present, is at offset 0;
    // two activation buffers of kMaxEntriesPerPass entries; the group table holds cap_groups)
    int off_ring, off_part, off_actq, off_act2, off_bar, off_misc, off_grp, off_ent;
    int act_cap;     // activation rows the act region holds (>= 8)
    int part_bytes;  // per-slot partial sums: nch x 4 entries x RT floats
    int nb;   // activation blocks per row (K/32)
    int nbp;  // padded block slots per activation half-row
};

struct GemvPlan {
    int NT, smem;
};

// Arguments of one fused layer launch (layer.cuh).
// The fused layer's sync array (int32 words): the exit counter, the global work-item counter, the
// call epoch and the largest number of h pairs any call on the array has used, then from word
// kSyncHx the flagged copy of h: per entry, nine rows (k = 0..8) of one 8-byte pair per h block
// (low word: the block's header for k = 0, code word k - 1 otherwise; high word: the writing
// call's flag, epoch + 1), so that a reader polls the data itself.
constexpr int kSyncExit = 0, kSyncWork = 1, kSyncEpoch = 2, kSyncExt = 3, kSyncHx = 4;
constexpr int kHxPairs = 9;  // pairs per q8_1 block
// Entries of a group the fused layer kernel applies per pass over its weights (a group of more
// streams them once per batch; at T <= 4 and top-8 of 64 or more experts a group of three or
// four entries is rare)
constexpr int kLayerBatch = 2;
constexpr int kMaxHBufs = 6;  // the fused layer kernel's down h-staging buffers at most

struct LayerArgs {
    GemvArgs gu, dn;     // per-phase geometry and pointers (shared ring, partials, barriers, misc)
    const int32_t* ids;  // [T][k] top-k expert ids
    const float* x;      // [T][n_embd]
    moe_q8_1* hq;        // [n][F/32]: the q8_1 h rows (exchanged between the CTAs)
    int32_t* sync;       // control words (kSync*) and the flagged h copy from kSyncHx (8-byte aligned)
    int32_t* sync_other; // the other half of a sync pair (reset by this call; nullptr: no pair)
    int32_t *o_ge, *o_gs, *o_ng, *o_es, *o_ed;  // optional copies of the grouping (CTA 0)
    moe_q8_1* o_xq;                             // optional copy of the activation q8_1 (CTA 0)
    int T, k, n;         // n = T * k entries (and the capacity of every per-group table)
    int F, nbj;          // n_ff, n_ff / 32
    int nsub;            // 32-row sub-tiles per down tile
    int upg, tpu;        // gate/up units (32 h values) per group, ring tiles per unit
    int off_route;       // shared-memory routing scratch
    int off_unit;        // shared-memory gate/up unit buffers: [4 units][4 entries][32] h values
    int off_ptr;         // shared-memory cache of both expert pointer tables (0: not cached)
    int test_expire;     // test hook: the down staging waits for a flag no call writes
    // pre-built groups (moe_expert_grouped_fused): given = 1 reads the grouping and the activation
    // q8_1 rows from these instead of routing ids and quantizing x
    int given;
    const int32_t *g_expert, *g_start, *g_ng, *g_src, *g_dst;
    int g_cap_groups, g_cap_entries;
    int64_t g_out_rows;
};

cudaError_t launch_quantize_q8_1(const float* x, int64_t rows, int64_t cols, moe_q8_1* xq, cudaStream_t s,
                                 bool pdl);
cudaError_t launch_swiglu_q8_1(const float* gu, int n_ff, const int32_t* grp_start, const int32_t* n_groups,
                               int cap_groups, int cap_entries, moe_q8_1* hq, int32_t* err, cudaStream_t s,
                               bool pdl);
cudaError_t launch_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base,
                               int32_t* grp_expert, int32_t* grp_start, int32_t* n_groups, int32_t* ent_src,
                               int32_t* ent_dst, int32_t* err, cudaStream_t s);

cudaError_t launch_router_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);
cudaError_t launch_combine(const float* out, int64_t os, const int32_t* ids, const float* w, int T, int k, int E, int N,
                           float* y, int64_t ys, cudaStream_t s);
cudaError_t launch_transcode_cb(int src_type, const int8_t* codebook, int dst_type, int K, int rows, int n_blobs,
                                const void* const* src_blobs, void* const* dst_blobs, int32_t* err, cudaStream_t s);

// The residency split's staging copies: blob i < n, bytes[i] (a multiple of 16) from src[i] (pinned
// host memory, device-accessible, 16-byte aligned) to dst[i] (device, 16-byte aligned), by one
// kernel per kStageMax blobs.
constexpr int kStageMax = 8;
cudaError_t launch_stage_blobs(const void* const* src, void* const* dst, const int64_t* bytes, int n, cudaStream_t s);

cudaError_t launch_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* scale, long long n_blocks,
                                    float* scores, cudaStream_t s);

// Per-format grouped GEMV and test-hook launchers (one translation unit per format).
#define MOE_DECLARE_FORMAT(NAME)                                                                       \
    cudaError_t launch_gemv_##NAME(const GemvArgs& a, int grid, int NT, int smem, cudaStream_t s, bool pdl); \
    cudaError_t gemv_occupancy_##NAME(int NT, int smem, int* ctas);                                     \
    cudaError_t launch_isum_##NAME(const int8_t* codebook, int K, const void* blob, int rows,           \
                                   const moe_q8_1* xq, int32_t* isum, cudaStream_t s);
MOE_DECLARE_FORMAT(q8_0)
MOE_DECLARE_FORMAT(q4b)
MOE_DECLARE_FORMAT(nl4)
MOE_DECLARE_FORMAT(cb2)
MOE_DECLARE_FORMAT(cb3)
MOE_DECLARE_FORMAT(cb3x)
MOE_DECLARE_FORMAT(cb2x)
#undef MOE_DECLARE_FORMAT

// Fused layer launchers, one translation unit per gate/up format (down: NL4 or Q8_0).
#define MOE_DECLARE_LAYER(NAME)                                                                         \
    cudaError_t launch_layer_##NAME(const LayerArgs& a, int dt, int grid, int NT, int smem, cudaStream_t s, \
                                    bool pdl);                                                          \
    cudaError_t layer_occupancy_##NAME(int dt, int NT, int smem, int* ctas);
MOE_DECLARE_LAYER(q8_0)
MOE_DECLARE_LAYER(q4b)
MOE_DECLARE_LAYER(nl4)
MOE_DECLARE_LAYER(cb2)
MOE_DECLARE_LAYER(cb3)
MOE_DECLARE_LAYER(cb3x)
MOE_DECLARE_LAYER(cb2x)
#undef MOE_DECLARE_LAYER

}  // namespace moe
