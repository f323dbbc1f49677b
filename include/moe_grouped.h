/* moe_grouped.h - C ABI of the grouped routed-expert decode for the verify window (GB300, sm_103a).
 *
 * The operation (from the pages of one inference engine):
 *  - #2058 "Verify window: the routed experts' gate/up with the group's q8_1 rows in shared
 *    memory", sections "Why" and "What changed": the window's T = 1-4 tokens are routed to top-k
 *    experts and grouped by expert; each group's block-quantized gate/up weights are read once
 *    and applied, as integer block dot products with fp32 block scales, to each of the group's
 *    1-4 q8_1 activation rows.
 *  - #363 "experts: smaller and fewer launches for the verify window's PCIe call", section "What
 *    changes": the group count n_groups lives on the device; group-stride launches sized by
 *    grid_groups (0 = cap_groups) make empty and near-empty calls cheap; SwiGLU and the q8_1
 *    quantization run as one kernel over the call's own entries [grp_start[0],
 *    grp_start[n_groups]); the SwiGLU product is rounded to fp32 on its own. Section
 *    "Exactness": a second call's entries may start past 0, its destinations are scattered, and
 *    rows a call does not own are never written.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless marked (host). The caller owns every buffer; no entry
 *    point allocates device memory, and every launch is asynchronous on `stream` (capturable in
 *    a CUDA graph).
 *  - The return value is MOE_OK or a negative MOE_E_* code for errors the host can see (null
 *    pointer, unsupported format, bad shape, bad capacity, a failed launch). Nothing is launched
 *    when an argument error is returned.
 *  - Errors in device-resident data (an expert id out of range, *n_groups above cap_groups,
 *    grp_start not monotone or outside [0, cap_entries], an entry's row index out of range, a
 *    weight pointer not 16-byte aligned, a bounded wait that gave up) are reported by OR-ing
 *    MOE_ERR_* bits into *err when err is not NULL; the offending group or entry is skipped (its
 *    rows are not written), *n_groups is clamped to cap_groups. Kernels never trap and never wait
 *    without a time limit.
 *  - Shapes: n_embd and n_ff are multiples of 256, at most 8192; cap_groups <= 1024,
 *    cap_entries <= 4096.
 *
 * Weight formats (this library's own byte layouts; the pages name real formats but print none).
 * Little-endian, fp16 fields are IEEE binary16. A row of K weights is K/32 blocks (K/256
 * super-blocks for CB2/CB3) packed without padding:
 *   MOE_Q8_0 (34 B / 32 w) : u16 d, i8 q[32]                         w = d*q
 *   MOE_Q4B  (20 B / 32 w) : u16 d, u16 m, u8 qs[16]                 w = d*code + m
 *   MOE_NL4  (18 B / 32 w) : u16 d, u8 qs[16]                        w = d*table[code]
 *        code j = qs[j] & 15 for j < 16, qs[j-16] >> 4 for j >= 16; table = 16 int8 (codebook)
 *   MOE_CB2  (70 B / 256 w): u16 D, u8 idx[32], u8 sign[32], u8 sub[4]
 *        weight n: +-grid[idx[n/8]][n%8], bit n%8 of sign[n/8] negates; grid = 256x8 int8
 *   MOE_CB3  (102 B / 256 w): u16 D, u8 idx[64], u8 sign[32], u8 sub[4]
 *        weight n: +-grid[idx[n/4]][n%4], bit n%8 of sign[n/8] negates; grid = 256x4 int8
 *   CB sub-block j (32 weights): ls = 2*((sub[j/2] >> 4*(j%2)) & 15) + 1, w = D*ls*(+-grid).
 *   CB grids must hold odd values only (the kernels rely on it; an even entry sets
 *   MOE_ERR_CODEBOOK).
 * Transcoded slot layouts (load-time re-encodings of CB2/CB3 by moe_transcode_cb, same integers,
 * decode without lookups; the idea of #3455 "GP100 (sm_60): 4-bit slots for resident IQ2_S /
 * IQ3_XXS / IQ3_S gate/up experts", "Problem and result"): each weight's signed odd value
 * v = +-grid is stored as u = (v-1)/2 + bias (v = 2*(u-bias) + 1). A row of K weights is K/256
 * code chunks, then K/256 scale records of 8 bytes (u16 D, u16 0, u8 sub[4]):
 *   MOE_CB3X (136 B / 256 w): 4-bit codes, bias 8 (|v| <= 15); in 32-weight sub-block j
 *        (16 bytes): low nibble of byte i = weight i, high nibble = weight 16+i.
 *   MOE_CB2X (72 B / 256 w): 2-bit codes, bias 2 (|v| <= 3); in sub-block j (8 bytes):
 *        bits 2p..2p+1 of byte i = weight 8p+i.
 * Gate/up blob of an expert: n_ff gate rows then n_ff up rows, each of n_embd weights.
 * Down blob of an expert: n_embd rows of n_ff weights. Blob pointers must be 16-byte aligned.
 *
 * q8_1 activation block (36 B per 32 values): fp16 d = amax/127, fp16 s = d * sum(q),
 * int8 q[32] = round-half-away-from-zero(x/d) (an all-zero block has d = s = 0, q = 0).
 */
#ifndef MOE_GROUPED_H
#define MOE_GROUPED_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- weight formats */
#define MOE_Q8_0 1
#define MOE_Q4B 2
#define MOE_NL4 3
#define MOE_CB2 4
#define MOE_CB3 5
#define MOE_CB3X 6
#define MOE_CB2X 7

/* ---- host-visible status codes */
#define MOE_OK 0
#define MOE_E_NULL (-1)  /* a required pointer is NULL */
#define MOE_E_TYPE (-2)  /* unsupported weight format, or a codebook missing for NL4/CB2/CB3 */
#define MOE_E_SHAPE (-3) /* n_embd / n_ff not a positive multiple of 256, bad rows/cols/T/k */
#define MOE_E_CAP (-4)   /* cap_groups / cap_entries / n_experts not positive, or too large */
#define MOE_E_CUDA (-5)  /* a CUDA runtime call failed (launch, attribute, device query) */
#define MOE_E_ALIGN (-6) /* a host-checkable pointer is not suitably aligned */
#define MOE_E_SCRATCH (-7) /* the call needs more scratch than the library's static buffer holds */

/* ---- device-side error bits, OR-ed into *err */
#define MOE_ERR_NGROUPS 1   /* *n_groups < 0 or > cap_groups (clamped) */
#define MOE_ERR_EXPERT 2    /* a group's expert id outside [0, n_experts) (group skipped) */
#define MOE_ERR_START 4     /* grp_start not monotone or outside [0, cap_entries] (group skipped) */
#define MOE_ERR_ENTRY 8     /* an entry's source or destination row out of range (entry skipped) */
#define MOE_ERR_ALIGN 16    /* an expert's weight pointer not 16-byte aligned (group skipped) */
#define MOE_ERR_CODEBOOK 32 /* a CB grid value is even (results of that call are unspecified) */
#define MOE_ERR_TIMEOUT 64  /* a bounded wait (a staged weight tile, another CTA's rows) gave up */
#define MOE_ERR_ROUTE 128   /* a routed expert id outside [0, n_experts) (entry dropped) */

/* One q8_1 block (36 bytes). d and s are IEEE binary16 bit patterns. */
typedef struct moe_q8_1 {
    uint16_t d;
    uint16_t s;
    int8_t q[32];
} moe_q8_1;

/* A weight format: type = MOE_*; codebook = device pointer (4-byte aligned) to the NL4 table
 * (16 int8), the CB2 grid (256x8 int8) or the CB3 grid (256x4 int8); NULL for Q8_0 and Q4B. */
typedef struct moe_wfmt {
    int32_t type;
    const int8_t* codebook;
} moe_wfmt;

/* Load-time transcoding of CB2/CB3 blobs into a slot layout (MOE_CB3X or MOE_CB2X). For every
 * blob b < n_blobs: dst_blobs[b] (rows x row_bytes(dst_type, K)) = the slot form of
 * src_blobs[b] (rows x row_bytes(src.type, K)). src_blobs / dst_blobs: device arrays of device
 * pointers. A source blob must be 2-byte and a destination blob 8-byte aligned (the decode
 * kernels want slot blobs 16-byte aligned); a blob off its boundary sets MOE_ERR_ALIGN and is
 * left unwritten. A value outside the slot's range (|v| > 15 for CB3X, > 3 for CB2X) sets
 * MOE_ERR_CODEBOOK; check *err before using the result. The integer dot products and scales of
 * the slot form equal the source's exactly. */
int moe_transcode_cb(moe_wfmt src, int dst_type, int K, int rows, int n_blobs,
                     const void* const* src_blobs, void* const* dst_blobs, int32_t* err,
                     cudaStream_t stream);

/* Bytes of one row of K weights in format `type` (0 if K is not valid for it). Host only. */
int64_t moe_row_bytes(int type, int K);

/* Text for a status code or for a set of MOE_ERR_* bits (static storage). Host only. */
const char* moe_strerror(int status);

/* q8_1 quantization of activations (a1 in the step list; the quantizer of #363 "What changes").
 * x: fp32 [rows][cols], row-major; xq: [rows][cols/32] blocks. cols % 32 == 0. */
int moe_quantize_q8_1(const float* x, int64_t rows, int64_t cols, moe_q8_1* xq,
                      cudaStream_t stream);

/* Routing/grouping of a window (the groups that #363 "What changes" passes to the calls).
 * topk_ids: int32 [T][k] expert ids (distinct per token). Groups are ordered by ascending expert
 * id; entries of a group by ascending (t, slot). Entries are numbered from entry_base.
 * Outputs: grp_expert[G], grp_start[G+1] (grp_start[G] = entry_base + valid entries),
 * *n_groups = G, and for every produced entry e: ent_src[e] = t (row of the q8_1 activations),
 * ent_dst[e] = t*k + slot (destination row). Ids outside [0, n_experts) are dropped and set
 * MOE_ERR_ROUTE. Arrays indexed by e must hold entry_base + T*k elements; grp_expert T*k and
 * grp_start T*k + 1. T*k <= 1024. */
int moe_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base,
                    int32_t* grp_expert, int32_t* grp_start, int32_t* n_groups,
                    int32_t* ent_src, int32_t* ent_dst, int32_t* err, cudaStream_t stream);

/* Grouped gate/up (a2). For each group g < *n_groups with expert x = grp_expert[g] and each
 * entry e in [grp_start[g], grp_start[g+1]): gu[e][r] = sum over 32-blocks b of the block
 * contribution of row r of w_gu[x] against xq[ent_src[e]] block b, for r < 2*n_ff (gate rows
 * then up rows). Block contributions: Q8_0/NL4 d_w*d_x*isum; Q4B d_w*d_x*isum + m_w*s_x;
 * CB2/CB3 D*d_x*(ls*isum) per 32-weight sub-block; isum = exact integer sum of w_code*q.
 * w_gu: device array of n_experts device pointers (host-written table). xq: [n_xq_rows][n_embd/32].
 * gu: fp32 [cap_entries][2*n_ff]; only the rows of this call's entries are written.
 * grid_groups: 0 = cap_groups, > cap_groups is treated as cap_groups; it sizes the launch only,
 * results do not depend on it. */
int moe_grouped_gu(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_gu, int n_experts,
                   const int32_t* grp_expert, const int32_t* grp_start, const int32_t* n_groups,
                   int cap_groups, int grid_groups, const moe_q8_1* xq, int n_xq_rows,
                   const int32_t* ent_src, int cap_entries, float* gu, int32_t* err,
                   cudaStream_t stream);

/* Fused SwiGLU + q8_1 (a3, #363 "What changes"). For e in [grp_start[0], grp_start[*n_groups])
 * and j < n_ff: h = fp32(silu(gu[e][j]) * gu[e][n_ff+j]), silu(g) = g / (1 + exp(-g)) in fp32,
 * then q8_1 of each 32 consecutive h into hq[e][j/32]. hq: [cap_entries][n_ff/32]. */
int moe_swiglu_q8_1(const float* gu, int n_ff, const int32_t* grp_start, const int32_t* n_groups,
                    int cap_groups, int cap_entries, moe_q8_1* hq, int32_t* err,
                    cudaStream_t stream);

/* Grouped down (a4). For each group and entry e: out[ent_dst[e]][n] = sum over blocks of row n
 * of w_down[x] against hq[e], for n < n_embd. out: fp32 with out_rows rows of stride
 * out_row_stride floats (>= n_embd); rows not named by this call's entries are not written. */
int moe_grouped_down(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_down,
                     int n_experts, const int32_t* grp_expert, const int32_t* grp_start,
                     const int32_t* n_groups, int cap_groups, int grid_groups,
                     const moe_q8_1* hq, int cap_entries, const int32_t* ent_dst, float* out,
                     int64_t out_rows, int64_t out_row_stride, int32_t* err,
                     cudaStream_t stream);

/* Flags for moe_expert_call.flags */
#define MOE_F_PDL 1 /* chain the three kernels with programmatic dependent launch */
#define MOE_F_SYNC_PAIR 2 /* moe_expert_layer: sync holds two halves used by alternate calls */
#define MOE_F_SYNC_ODD 4  /* moe_expert_layer with MOE_F_SYNC_PAIR: this call uses the second half */
/* moe_expert_layer, test hook only: the down staging waits for a flag no call writes, so every CTA
 * that reaches a down item gives up after the wait limit (~1 s) and the call takes its timeout
 * path (MOE_ERR_TIMEOUT, the work left undone, the CTA's copies in flight awaited). The call's out
 * rows are then unspecified; zero the sync array before the next call. */
#define MOE_F_TEST_EXPIRE 8

/* One native_expert_grouped-style call (#363): gate/up, SwiGLU + q8_1, down on one stream. */
typedef struct moe_expert_call {
    moe_wfmt gu_fmt, down_fmt;
    int32_t n_embd, n_ff, n_experts;
    const void* const* w_gu;   /* [n_experts] device pointers to gate/up blobs */
    const void* const* w_down; /* [n_experts] device pointers to down blobs */
    const int32_t* grp_expert; /* [cap_groups] */
    const int32_t* grp_start;  /* [cap_groups + 1] */
    const int32_t* n_groups;   /* device scalar */
    int32_t cap_groups, grid_groups, cap_entries;
    const moe_q8_1* xq;        /* [n_xq_rows][n_embd/32] */
    int32_t n_xq_rows;
    const int32_t* ent_src;    /* [cap_entries] */
    const int32_t* ent_dst;    /* [cap_entries] */
    float* gu;                 /* scratch [cap_entries][2*n_ff] */
    moe_q8_1* hq;              /* scratch [cap_entries][n_ff/32] */
    float* out;                /* [out_rows][out_row_stride] */
    int64_t out_rows, out_row_stride;
    int32_t* err;              /* optional */
    int32_t flags;             /* MOE_F_* */
} moe_expert_call;

int moe_expert_grouped(const moe_expert_call* call, cudaStream_t stream);

/* Allocation-free variant of moe_expert_grouped (the pages have no counterpart; this is a
 * library convenience).
 *
 * Some callers cannot allocate device memory for the call's scratch: an engine that reserves all
 * of its device memory up front and forbids allocation afterwards, a plugin running inside a host
 * framework that owns every allocation, or a latency-critical path that cannot afford the
 * implicit device synchronisation of cudaMalloc/cudaFree. This entry point takes the same
 * arguments as moe_expert_grouped but ignores call->gu and call->hq: the gate/up rows and the
 * q8_1 h rows live in one buffer of MOE_STATIC_SCRATCH_BYTES bytes that the library declares as
 * static device memory, so nothing is allocated at call time. Every GPU that loads the library
 * holds that buffer until the process exits.
 *  - Limit: cap_entries * (2*n_ff*4 + (n_ff/32)*36) bytes (each part rounded up to 256) must not
 *    exceed MOE_STATIC_SCRATCH_BYTES, else MOE_E_SCRATCH is returned and nothing is launched
 *    (e.g. 32 entries at n_ff 768 need about 0.2 MB; 256 entries at n_ff 1536 about 3.6 MB).
 *  - The first call on each device looks up the buffer's device address (once per device, with
 *    that device current); make that first call before any stream capture on the device. The
 *    address is kept for the life of the process, so do not use this entry point across a
 *    device reset (cudaDeviceReset or anything else that tears down and rebuilds the context).
 *  - Every call shares the one buffer and it keeps the previous call's contents; the call writes
 *    every scratch row it later reads, so nothing needs clearing, but calls that overlap on the
 *    GPU (other streams, other threads) race on the buffer and must be serialised by the caller.
 */
#define MOE_STATIC_SCRATCH_BYTES (4u << 20)
int moe_expert_grouped_static(const moe_expert_call* call, cudaStream_t stream);

/* ---------------------------------------------------------------- fused layer call
 * The whole hot path of one layer in one kernel launch (the pages split it into a routing step
 * and three kernels, #363 "experts: smaller and fewer launches for the verify window's PCIe
 * call", "What changes"; this call fuses them): routing/grouping of topk_ids (as
 * moe_route_group with entry_base 0), q8_1 of x (as moe_quantize_q8_1), grouped gate/up, SwiGLU +
 * q8_1 and grouped down (as moe_expert_grouped with cap_groups = cap_entries = T*k, n_xq_rows = T,
 * out_rows = T*k). Every output equals that sequence's bit for bit.
 *  - out row t*k + slot receives entry (t, slot)'s n_embd values; rows of dropped ids (outside
 *    [0, n_experts), reported as MOE_ERR_ROUTE) are not written.
 *  - gu, hq: scratch [T*k][2*n_ff] and [T*k][n_ff/32] as in moe_expert_call, rows indexed by
 *    entry (groups by ascending expert id, entries of a group by ascending (t, slot)); after the
 *    call they hold the gate/up rows and the q8_1 h rows.
 *  - sync: moe_layer_sync_ints(T, k, n_ff) int32 words (8-byte aligned, else MOE_E_ALIGN) the
 *    launch's CTAs synchronise through: word 0 an exit counter, word 1 the work-item counter,
 *    word 2 the call epoch, word 3 the largest number of h pairs a call on the array has used,
 *    and from word 4 a flagged copy of the q8_1 h rows (per entry nine rows of one 8-byte pair
 *    per h block: a header or code word and the writing call's flag, epoch + 1), which the down
 *    phase polls instead of a counter, so the gate/up side needs no fence. The caller zeroes the
 *    array once before the first call (e.g. cudaMemsetAsync); every call leaves words 0 and 1
 *    zero and advances the epoch, so no pair left by an earlier call carries the next call's
 *    flag. The epoch is 32 bits and skips 2^32 - 1 (whose flag would be 0, the value of a pair
 *    never written): the call that would advance it there zeroes every pair word 3 counts and
 *    restarts it at 0, so the array never needs zeroing again. Without MOE_F_SYNC_PAIR an array
 *    may serve calls of different T if it is sized for the largest. A call that reported MOE_ERR_TIMEOUT may leave
 *    the array inconsistent: zero it again. Calls that may overlap on the GPU need separate sync
 *    arrays (and scratch).
 *    With MOE_F_SYNC_PAIR in flags, sync holds two halves of moe_layer_sync_ints words: the call
 *    uses the first half (the second with MOE_F_SYNC_ODD) and resets the other one (zero counters,
 *    epoch advanced; its CTA 0 does that on the way out, the other half's last call having
 *    completed before this call's dependency wait returned), instead of having its last CTA reset
 *    its own half (a device-wide fence and an atomic per CTA less at the end of every call).
 *    Consecutive calls on one stream that share the array must alternate halves; zero both halves
 *    before the first call. The halves are located by the call's own T, k and n_ff, so every call
 *    on a pair array has the same ones.
 *  - grp_expert [T*k], grp_start [T*k+1], n_groups [1], ent_src / ent_dst [T*k], xq
 *    [T][n_embd/32]: optional (NULL = not written) copies of the grouping and of the activation
 *    q8_1, for inspection.
 *  - x and gu must be 16-byte aligned, sync 8-byte aligned (else MOE_E_ALIGN).
 *  - Formats: any gate/up format; down MOE_NL4 or MOE_Q8_0 (else MOE_E_TYPE).
 *  - Limits: 0 < n_experts <= 2^26, T*k <= 512 and the T activation rows staged in shared memory (44 bytes per 32
 *    values, padded) must fit 64 KB (e.g. T <= 18 at n_embd 2560), else MOE_E_CAP; 32 rows of
 *    either blob must fit 96 KB, else MOE_E_SHAPE.
 *  - The launch's CTAs wait on one another (bounded, ~1 s, then MOE_ERR_TIMEOUT); the grid never
 *    exceeds one CTA per SM, so it needs the GPU's SMs to itself for the duration of the call.
 * MOE_F_PDL in flags chains the launch to the previous work on the stream with programmatic
 * dependent launch (it reads topk_ids and x only after that work has completed). */
typedef struct moe_layer_call {
    moe_wfmt gu_fmt, down_fmt;
    int32_t n_embd, n_ff, n_experts;
    const void* const* w_gu;   /* [n_experts] device pointers to gate/up blobs */
    const void* const* w_down; /* [n_experts] device pointers to down blobs */
    const int32_t* topk_ids;   /* [T][k] */
    int32_t T, k;
    const float* x;            /* [T][n_embd] */
    float* out;                /* [T*k][out_row_stride] */
    int64_t out_row_stride;
    float* gu;                 /* scratch [T*k][2*n_ff] */
    moe_q8_1* hq;              /* scratch [T*k][n_ff/32] */
    int32_t* sync;             /* [moe_layer_sync_ints(T, k, n_ff)], 8-byte aligned, zero before the first call */
    int32_t* grp_expert;       /* optional */
    int32_t* grp_start;        /* optional */
    int32_t* n_groups;         /* optional */
    int32_t* ent_src;          /* optional */
    int32_t* ent_dst;          /* optional */
    moe_q8_1* xq;              /* optional */
    int32_t* err;              /* optional */
    int32_t flags;             /* MOE_F_* */
} moe_layer_call;

/* Number of int32 sync words moe_expert_layer needs for windows of T tokens, top-k, n_ff:
 * 4 + T*k * (n_ff/32) * 18 (always even; 0 for invalid arguments). */
int64_t moe_layer_sync_ints(int T, int k, int n_ff);

int moe_expert_layer(const moe_layer_call* call, cudaStream_t stream);

/* One-launch form of moe_expert_grouped (#363 "experts: smaller and fewer launches for the
 * verify window's PCIe call", "What changes" and "Measured": the layer's second call, with no
 * group or with one group of two entries, should cost little). The same call - pre-built groups,
 * a device-side n_groups, entries that may start past 0, scattered destinations, rows outside the
 * call untouched - runs as one fused launch (gate/up, SwiGLU + q8_1 and down) instead of three, so
 * an empty call costs one launch: with *n_groups == 0 it reads nothing else and writes only the
 * sync words. Arguments as moe_expert_grouped, with:
 *  - grid_groups ignored (one CTA per SM takes the call's work items from a device counter);
 *  - sync: moe_grouped_fused_sync_ints(cap_groups, cap_entries, n_ff) int32 words, 8-byte aligned,
 *    zeroed before the first call, used like moe_expert_layer's (MOE_F_SYNC_PAIR / MOE_F_SYNC_ODD
 *    select halves the same way; the halves are located by cap_groups, cap_entries and n_ff);
 *  - down format MOE_NL4 or MOE_Q8_0; the n_xq_rows activation rows within moe_expert_layer's
 *    staging budget for T; max(cap_groups, cap_entries) <= 512 (else MOE_E_CAP); xq 4-byte and gu
 *    16-byte aligned.
 * Every gu, hq and out row of a computed group equals moe_expert_grouped's bit for bit. On bad
 * data one thing differs: a group holding an entry whose source or destination row is out of
 * range is skipped whole (MOE_ERR_ENTRY), where moe_expert_grouped skips that entry alone. The
 * launch's CTAs wait on one another as moe_expert_layer's do (bounded, MOE_ERR_TIMEOUT). */
int64_t moe_grouped_fused_sync_ints(int cap_groups, int cap_entries, int n_ff);
int moe_expert_grouped_fused(const moe_expert_call* call, int32_t* sync, cudaStream_t stream);

/* The residency split of #363 "experts: smaller and fewer launches for the verify window's PCIe
 * call" ("What changes": one call for the experts in VRAM, one for those that come over PCIe):
 * copy n host-resident blobs (an expert's gate/up and down blobs) into device staging slots before
 * the second call, whose pointer tables name the slots. Blobs in pinned (page-locked,
 * device-accessible) host memory that are 16-byte aligned with sizes a multiple of 16 are copied
 * by one kernel on `stream` that reads them over the CPU-GPU link through unified addressing (so
 * the expert call that follows may be launched with MOE_F_PDL and overlap its prologue with the
 * copy); any other blob by cudaMemcpyAsync (host_src should be pinned for the copies to be
 * asynchronous and capturable in a CUDA graph). dev_dst slots are 16-byte aligned device buffers
 * of at least bytes[i] bytes, owned by the caller. Errors: MOE_E_NULL, MOE_E_SHAPE (n < 0, a size
 * <= 0), MOE_E_ALIGN (a slot), MOE_E_CUDA. */
int moe_stage_blobs(const void* const* host_src, void* const* dev_dst, const int64_t* bytes, int n,
                    cudaStream_t stream);

/* ---------------------------------------------------------------- the steps either side
 * The router before the grouped call and the combine after it. The pages do not define the
 * router; this library takes the plainest reading. "The combined output" is what #3455 "GP100
 * (sm_60): 4-bit slots for resident IQ2_S / IQ3_XXS / IQ3_S gate/up experts" checks in "Passed". */

/* Router: for each token t < T, the k largest of logits[t][0 .. n_experts) (fp32, finite; ties:
 * the lower expert id first), in descending order, to topk_ids[t][0 .. k) (int32), and
 * weights[t][j] = e^(l_j - l_0) / sum over the k selected of e^(l_i - l_0) (fp32; this library's
 * exp, the sum in slot order, an IEEE divide). The ids feed moe_route_group / moe_expert_layer.
 * Limits: 1 <= k <= 32, k <= n_experts <= 1024, else MOE_E_SHAPE. */
int moe_router_topk(const float* logits, int T, int n_experts, int k, int32_t* topk_ids, float* weights,
                    cudaStream_t stream);

/* Combine: y[t][n] = sum over j < k of weights[t][j] * out[t*k + j][n] for n < n_embd, skipping
 * slots whose topk_ids[t][j] lies outside [0, n_experts) (ids the routing dropped: their out rows
 * are never written and never read). out rows are the entries' destination rows of the grouped
 * call (out_row_stride floats apart), y rows y_row_stride floats apart; fp32 fused multiply-adds
 * from zero in slot order. Errors: MOE_E_NULL, MOE_E_SHAPE (T outside [1, 65535], k <= 0, n_embd
 * <= 0, a stride below n_embd), MOE_E_CAP (n_experts <= 0). */
int moe_combine(const float* out, int64_t out_row_stride, const int32_t* topk_ids, const float* weights, int T, int k,
                int n_experts, int n_embd, float* y, int64_t y_row_stride, cudaStream_t stream);

/* ---------------------------------------------------------------- QSA decode block scores
 * A second decode workload of the verify window: #2059 "QSA decode: the window's block scores
 * with the queries in registers and six shuffles per block" ("What changed", "Bit for bit").
 *  - q: fp32 [T][MOE_QSA_HEADS][MOE_QSA_DIM], the window's queries, 1 <= T <= 4 (16-byte aligned);
 *  - keys: int8 [n_blocks][MOE_QSA_DIM], one pooled key per block of the context (4-byte
 *    aligned), key_scale: fp32 [n_blocks] (finite, > 0);
 *  - scores: fp32 [T][n_blocks].
 * For query t, block b and head h: lane l (0..31) takes dims 4l..4l+3, p_l = q0*k0, then
 * p_l = fma(q_i, k_i, p_l) for i = 1, 2, 3 (keys exact in fp32); the 32 partials are summed with
 * the warp sum's pairings (level j = 16, 8, 4, 2, 1: p_l <- p_l + p_(l xor j)); r_h =
 * max(dot_h * key_scale[b], 0); scores[t][b] = ((r_0 + r_1) + r_2) + r_3, plus 1e9 on the tail
 * block b = n_blocks - 1 (so that a top-k selection that follows always keeps it). Each step is
 * one fp32 rounding in that order, so the result does not depend on the launch. All pointers are
 * device pointers owned by the caller; nothing is allocated. Errors: MOE_E_NULL, MOE_E_SHAPE (T
 * outside [1, 4], n_blocks < 1 or > 2^40), MOE_E_ALIGN, MOE_E_CUDA. */
#define MOE_QSA_HEADS 4
#define MOE_QSA_DIM 128
int moe_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* key_scale, int64_t n_blocks,
                         float* scores, cudaStream_t stream);

/* Test hook: the per-32-block integer sums of `rows` consecutive rows of one blob (row bytes
 * apart) against one q8_1 row xq[K/32], computed by the same device decode and dot-product
 * code as the grouped kernels: isum[r][b] = sum_i w_code_i * q_i (exact int32). */
int moe_test_block_isum(moe_wfmt fmt, int K, const void* blob, int rows, const moe_q8_1* xq,
                        int32_t* isum, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GROUPED_H */
