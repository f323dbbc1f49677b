// api.cu - the C ABI (moe_grouped.h): host-side argument checks, launch planning and launches.
// Every function validates what the host can see, plans the launch geometry from the shapes
// and the device's SM count, and enqueues kernels on the caller's stream. Nothing here reads
// device memory or allocates.
#include <cstdio>
#include <mutex>

#include "internal.h"

using namespace moe;

namespace {

constexpr int kSmemPerSm = 228 * 1024;
constexpr int kMaxGroups = 1024;
constexpr int kMaxEntries = 4096;

bool cb_type(int t) { return t == MOE_CB2 || t == MOE_CB3; }
bool valid_type(int t) { return t >= MOE_Q8_0 && t <= MOE_CB2X; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static int cache[64] = {0};
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev] = n;
    return n;
}

int check_fmt(const moe_wfmt& f) {
    if (!valid_type(f.type)) return MOE_E_TYPE;
    if ((f.type == MOE_NL4 || cb_type(f.type)) && f.codebook == nullptr) return MOE_E_TYPE;
    if (reinterpret_cast<uintptr_t>(f.codebook) & 3u) return MOE_E_ALIGN;
    return MOE_OK;
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Launch geometry and shared-memory layout of one grouped GEMV (K weights per row, `rows`
// rows per expert), filled into `a` and `p`. One CTA per SM: a producer warp and up to 15
// consumer warps grouped in warp-sets; a set works on one tile (32 rows, lane = row) at a time,
// its warps splitting the row's 256-weight chunks; as many sets as fit in 15 warps.
int plan_gemv(int type, int K, int rows, int cap_groups, int cap_entries, int n_act_rows, GemvArgs& a,
              GemvPlan& p) {
    const int nch = K / 256;
    const int64_t rb = moe_row_bytes(type, K);
    if (nch <= 0 || nch > 32 || rb <= 0 || rows <= 0 || rows % 8) return MOE_E_SHAPE;
    if (cap_groups <= 0 || cap_groups > kMaxGroups || cap_entries <= 0 || cap_entries > kMaxEntries) return MOE_E_CAP;
    const bool cb = cb_type(type);
    // chunks per warp: the smallest that gives the most consumer warps (at most 15; warp-sets
    // of WPS = ceil(nch / CPW) warps, TP = 15 / WPS sets)
    int CPW = 1, best = 0;
    for (int cpw = 1; cpw <= nch; ++cpw) {
        const int wps = (nch + cpw - 1) / cpw;
        if (wps > 15) continue;
        const int cw = wps * (15 / wps);
        if (cw > best) { best = cw; CPW = cpw; }
    }
    const int WPS = (nch + CPW - 1) / CPW;
    const int RT = 32 * rb <= 96 * 1024 ? 32 : 16;
    const int nb = K / 32, nbp = nb + nb / 8;
    // activation rows: the whole matrix when it fits in 64 KB, else two 4-entry buffers
    const int act_row = 2 * nbp * 16 + nb * 8;
    const int act_cap = n_act_rows > 8 && n_act_rows * act_row <= 64 * 1024 ? n_act_rows : 8;
    const int actq = round_up(act_cap * 2 * nbp * 16, 128), act2 = round_up(act_cap * nb * 8, 128);
    const int grp = round_up(24 * cap_groups + 8 * (cap_groups + 1), 128);
    const int entb = round_up(8 * cap_entries, 128);
    const int fixed = (cb ? 32768 : 0) + actq + act2 + grp + entb + 256 + 512;
    const int stage_bytes = round_up(static_cast<int>(RT * rb) + 16, 128);
    const int part_bytes = nch * 4 * RT * 4;
    for (int TP = 15 / WPS > 0 ? 15 / WPS : 1; TP >= 1; --TP) {
        int stages = (kSmemPerSm - 1024 - fixed) / (stage_bytes + part_bytes);
        if (stages > 8) stages = 8;
        if (stages < 2 || stages < TP + 1) continue;
        int off = cb ? 32768 : 0;  // the codebook sits at offset 0
        a.off_ring = off;
        off += stages * stage_bytes;
        a.off_part = off;
        off += stages * part_bytes;
        a.off_actq = off;
        off += actq;
        a.off_act2 = off;
        off += act2;
        a.off_grp = off;
        off += grp;
        a.off_ent = off;
        off += entb;
        a.off_bar = off;
        off += 256;
        a.off_misc = off;
        off += 512;
        p.NT = 32 * (WPS * TP + 1);
        p.smem = off;
        a.K = K;
        a.rows = rows;
        a.row_bytes = static_cast<int>(rb);
        a.nch = nch;
        a.CPW = CPW;
        a.WPS = WPS;
        a.TP = TP;
        a.CW = WPS * TP;
        a.RT = RT;
        a.stages = stages;
        a.stage_bytes = stage_bytes;
        a.part_bytes = part_bytes;
        a.nb = nb;
        a.nbp = nbp;
        a.act_cap = act_cap;
        return MOE_OK;
    }
    return MOE_E_SHAPE;
}

cudaError_t occupancy(int type, int NT, int smem, int* ctas) {
    switch (type) {
    case MOE_Q8_0: return gemv_occupancy_q8_0(NT, smem, ctas);
    case MOE_Q4B: return gemv_occupancy_q4b(NT, smem, ctas);
    case MOE_NL4: return gemv_occupancy_nl4(NT, smem, ctas);
    case MOE_CB2: return gemv_occupancy_cb2(NT, smem, ctas);
    case MOE_CB3X: return gemv_occupancy_cb3x(NT, smem, ctas);
    case MOE_CB2X: return gemv_occupancy_cb2x(NT, smem, ctas);
    default: return gemv_occupancy_cb3(NT, smem, ctas);
    }
}

cudaError_t launch_gemv(int type, const GemvArgs& a, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    switch (type) {
    case MOE_Q8_0: return launch_gemv_q8_0(a, grid, NT, smem, s, pdl);
    case MOE_Q4B: return launch_gemv_q4b(a, grid, NT, smem, s, pdl);
    case MOE_NL4: return launch_gemv_nl4(a, grid, NT, smem, s, pdl);
    case MOE_CB2: return launch_gemv_cb2(a, grid, NT, smem, s, pdl);
    case MOE_CB3X: return launch_gemv_cb3x(a, grid, NT, smem, s, pdl);
    case MOE_CB2X: return launch_gemv_cb2x(a, grid, NT, smem, s, pdl);
    default: return launch_gemv_cb3(a, grid, NT, smem, s, pdl);
    }
}

// Persistent grid: every SM's resident CTAs, but no more than grid_groups x tiles per group.
int run_gemv(int type, GemvArgs& a, int grid_groups, cudaStream_t s, bool pdl) {
    GemvPlan p;
    int rc = plan_gemv(type, a.K, a.rows, a.cap_groups, a.cap_entries, a.n_act_rows, a, p);
    if (rc != MOE_OK) return rc;
    int ctas = 0;
    if (occupancy(type, p.NT, p.smem, &ctas) != cudaSuccess || ctas < 1) return MOE_E_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return MOE_E_CUDA;
    const int gg = grid_groups <= 0 || grid_groups > a.cap_groups ? a.cap_groups : grid_groups;
    const int64_t tiles = (a.rows + a.RT - 1) / a.RT;  // tiles of one group
    int64_t grid = static_cast<int64_t>(gg) * tiles;
    if (grid > static_cast<int64_t>(sms) * ctas) grid = static_cast<int64_t>(sms) * ctas;
    if (grid < 1) grid = 1;
    if (launch_gemv(type, a, static_cast<int>(grid), p.NT, p.smem, s, pdl) != cudaSuccess) return MOE_E_CUDA;
    return MOE_OK;
}

int check_dims(int n_embd, int n_ff) {
    if (n_embd <= 0 || n_ff <= 0 || n_embd % 256 || n_ff % 256) return MOE_E_SHAPE;
    return MOE_OK;
}

int gu_impl(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_gu, int n_experts, const int32_t* grp_expert,
            const int32_t* grp_start, const int32_t* n_groups, int cap_groups, int grid_groups, const moe_q8_1* xq,
            int n_xq_rows, const int32_t* ent_src, int cap_entries, float* gu, int32_t* err, cudaStream_t stream,
            bool pdl) {
    int rc = check_fmt(fmt);
    if (rc) return rc;
    if ((rc = check_dims(n_embd, n_ff))) return rc;
    if (!w_gu || !grp_expert || !grp_start || !n_groups || !xq || !ent_src || !gu) return MOE_E_NULL;
    if (n_experts <= 0 || cap_groups <= 0 || cap_entries <= 0 || n_xq_rows <= 0) return MOE_E_CAP;
    GemvArgs a = {};
    a.w = w_gu;
    a.n_experts = n_experts;
    a.K = n_embd;
    a.rows = 2 * n_ff;
    a.grp_expert = grp_expert;
    a.grp_start = grp_start;
    a.n_groups = n_groups;
    a.cap_groups = cap_groups;
    a.cap_entries = cap_entries;
    a.act = xq;
    a.n_act_rows = n_xq_rows;
    a.ent_in = ent_src;
    a.ent_out = nullptr;
    a.out = gu;
    a.out_rows = cap_entries;
    a.out_stride = 2 * static_cast<int64_t>(n_ff);
    a.err = err;
    a.codebook = fmt.codebook;
    a.prefetch_before_wait = 0;
    return run_gemv(fmt.type, a, grid_groups, stream, pdl);
}

int down_impl(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_down, int n_experts,
              const int32_t* grp_expert, const int32_t* grp_start, const int32_t* n_groups, int cap_groups,
              int grid_groups, const moe_q8_1* hq, int cap_entries, const int32_t* ent_dst, float* out,
              int64_t out_rows, int64_t out_row_stride, int32_t* err, cudaStream_t stream, bool pdl,
              bool prefetch_before_wait) {
    int rc = check_fmt(fmt);
    if (rc) return rc;
    if ((rc = check_dims(n_embd, n_ff))) return rc;
    if (!w_down || !grp_expert || !grp_start || !n_groups || !hq || !ent_dst || !out) return MOE_E_NULL;
    if (n_experts <= 0 || cap_groups <= 0 || cap_entries <= 0 || out_rows <= 0) return MOE_E_CAP;
    if (out_row_stride < n_embd) return MOE_E_SHAPE;
    GemvArgs a = {};
    a.w = w_down;
    a.n_experts = n_experts;
    a.K = n_ff;
    a.rows = n_embd;
    a.grp_expert = grp_expert;
    a.grp_start = grp_start;
    a.n_groups = n_groups;
    a.cap_groups = cap_groups;
    a.cap_entries = cap_entries;
    a.act = hq;
    a.n_act_rows = cap_entries;
    a.ent_in = nullptr;
    a.ent_out = ent_dst;
    a.out = out;
    a.out_rows = out_rows;
    a.out_stride = out_row_stride;
    a.err = err;
    a.codebook = fmt.codebook;
    a.prefetch_before_wait = prefetch_before_wait ? 1 : 0;
    return run_gemv(fmt.type, a, grid_groups, stream, pdl);
}

// ---------------------------------------------------------------- fused layer call

constexpr int kLayerMaxEntries = 512;  // routing: one thread per id

// Warp organisation of one phase: chunks per warp and warps per set as plan_gemv chooses them.
void phase_warps(int nch, GemvArgs& a) {
    int CPW = 1, best = 0;
    for (int cpw = 1; cpw <= nch; ++cpw) {
        const int wps = (nch + cpw - 1) / cpw;
        if (wps > 15) continue;
        const int cw = wps * (15 / wps);
        if (cw > best) { best = cw; CPW = cpw; }
    }
    a.CPW = CPW;
    a.WPS = (nch + CPW - 1) / CPW;
    a.TP = 15 / a.WPS;
    a.CW = a.WPS * a.TP;
}

// Geometry and shared-memory layout of one fused layer launch. The ring slot holds a gate/up
// tile (32 rows, or 16 when 32 rows exceed 96 KB) or a down tile of nsub x 32 rows.
constexpr int kLayerPtrCache = 256;  // experts whose pointers are cached in shared memory
constexpr int kUnitBytes = 4 * kLayerBatch * 32 * 4;  // gate/up unit buffers (4 units x kLayerBatch entries x 32 floats)
constexpr int kLayerThreads = 512;   // producer warp + 15 consumer warps
constexpr int kBatch = kLayerBatch;  // entries staged per down batch

// T activation rows; tables for n_tables entries and groups (0: T * k, a routed window's)
int plan_layer(int gt, int dt, int N, int F, int T, int k, int E, LayerArgs& L, int& NT, int& smem,
               int n_tables = 0) {
    const int n = n_tables > 0 ? n_tables : T * k;
    if (n <= 0 || n > kLayerMaxEntries) return MOE_E_CAP;
    GemvArgs& A = L.gu;
    GemvArgs& D = L.dn;
    const int64_t rbA = moe_row_bytes(gt, N), rbD = moe_row_bytes(dt, F);
    A.K = N; A.rows = 2 * F; A.nch = N / 256; A.nb = N / 32; A.nbp = A.nb + A.nb / 8;
    D.K = F; D.rows = N; D.nch = F / 256; D.nb = F / 32; D.nbp = D.nb + D.nb / 8;
    if (rbA <= 0 || rbD <= 0 || A.nch > 32 || D.nch > 32) return MOE_E_SHAPE;
    if (32 * rbD > 96 * 1024 || 16 * rbA > 96 * 1024) return MOE_E_SHAPE;
    A.row_bytes = static_cast<int>(rbA);
    D.row_bytes = static_cast<int>(rbD);
    phase_warps(A.nch, A);
    phase_warps(D.nch, D);
    A.RT = 32 * rbA <= 96 * 1024 ? 32 : 16;
    // activations: T token rows (gate/up role) and nbuf buffers of kLayerBatch entry rows (down
    // role, staged by the producer warp while the consumers work on the others; as many as fit, up
    // to kMaxHBufs, without a shallower ring, at least two), separate regions
    const int actqA = round_up(T * 2 * A.nbp * 16, 128), act2A = round_up(T * A.nb * 8, 128);
    if (actqA + act2A > 64 * 1024) return MOE_E_CAP;
    auto act_bytes = [&](int nbuf) {
        return actqA + act2A + round_up(nbuf * kBatch * 2 * D.nbp * 16, 128) + round_up(nbuf * kBatch * D.nb * 8, 128);
    };
    const int grp = round_up(24 * n + 4 * (n + 1), 128), entb = round_up(8 * n, 128);
    const int route = round_up(4 * (6 * n + 4), 128);
    const int cbb = cb_type(gt) ? 32768 : 0;
    const int ptrs = E <= kLayerPtrCache ? round_up(16 * E, 128) : 0;
    const int fixed2 = cbb + act_bytes(2) + 2 * grp + 2 * entb + route + ptrs + kUnitBytes + 512 + 1024;
    // one ring for both phases: a slot holds a gate/up tile (RT rows) or a down tile of nsub 32-row
    // sub-tiles; per stage a slot and its partial sums
    const int64_t tileA = A.RT * rbA;
    int nsub = static_cast<int>(tileA / (32 * rbD));
    nsub = nsub < 1 ? 1 : nsub > 4 ? 4 : nsub;
    D.RT = 32 * nsub;
    const int64_t tile = tileA > D.RT * rbD ? tileA : D.RT * rbD;
    const int stage = round_up(static_cast<int>(tile) + 16, 128);
    const int pA = A.nch * kLayerBatch * A.RT, pD = D.nch * kLayerBatch * D.RT;
    const int part = 4 * (pA > pD ? pA : pD);
    int S = (kSmemPerSm - 1024 - fixed2) / (stage + part);
    S = S > 8 ? 8 : S;
    if (S < 2) return MOE_E_SHAPE;
    int nbuf = 2;  // the most (up to kMaxHBufs) that keep the ring as deep as with two
    while (nbuf < kMaxHBufs && (kSmemPerSm - 1024 - (fixed2 - act_bytes(2) + act_bytes(nbuf + 1))) / (stage + part) >= S)
        ++nbuf;
    const int act = act_bytes(nbuf);
    const int actqD = round_up(nbuf * kBatch * 2 * D.nbp * 16, 128);
    int off = cbb;  // the gate/up codebook sits at offset 0
    A.off_ring = D.off_ring = off;
    off += S * stage;
    A.off_part = D.off_part = off;
    off += S * part;
    L.off_unit = off;
    off += kUnitBytes;
    A.off_actq = off;
    A.off_act2 = off + actqA;
    D.off_actq = off + actqA + act2A;
    D.off_act2 = D.off_actq + actqD;
    off += act;
    A.off_grp = off;
    off += grp;
    D.off_grp = off;
    off += grp;
    A.off_ent = off;
    off += entb;
    D.off_ent = off;
    off += entb;
    L.off_route = off;
    off += route;
    L.off_ptr = ptrs ? off : 0;
    off += ptrs;
    A.off_bar = D.off_bar = off;
    off += 512;  // 2 x 8 ring mbarriers, 2 x 16 descriptor mbarriers, 4 unit mbarriers (416 bytes)
    A.off_misc = D.off_misc = off;
    off += 1024;
    A.stages = D.stages = S;
    A.stage_bytes = D.stage_bytes = stage;
    A.part_bytes = D.part_bytes = part;
    A.act_cap = T;
    D.act_cap = nbuf * kBatch;
    A.cap_groups = A.cap_entries = D.cap_groups = D.cap_entries = n;
    L.T = T;
    L.k = k;
    L.n = n;
    L.F = F;
    L.nbj = F / 32;
    L.nsub = nsub;
    L.upg = F / 32;
    L.tpu = 64 / A.RT;
    NT = kLayerThreads;
    smem = off;
    return MOE_OK;
}

cudaError_t layer_occupancy(int gt, int dt, int NT, int smem, int* ctas) {
    switch (gt) {
    case MOE_Q8_0: return layer_occupancy_q8_0(dt, NT, smem, ctas);
    case MOE_Q4B: return layer_occupancy_q4b(dt, NT, smem, ctas);
    case MOE_NL4: return layer_occupancy_nl4(dt, NT, smem, ctas);
    case MOE_CB2: return layer_occupancy_cb2(dt, NT, smem, ctas);
    case MOE_CB3X: return layer_occupancy_cb3x(dt, NT, smem, ctas);
    case MOE_CB2X: return layer_occupancy_cb2x(dt, NT, smem, ctas);
    default: return layer_occupancy_cb3(dt, NT, smem, ctas);
    }
}

cudaError_t launch_layer(int gt, int dt, const LayerArgs& a, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    switch (gt) {
    case MOE_Q8_0: return launch_layer_q8_0(a, dt, grid, NT, smem, s, pdl);
    case MOE_Q4B: return launch_layer_q4b(a, dt, grid, NT, smem, s, pdl);
    case MOE_NL4: return launch_layer_nl4(a, dt, grid, NT, smem, s, pdl);
    case MOE_CB2: return launch_layer_cb2(a, dt, grid, NT, smem, s, pdl);
    case MOE_CB3X: return launch_layer_cb3x(a, dt, grid, NT, smem, s, pdl);
    case MOE_CB2X: return launch_layer_cb2x(a, dt, grid, NT, smem, s, pdl);
    default: return launch_layer_cb3(a, dt, grid, NT, smem, s, pdl);
    }
}

}  // namespace

extern "C" {

int64_t moe_row_bytes(int type, int K) {
    if (K <= 0 || K % 32) return 0;
    switch (type) {
    case MOE_Q8_0: return static_cast<int64_t>(K / 32) * 34;
    case MOE_Q4B: return static_cast<int64_t>(K / 32) * 20;
    case MOE_NL4: return static_cast<int64_t>(K / 32) * 18;
    case MOE_CB2: return K % 256 ? 0 : static_cast<int64_t>(K / 256) * 70;
    case MOE_CB3: return K % 256 ? 0 : static_cast<int64_t>(K / 256) * 102;
    case MOE_CB3X: return K % 256 ? 0 : static_cast<int64_t>(K / 256) * (128 + 8);
    case MOE_CB2X: return K % 256 ? 0 : static_cast<int64_t>(K / 256) * (64 + 8);
    }
    return 0;
}

const char* moe_strerror(int status) {
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_E_NULL: return "a required pointer is NULL";
    case MOE_E_TYPE: return "unsupported weight format or missing codebook";
    case MOE_E_SHAPE: return "unsupported shape (n_embd and n_ff must be positive multiples of 256)";
    case MOE_E_CAP: return "capacity or count not positive or too large";
    case MOE_E_CUDA: return "a CUDA runtime call failed";
    case MOE_E_ALIGN: return "pointer not suitably aligned";
    case MOE_E_SCRATCH: return "the call needs more scratch than the static buffer (MOE_STATIC_SCRATCH_BYTES) holds";
    }
    return "unknown status";
}

int moe_quantize_q8_1(const float* x, int64_t rows, int64_t cols, moe_q8_1* xq, cudaStream_t stream) {
    if (!x || !xq) return MOE_E_NULL;
    if (rows < 0 || cols <= 0 || cols % 32) return MOE_E_SHAPE;
    return launch_quantize_q8_1(x, rows, cols, xq, stream, false) == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int moe_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base, int32_t* grp_expert,
                    int32_t* grp_start, int32_t* n_groups, int32_t* ent_src, int32_t* ent_dst, int32_t* err,
                    cudaStream_t stream) {
    if (!topk_ids || !grp_expert || !grp_start || !n_groups || !ent_src || !ent_dst) return MOE_E_NULL;
    if (T <= 0 || k <= 0 || T * k > 1024) return MOE_E_SHAPE;
    if (n_experts <= 0 || entry_base < 0) return MOE_E_CAP;
    return launch_route_group(topk_ids, T, k, n_experts, entry_base, grp_expert, grp_start, n_groups, ent_src,
                              ent_dst, err, stream) == cudaSuccess
               ? MOE_OK
               : MOE_E_CUDA;
}

int moe_grouped_gu(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_gu, int n_experts,
                   const int32_t* grp_expert, const int32_t* grp_start, const int32_t* n_groups, int cap_groups,
                   int grid_groups, const moe_q8_1* xq, int n_xq_rows, const int32_t* ent_src, int cap_entries,
                   float* gu, int32_t* err, cudaStream_t stream) {
    return gu_impl(fmt, n_embd, n_ff, w_gu, n_experts, grp_expert, grp_start, n_groups, cap_groups, grid_groups, xq,
                   n_xq_rows, ent_src, cap_entries, gu, err, stream, false);
}

int moe_swiglu_q8_1(const float* gu, int n_ff, const int32_t* grp_start, const int32_t* n_groups, int cap_groups,
                    int cap_entries, moe_q8_1* hq, int32_t* err, cudaStream_t stream) {
    if (!gu || !grp_start || !n_groups || !hq) return MOE_E_NULL;
    if (n_ff <= 0 || n_ff % 32) return MOE_E_SHAPE;
    if (cap_groups <= 0 || cap_entries <= 0) return MOE_E_CAP;
    return launch_swiglu_q8_1(gu, n_ff, grp_start, n_groups, cap_groups, cap_entries, hq, err, stream, false) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_E_CUDA;
}

int moe_grouped_down(moe_wfmt fmt, int n_embd, int n_ff, const void* const* w_down, int n_experts,
                     const int32_t* grp_expert, const int32_t* grp_start, const int32_t* n_groups, int cap_groups,
                     int grid_groups, const moe_q8_1* hq, int cap_entries, const int32_t* ent_dst, float* out,
                     int64_t out_rows, int64_t out_row_stride, int32_t* err, cudaStream_t stream) {
    return down_impl(fmt, n_embd, n_ff, w_down, n_experts, grp_expert, grp_start, n_groups, cap_groups, grid_groups,
                     hq, cap_entries, ent_dst, out, out_rows, out_row_stride, err, stream, false, false);
}

int moe_expert_grouped(const moe_expert_call* c, cudaStream_t stream) {
    if (!c) return MOE_E_NULL;
    int rc;
    if ((rc = check_fmt(c->gu_fmt)) || (rc = check_fmt(c->down_fmt))) return rc;
    if ((rc = check_dims(c->n_embd, c->n_ff))) return rc;
    if (!c->w_gu || !c->w_down || !c->grp_expert || !c->grp_start || !c->n_groups || !c->xq || !c->ent_src ||
        !c->ent_dst || !c->gu || !c->hq || !c->out)
        return MOE_E_NULL;
    if (c->n_experts <= 0 || c->cap_groups <= 0 || c->cap_entries <= 0 || c->n_xq_rows <= 0 || c->out_rows <= 0)
        return MOE_E_CAP;
    if (c->out_row_stride < c->n_embd) return MOE_E_SHAPE;
    const bool pdl = (c->flags & MOE_F_PDL) != 0;
    rc = gu_impl(c->gu_fmt, c->n_embd, c->n_ff, c->w_gu, c->n_experts, c->grp_expert, c->grp_start, c->n_groups,
                 c->cap_groups, c->grid_groups, c->xq, c->n_xq_rows, c->ent_src, c->cap_entries, c->gu, c->err, stream,
                 pdl);
    if (rc) return rc;
    if (launch_swiglu_q8_1(c->gu, c->n_ff, c->grp_start, c->n_groups, c->cap_groups, c->cap_entries, c->hq, c->err,
                           stream, pdl) != cudaSuccess)
        return MOE_E_CUDA;
    // the down kernel's weights and groups are inputs of this call (complete before its gate/up
    // ran), so under PDL it may start streaming weight tiles before its dependency wait
    return down_impl(c->down_fmt, c->n_embd, c->n_ff, c->w_down, c->n_experts, c->grp_expert, c->grp_start,
                     c->n_groups, c->cap_groups, c->grid_groups, c->hq, c->cap_entries, c->ent_dst, c->out,
                     c->out_rows, c->out_row_stride, c->err, stream, pdl, pdl);
}

int64_t moe_layer_sync_ints(int T, int k, int n_ff) {
    if (T <= 0 || k <= 0 || n_ff <= 0 || n_ff % 32) return 0;
    // control words, then per entry and h block the flagged copy (kHxPairs 8-byte pairs); even, so
    // both halves of a sync pair stay 8-byte aligned
    return kSyncHx + static_cast<int64_t>(T) * k * (n_ff / 32) * kHxPairs * 2;
}

// The fused launch shared by moe_expert_layer (routed from ids) and moe_expert_grouped_fused
// (pre-built groups): formats, pointers and geometry already checked.
static int launch_fused(moe_wfmt gu_fmt, moe_wfmt down_fmt, int n_embd, int n_ff, int n_experts, const void* const* w_gu,
                        const void* const* w_down, LayerArgs& L, int NT, int smem, float* gu, int64_t gu_rows,
                        const moe_q8_1* act, float* out, int64_t out_rows, int64_t out_row_stride, moe_q8_1* hq,
                        int32_t* sync, int64_t half, int32_t* err, int32_t flags, cudaStream_t stream) {
    int ctas = 0;
    if (layer_occupancy(gu_fmt.type, down_fmt.type, NT, smem, &ctas) != cudaSuccess || ctas < 1) return MOE_E_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return MOE_E_CUDA;
    GemvArgs& A = L.gu;
    GemvArgs& D = L.dn;
    A.w = w_gu;
    D.w = w_down;
    A.n_experts = D.n_experts = n_experts;
    A.codebook = gu_fmt.codebook;
    D.codebook = down_fmt.codebook;
    A.err = D.err = err;
    A.act = act;
    A.n_act_rows = L.T;
    A.out = gu;
    A.out_rows = gu_rows;
    A.out_stride = 2 * static_cast<int64_t>(n_ff);
    D.act = hq;
    D.n_act_rows = L.n;
    D.out = out;
    D.out_rows = out_rows;
    D.out_stride = out_row_stride;
    L.hq = hq;
    L.sync = sync;
    L.sync_other = nullptr;
    if (flags & MOE_F_SYNC_PAIR) {  // two halves; this call uses one and zeroes the other
        const bool odd = (flags & MOE_F_SYNC_ODD) != 0;
        L.sync = sync + (odd ? half : 0);
        L.sync_other = sync + (odd ? 0 : half);
    }
    L.test_expire = (flags & MOE_F_TEST_EXPIRE) != 0;
    // one CTA per SM (co-resident), split on the device between the gate/up and the down roles
    const bool pdl = (flags & MOE_F_PDL) != 0;
    if (launch_layer(gu_fmt.type, down_fmt.type, L, sms, NT, smem, stream, pdl) != cudaSuccess) return MOE_E_CUDA;
    (void)n_embd;
    return MOE_OK;
}

int moe_expert_layer(const moe_layer_call* c, cudaStream_t stream) {
    if (!c) return MOE_E_NULL;
    int rc;
    if ((rc = check_fmt(c->gu_fmt)) || (rc = check_fmt(c->down_fmt))) return rc;
    if (c->down_fmt.type != MOE_NL4 && c->down_fmt.type != MOE_Q8_0) return MOE_E_TYPE;
    if ((rc = check_dims(c->n_embd, c->n_ff))) return rc;
    if (!c->w_gu || !c->w_down || !c->topk_ids || !c->x || !c->out || !c->gu || !c->hq || !c->sync)
        return MOE_E_NULL;
    if (c->T <= 0 || c->k <= 0) return MOE_E_SHAPE;
    if (c->n_experts <= 0 || c->n_experts > (1 << 26)) return MOE_E_CAP;  // routing keys: id << 5 | lane
    if (c->out_row_stride < c->n_embd) return MOE_E_SHAPE;
    if ((reinterpret_cast<uintptr_t>(c->x) | reinterpret_cast<uintptr_t>(c->gu)) & 15u) return MOE_E_ALIGN;
    if (reinterpret_cast<uintptr_t>(c->sync) & 7u) return MOE_E_ALIGN;
    LayerArgs L = {};
    int NT = 0, smem = 0;
    if ((rc = plan_layer(c->gu_fmt.type, c->down_fmt.type, c->n_embd, c->n_ff, c->T, c->k, c->n_experts, L, NT, smem)))
        return rc;
    L.ids = c->topk_ids;
    L.x = c->x;
    L.o_ge = c->grp_expert;
    L.o_gs = c->grp_start;
    L.o_ng = c->n_groups;
    L.o_es = c->ent_src;
    L.o_ed = c->ent_dst;
    L.o_xq = c->xq;
    return launch_fused(c->gu_fmt, c->down_fmt, c->n_embd, c->n_ff, c->n_experts, c->w_gu, c->w_down, L, NT, smem,
                        c->gu, L.n, nullptr, c->out, L.n, c->out_row_stride, c->hq, c->sync,
                        moe_layer_sync_ints(c->T, c->k, c->n_ff), c->err, c->flags, stream);
}

int64_t moe_grouped_fused_sync_ints(int cap_groups, int cap_entries, int n_ff) {
    if (cap_groups <= 0 || cap_entries <= 0) return 0;
    return moe_layer_sync_ints(cap_groups > cap_entries ? cap_groups : cap_entries, 1, n_ff);
}

int moe_expert_grouped_fused(const moe_expert_call* c, int32_t* sync, cudaStream_t stream) {
    if (!c) return MOE_E_NULL;
    int rc;
    if ((rc = check_fmt(c->gu_fmt)) || (rc = check_fmt(c->down_fmt))) return rc;
    if (c->down_fmt.type != MOE_NL4 && c->down_fmt.type != MOE_Q8_0) return MOE_E_TYPE;
    if ((rc = check_dims(c->n_embd, c->n_ff))) return rc;
    if (!c->w_gu || !c->w_down || !c->grp_expert || !c->grp_start || !c->n_groups || !c->xq || !c->ent_src ||
        !c->ent_dst || !c->gu || !c->hq || !c->out || !sync)
        return MOE_E_NULL;
    if (c->n_experts <= 0 || c->n_experts > (1 << 26) || c->cap_groups <= 0 || c->cap_entries <= 0 ||
        c->n_xq_rows <= 0 || c->out_rows <= 0)
        return MOE_E_CAP;
    if (c->out_row_stride < c->n_embd) return MOE_E_SHAPE;
    if ((reinterpret_cast<uintptr_t>(c->xq) & 3u) || (reinterpret_cast<uintptr_t>(c->gu) & 15u)) return MOE_E_ALIGN;
    if (reinterpret_cast<uintptr_t>(sync) & 7u) return MOE_E_ALIGN;
    const int n = c->cap_groups > c->cap_entries ? c->cap_groups : c->cap_entries;
    LayerArgs L = {};
    int NT = 0, smem = 0;
    if ((rc = plan_layer(c->gu_fmt.type, c->down_fmt.type, c->n_embd, c->n_ff, c->n_xq_rows, 1, c->n_experts, L, NT,
                         smem, n)))
        return rc;
    L.given = 1;
    L.g_expert = c->grp_expert;
    L.g_start = c->grp_start;
    L.g_ng = c->n_groups;
    L.g_src = c->ent_src;
    L.g_dst = c->ent_dst;
    L.g_cap_groups = c->cap_groups;
    L.g_cap_entries = c->cap_entries;
    L.g_out_rows = c->out_rows;
    return launch_fused(c->gu_fmt, c->down_fmt, c->n_embd, c->n_ff, c->n_experts, c->w_gu, c->w_down, L, NT, smem,
                        c->gu, c->cap_entries, c->xq, c->out, c->out_rows, c->out_row_stride, c->hq, sync,
                        moe_grouped_fused_sync_ints(c->cap_groups, c->cap_entries, c->n_ff), c->err, c->flags,
                        stream);
}

int moe_stage_blobs(const void* const* host_src, void* const* dev_dst, const int64_t* bytes, int n,
                    cudaStream_t stream) {
    if (n < 0) return MOE_E_SHAPE;
    if (n > 0 && (!host_src || !dev_dst || !bytes)) return MOE_E_NULL;
    for (int i = 0; i < n; ++i) {
        if (!host_src[i] || !dev_dst[i]) return MOE_E_NULL;
        if (bytes[i] <= 0) return MOE_E_SHAPE;
        if (reinterpret_cast<uintptr_t>(dev_dst[i]) & 15u) return MOE_E_ALIGN;
    }
    // pinned (device-accessible) 16-byte aligned blobs of whole 16-byte words: one copy kernel
    // that reads them through unified addressing; any other blob: cudaMemcpyAsync (a kernel must
    // never dereference pageable host memory)
    const void* ksrc[kStageMax];
    void* kdst[kStageMax];
    int64_t kbytes[kStageMax];
    int nk = 0;
    for (int i = 0; i < n; ++i) {
        cudaPointerAttributes at{};
        const bool pinned = cudaPointerGetAttributes(&at, host_src[i]) == cudaSuccess &&
                            at.type == cudaMemoryTypeHost && at.devicePointer != nullptr;
        if (!pinned) cudaGetLastError();  // (clear a lookup's error state)
        const uintptr_t al =
            reinterpret_cast<uintptr_t>(pinned ? at.devicePointer : host_src[i]) | reinterpret_cast<uintptr_t>(dev_dst[i]) |
            static_cast<uintptr_t>(bytes[i]);
        if (pinned && (al & 15u) == 0) {
            ksrc[nk] = at.devicePointer;
            kdst[nk] = dev_dst[i];
            kbytes[nk] = bytes[i];
            if (++nk == kStageMax) {
                if (launch_stage_blobs(ksrc, kdst, kbytes, nk, stream) != cudaSuccess) return MOE_E_CUDA;
                nk = 0;
            }
        } else if (cudaMemcpyAsync(dev_dst[i], host_src[i], static_cast<size_t>(bytes[i]), cudaMemcpyHostToDevice,
                                   stream) != cudaSuccess) {
            return MOE_E_CUDA;
        }
    }
    if (nk && launch_stage_blobs(ksrc, kdst, kbytes, nk, stream) != cudaSuccess) return MOE_E_CUDA;
    return MOE_OK;
}

int moe_router_topk(const float* logits, int T, int n_experts, int k, int32_t* topk_ids, float* weights,
                    cudaStream_t stream) {
    if (!logits || !topk_ids || !weights) return MOE_E_NULL;
    if (T <= 0 || k <= 0 || k > 32 || n_experts < k || n_experts > 1024) return MOE_E_SHAPE;
    return launch_router_topk(logits, T, n_experts, k, topk_ids, weights, stream) == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

int moe_combine(const float* out, int64_t out_row_stride, const int32_t* topk_ids, const float* weights, int T, int k,
                int n_experts, int n_embd, float* y, int64_t y_row_stride, cudaStream_t stream) {
    if (!out || !topk_ids || !weights || !y) return MOE_E_NULL;
    if (T <= 0 || T > 65535 || k <= 0 || n_embd <= 0 || out_row_stride < n_embd || y_row_stride < n_embd)
        return MOE_E_SHAPE;
    if (n_experts <= 0) return MOE_E_CAP;
    return launch_combine(out, out_row_stride, topk_ids, weights, T, k, n_experts, n_embd, y, y_row_stride, stream) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_E_CUDA;
}

int moe_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* key_scale, int64_t n_blocks,
                         float* scores, cudaStream_t stream) {
    if (!q || !keys || !key_scale || !scores) return MOE_E_NULL;
    if (T < 1 || T > 4 || n_blocks < 1 || n_blocks > (int64_t{1} << 40)) return MOE_E_SHAPE;
    if ((reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(keys) & 3u) ||
        (reinterpret_cast<uintptr_t>(key_scale) & 3u) || (reinterpret_cast<uintptr_t>(scores) & 3u))
        return MOE_E_ALIGN;
    return launch_qsa_block_scores(q, T, keys, key_scale, n_blocks, scores, stream) == cudaSuccess ? MOE_OK
                                                                                                   : MOE_E_CUDA;
}

int moe_transcode_cb(moe_wfmt src, int dst_type, int K, int rows, int n_blobs, const void* const* src_blobs,
                     void* const* dst_blobs, int32_t* err, cudaStream_t stream) {
    if (!cb_type(src.type) || (dst_type != MOE_CB3X && dst_type != MOE_CB2X)) return MOE_E_TYPE;
    int rc = check_fmt(src);
    if (rc) return rc;
    if (!src_blobs || !dst_blobs) return MOE_E_NULL;
    if (K <= 0 || K % 256 || rows <= 0 || n_blobs <= 0) return MOE_E_SHAPE;
    return launch_transcode_cb(src.type, src.codebook, dst_type, K, rows, n_blobs, src_blobs, dst_blobs, err,
                               stream) == cudaSuccess
               ? MOE_OK
               : MOE_E_CUDA;
}

int moe_test_block_isum(moe_wfmt fmt, int K, const void* blob, int rows, const moe_q8_1* xq, int32_t* isum,
                        cudaStream_t stream) {
    int rc = check_fmt(fmt);
    if (rc) return rc;
    if (!blob || !xq || !isum) return MOE_E_NULL;
    if (K <= 0 || K % 256 || rows <= 0) return MOE_E_SHAPE;
    cudaError_t e;
    switch (fmt.type) {
    case MOE_Q8_0: e = launch_isum_q8_0(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    case MOE_Q4B: e = launch_isum_q4b(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    case MOE_NL4: e = launch_isum_nl4(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    case MOE_CB2: e = launch_isum_cb2(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    case MOE_CB3X: e = launch_isum_cb3x(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    case MOE_CB2X: e = launch_isum_cb2x(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    default: e = launch_isum_cb3(fmt.codebook, K, blob, rows, xq, isum, stream); break;
    }
    return e == cudaSuccess ? MOE_OK : MOE_E_CUDA;
}

}  // extern "C"
