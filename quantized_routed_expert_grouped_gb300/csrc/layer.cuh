// layer.cuh - the fused layer kernel: one launch runs a layer's whole hot path (routing/grouping,
// activation q8_1, grouped gate/up, SwiGLU + q8_1, grouped down) for one verify window.
//
// What it computes is the composition of the separate steps (#363 "experts: smaller and fewer
// launches for the verify window's PCIe call", "What changes"; #2058 "Verify window: the routed
// experts' gate/up with the group's q8_1 rows in shared memory", "What changed"), with the same
// arithmetic in the same order, so its outputs equal the separate kernels' bit for bit.
//
// How (GB300 design):
//  * Every CTA groups the window's top-k ids itself (one warp: ballots and shuffles when T*k <= 32);
//    CTA 0 also writes the grouping and the activation q8_1 rows to global memory for inspection.
//    The expert pointer tables, like the codebooks, are read before the dependency wait.
//  * Two phases on every CTA, one after the other: gate/up, then down. Gate/up work comes in units
//    of one 32-value h block of one group, dealt round-robin in group order (tile-sized work,
//    evenly spread); down work is a contiguous, cost-balanced run of (group, 8-row block) pairs
//    per CTA, which waits only for its own (at most two) groups.
//  * A gate/up unit is gate rows 32jb .. 32jb+31 and up rows F+32jb .. F+32jb+31 of one expert:
//    two ring tiles (four when rows are long) of 16 gate rows and the matching 16 up rows (two
//    bulk copies into one slot). Chunk warps (a warp per 256-weight chunk, lane = row) only compute
//    and arrive on the slot's chunk-done barrier; an epilogue warp per unit sums the chunk
//    partials, releases the slot, writes the gate/up rows and keeps SwiGLU(gate, up) (product
//    rounded on its own) in its lanes, so the unit's 32 h values per entry end up one per lane: it
//    writes their q8_1 block to hq and adds one to the group's counter (after a fence). Every h
//    block is computed once, and no compute warp waits on an epilogue.
//  * The activations are staged as q8_1 by every CTA (one lane quad per block).
//  * A down tile holds up to nsub 32-row sub-tiles (the ring slot is sized for a gate/up tile); its
//    (sub-tile, 256-weight chunk) work items are dealt to the consumer warps in turn across tiles;
//    the CTA waits (bounded) for its groups' counters to reach F/32 and stages their q8_1 h rows
//    from hq once (two groups of up to 4 entries; larger runs restage per group or 4-entry batch).
//  * Both phases stream their tiles through one ring of shared-memory slots (1-D bulk copies and
//    mbarriers, issued by a producer warp); the down tiles follow the gate/up tiles in the ring,
//    so they are prefetched while the last gate/up tiles are computed.
//  * The counters live in a caller-owned int array that must be zero before the first call; the
//    last CTA to finish (a global exit counter) zeroes them again, so every call starts clean.
//  * Every wait (mbarriers, group counters) has a time limit; on expiry the kernel sets
//    MOE_ERR_TIMEOUT, skips the remaining work, waits (bounded) for its own copies in flight
//    and still takes part in the exit count.
#pragma once

#include "gemv.cuh"
#include "q8_1.cuh"
#include "route.cuh"

namespace moe {

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until *p >= target (acquire); false after kWaitLimitNs.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target) {
    if (ld_acquire(p) >= target) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(64);
        if (ld_acquire(p) >= target) return true;
        if ((it & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// q8_1 of one 32-value block held by the 4 lanes of an aligned lane quad (quad lane j holds
// values 8j .. 8j+7; qmask: the quad's lanes): the lane's code words (codes 8j .. 8j+7), and on
// every quad lane the header d16 | s16 << 16 and the exact code sum. Same arithmetic as
// warp_q8_1 (exact maximum, IEEE divides, round half away from zero), so the same bytes.
__device__ __forceinline__ void quad_q8_1(const float v[8], unsigned qmask, uint32_t w[2], uint32_t& hdr, int& S) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 1, 4));
    amax = fmaxf(amax, __shfl_xor_sync(qmask, amax, 2, 4));
    const float d = __fdiv_rn(amax, 127.0f);
    int s = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int q = d == 0.0f ? 0 : static_cast<int>(roundf(__fdiv_rn(v[4 * k + b], d)));
            s += q;
            word |= (static_cast<uint32_t>(q) & 0xffu) << (8 * b);
        }
        w[k] = word;
    }
    s += __shfl_xor_sync(qmask, s, 1, 4);
    s += __shfl_xor_sync(qmask, s, 2, 4);
    S = s;
    const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
    const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, static_cast<float>(s))));
    hdr = d16 | (s16 << 16);
}

// Quad lane j's part of a q8_1 block into staged slot `slot`, block b (the layout stage_block
// writes): code words 2j, 2j+1; lane 0 also the (d, aux) pair.
template <int TYPE>
__device__ __forceinline__ void stage_quad(const GemvArgs& a, uint8_t* smem, int slot, int b, int j, const uint32_t w[2],
                                           uint32_t hdr, int S) {
    uint32_t c0 = w[0], c1 = w[1];
    if constexpr (TYPE == MOE_NL4) {
        c0 = prmt(c0, 0u, 0x3120u);
        c1 = prmt(c1, 0u, 0x3120u);
    }
    const int bp = b + (b >> 3);
    *reinterpret_cast<uint2*>(smem + a.off_actq + ((slot * 2 + (j >> 1)) * a.nbp + bp) * 16 + (j & 1) * 8) =
        make_uint2(c0, c1);
    if (j == 0) {
        float aux = 0.0f;
        if constexpr (Fmt<TYPE>::SLOT) {
            aux = __int_as_float(S * -(2 * Fmt<TYPE>::BIAS - 1));
        } else if constexpr (Fmt<TYPE>::CB) {
            aux = __int_as_float(S);
        } else if constexpr (TYPE == MOE_Q4B) {
            aux = h2f_bits(hdr >> 16);
        }
        reinterpret_cast<float2*>(smem + a.off_act2)[slot * a.nb + b] = make_float2(h2f_bits(hdr), aux);
    }
}

// Quad lane j's part of a q8_1 block stored at dst (36 bytes, 4-byte aligned).
__device__ __forceinline__ void put_quad(moe_q8_1* dst, int j, const uint32_t w[2], uint32_t hdr) {
    uint32_t* p = reinterpret_cast<uint32_t*>(dst);
    if (j == 0) p[0] = hdr;
    p[1 + 2 * j] = w[0];
    p[2 + 2 * j] = w[1];
}

// Routing/grouping of n <= 32 ids by one warp (lane i owns id i): the same grouping as route_cta
// (groups by ascending expert id, entries by ascending (t, slot), numbered from 0), from ballots and
// shuffles. Writes grp_expert, grp_start (G+1), *n_groups, ent_src, ent_dst (shared memory).
__device__ __forceinline__ void route_warp(const int32_t* ids, int n, int k, int n_experts, int* rgx, int* rgs, int* rng,
                                           int* rsrc, int* rdst, int32_t* err, bool report, int lane) {
    int v = -1;
    if (lane < n) {
        v = ids[lane];
        if (v < 0 || v >= n_experts) {
            if (report) set_err(err, MOE_ERR_ROUTE);
            v = -1;
        }
    }
    const bool valid = v >= 0;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned same = __match_any_sync(0xffffffffu, v);
    const bool first = valid && __ffs(same) - 1 == lane;
    const unsigned fmask = __ballot_sync(0xffffffffu, first);
    int rank = 0, grp = 0;
#pragma unroll
    for (int jl = 0; jl < 32; ++jl) {
        const int vj = __shfl_sync(0xffffffffu, v, jl);
        const bool lt = vj >= 0 && vj < v;
        rank += lt || (vj == v && jl < lane);
        grp += lt && ((fmask >> jl) & 1u);
    }
    if (valid) {
        rsrc[rank] = lane / k;
        rdst[rank] = lane;
        if (first) {
            rgx[grp] = v;
            rgs[grp] = rank;
        }
    }
    if (lane == 0) {
        rgs[__popc(fmask)] = __popc(vmask);
        *rng = __popc(fmask);
    }
}

// Flattened (group, 8-row block) index at which the cumulative cost reaches `target` (cum: int32
// inclusive prefix of cost * rbpg, cum[0] = 0).
__device__ __forceinline__ int locate32(const GroupInfo* gi, const int* cum, int G, int rbpg, int target) {
    if (target >= cum[G]) return G * rbpg;
    int lo = 0, hi = G - 1;  // first g with cum[g+1] > target (its cost is > 0)
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid + 1] > target) hi = mid;
        else lo = mid + 1;
    }
    return lo * rbpg + (target - cum[lo]) / gi[lo].cost;
}

// One warp: group tables for both phases (weight pointers from the shared-memory cache when it
// holds them; cost 0 marks a skipped group; a down 8-row block of a group of n entries costs
// alpha + n), the entry tables, the inspection copies (CTA 0) and this CTA's down range
// misc[10..11] (a contiguous, cost-balanced run of (group, 8-row block) pairs).
template <int GT, int DT>
__device__ __forceinline__ void build_tables(const LayerArgs& L, const uint8_t* const* pcA, const uint8_t* const* pcD,
                                             const int* rgx, const int* rgs, const int* rng, const int* rsrc,
                                             const int* rdst, GroupInfo* giA, GroupInfo* giD, int* cumD, int2* entA,
                                             int2* entD, int* misc, int lane) {
    const GemvArgs& A = L.gu;
    const GemvArgs& D = L.dn;
    const int G = *rng, ntot = rgs[G], rbpgD = D.rows >> 3;
    const bool report = blockIdx.x == 0;
    int run = 0;
    for (int base = 0; base < G; base += 32) {
        const int g = base + lane;
        int cD = 0;
        if (g < G) {
            const int x = rgx[g], e0 = rgs[g], e1 = rgs[g + 1];
            const uint8_t* pa = pcA ? pcA[x] : static_cast<const uint8_t*>(A.w[x]);
            const uint8_t* pd = pcD ? pcD[x] : static_cast<const uint8_t*>(D.w[x]);
            const bool ok = ((reinterpret_cast<uintptr_t>(pa) | reinterpret_cast<uintptr_t>(pd)) & 15u) == 0;
            if (!ok && report) set_err(A.err, MOE_ERR_ALIGN);
            cD = ok ? D.alpha + (e1 - e0) : 0;
            giA[g] = GroupInfo{pa, x, e0, e1, ok ? 1 : 0};
            giD[g] = GroupInfo{pd, x, e0, e1, cD};
        }
        int sD = cD * rbpgD;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, sD, o);
            if (lane >= o) sD += y;
        }
        if (g < G) cumD[g + 1] = run + sD;
        run += __shfl_sync(0xffffffffu, sD, 31);
    }
    if (lane == 0) cumD[0] = 0;
    for (int e = lane; e < ntot; e += 32) {
        entA[e] = make_int2(rsrc[e], e);
        entD[e] = make_int2(e, rdst[e]);
    }
    if (report) {
        if (L.o_ng && lane == 0) *L.o_ng = G;
        for (int g = lane; g <= G; g += 32) {
            if (L.o_gs) L.o_gs[g] = rgs[g];
            if (L.o_ge && g < G) L.o_ge[g] = rgx[g];
        }
        for (int e = lane; e < ntot; e += 32) {
            if (L.o_es) L.o_es[e] = rsrc[e];
            if (L.o_ed) L.o_ed[e] = rdst[e];
        }
    }
    __syncwarp();
    if (lane < 2) {  // boundary c * tot / grid without 64-bit division (tot < 2^31)
        const int c = blockIdx.x + lane, grid = gridDim.x;
        const int target = (run / grid) * c + ((run % grid) * c) / grid;
        misc[10 + lane] = locate32(giD, cumD, G, rbpgD, target);
    }
    __syncwarp();
}

__device__ __forceinline__ void bar_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// One warp's partial sums for one 256-weight chunk c of 32 rows at `rows` (lane = row):
// part[(c*4 + e)*RT + lane] for the batch's ne entries, staged in slots[0 .. ne-1].
template <int TYPE>
__device__ __forceinline__ void chunk_part(const GemvArgs& a, const uint8_t* smem, const uint8_t* rows, float* part, int ne,
                                           int c, int lane, uint32_t loff, const uint32_t tab[4], const int slots[4]) {
    if (ne == 1) {
        float acc[1];
        lane_chunk<TYPE, 1>(a, smem, rows, lane, c, loff, tab, slots, acc);
        part[c * kMaxEntriesPerPass * a.RT + lane] = acc[0];
    } else if (ne == 2) {
        float acc[2];
        lane_chunk<TYPE, 2>(a, smem, rows, lane, c, loff, tab, slots, acc);
#pragma unroll
        for (int e = 0; e < 2; ++e) part[(c * kMaxEntriesPerPass + e) * a.RT + lane] = acc[e];
    } else {  // 3 entries run the 4-entry code (the fourth slot repeats the third)
        float acc[4];
        lane_chunk<TYPE, 4>(a, smem, rows, lane, c, loff, tab, slots, acc);
#pragma unroll
        for (int e = 0; e < 4; ++e) part[(c * kMaxEntriesPerPass + e) * a.RT + lane] = acc[e];
    }
}

template <int GT, int DT>
__global__ void __launch_bounds__(kMaxThreads, 1) layer_kernel(const LayerArgs L) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const GemvArgs& A = L.gu;
    const GemvArgs& D = L.dn;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NT = blockDim.x;
    const int n = L.n, F = L.F, upg = L.upg, tpu = L.tpu;
    const int SB = A.stages;  // ring slots
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + A.off_bar);
    uint64_t* empty = full + SB;
    uint64_t* cdone = empty + SB;  // gate/up: a tile's chunk partials are written (one arrival per chunk)
    // misc: [0] tiles issued, [1] abort flag, [2] last-CTA flag, [12] gate/up CTAs,
    // [16 + u] tiles done of unit buffer u, [32 + s] sub-tiles done of slot s,
    // [64 + 8s + b] warps done with sub-tile b of slot s
    int* misc = reinterpret_cast<int*>(smem + A.off_misc);
    volatile int* vmisc = misc;
    GroupInfo* giA = reinterpret_cast<GroupInfo*>(smem + A.off_grp);
    GroupInfo* giD = reinterpret_cast<GroupInfo*>(smem + D.off_grp);
    int* cumD = reinterpret_cast<int*>(giD + n);  // down cost prefix [G + 1]
    int2* entA = reinterpret_cast<int2*>(smem + A.off_ent);  // entry -> (token row, gate/up row)
    int2* entD = reinterpret_cast<int2*>(smem + D.off_ent);  // entry -> (h row, output row)
    int* rs = reinterpret_cast<int*>(smem + L.off_route);
    int* sid = rs;
    int* sfirst = rs + n;
    int* scount = rs + 2 * n;
    int* rgx = scount + 2;
    int* rgs = rgx + n;
    int* rng = rgs + n + 1;
    int* rsrc = rng + 1;
    int* rdst = rsrc + n;
    float* ubuf = reinterpret_cast<float*>(smem + L.off_unit);  // [stages][4 entries][32] h values
    // expert pointer tables cached in shared memory (static data: read before the dependency wait)
    const uint8_t** pcA = L.off_ptr ? reinterpret_cast<const uint8_t**>(smem + L.off_ptr) : nullptr;
    const uint8_t** pcD = pcA ? pcA + A.n_experts : nullptr;

    if (tid < 128) misc[tid] = 0;
    if (tid == 0)
        for (int s = 0; s < SB; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&cdone[s], A.nch);
        }
    fence_barrier_init();
    // static data before the dependency wait: codebook replicas, NL4 tables, pointer tables
    if (warp > 0) stage_codebook<GT>(A, smem, tid - 32, NT - 32);
    if (pcA)
        for (int x = tid; x < A.n_experts; x += NT) {
            pcA[x] = static_cast<const uint8_t*>(A.w[x]);
            pcD[x] = static_cast<const uint8_t*>(D.w[x]);
        }
    uint32_t tabA[4], tabD[4];
    load_table<GT>(A, tabA);
    load_table<DT>(D, tabD);
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    // ---- routing/grouping and tables: one warp when n <= 32, else the whole CTA routes and
    // warp 0 builds the tables
    if (n > 32) {
        route_cta(L.ids, n, L.k, A.n_experts, 0, sid, sfirst, scount, rgx, rgs, rng, rsrc, rdst, A.err,
                  blockIdx.x == 0);
        __syncthreads();
    }
    if (warp == 0) {
        if (n <= 32) route_warp(L.ids, n, L.k, A.n_experts, rgx, rgs, rng, rsrc, rdst, A.err, blockIdx.x == 0, lane);
        __syncwarp();
        build_tables<GT, DT>(L, pcA, pcD, rgx, rgs, rng, rsrc, rdst, giA, giD, cumD, entA, entD, misc, lane);
        __threadfence_block();
        bar_arrive(3, NT);  // tables ready
    } else {
        // meanwhile the consumer warps quantize the activations (independent of the grouping)
        const int ct = tid - 32, cnt = NT - 32;
        // ---- activations: x -> q8_1 of all T tokens, staged in slot t; one lane quad per block
        {
            const int nb = A.nb, j = ct & 3, nq = cnt >> 2, tot = L.T * nb;
            const unsigned qmask = 0xFu << (lane & 28);
            for (int i0 = ct >> 2; i0 < tot; i0 += 4 * nq) {
                float4 f[4][2];  // four blocks' loads in flight before any arithmetic
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * nq;
                    if (i < tot) {
                        const int t = i / nb, b = i - t * nb;
                        const float4* xp =
                            reinterpret_cast<const float4*>(L.x + static_cast<int64_t>(t) * A.K + b * 32 + 8 * j);
                        f[u][0] = __ldg(xp);
                        f[u][1] = __ldg(xp + 1);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + u * nq;
                    if (i >= tot) break;
                    const int t = i / nb, b = i - t * nb;
                    const float v[8] = {f[u][0].x, f[u][0].y, f[u][0].z, f[u][0].w,
                                        f[u][1].x, f[u][1].y, f[u][1].z, f[u][1].w};
                    uint32_t w[2], hdr;
                    int Ssum;
                    quad_q8_1(v, qmask, w, hdr, Ssum);
                    stage_quad<GT>(A, smem, t, b, j, w, hdr, Ssum);
                    if (blockIdx.x == 0 && L.o_xq) put_quad(L.o_xq + i, j, w, hdr);
                }
            }
        }
        named_sync(3, NT);  // with warp 0's arrival: tables ready, activations staged
    }
    const int G = *rng, ngu = gridDim.x;
    const int32_t* ready = L.sync;  // per group: h blocks written (complete at F/32)
    int qA = 0;  // gate/up tiles of this CTA (the down ring's tiles are numbered after them)

    {
        const int S = A.stages, RT = A.RT, half = RT >> 1, nunits = G * upg;
        if (warp == 0) {
            // ---- gate/up producer: this CTA's units (round-robin in group order), tpu tiles each,
            // each tile two bulk copies (gate rows, up rows) into one slot
            if (lane == 0) {
                int issued = 0;
                const uint32_t hb = static_cast<uint32_t>(half) * static_cast<uint32_t>(A.row_bytes);
                for (int i = blockIdx.x; i < nunits; i += ngu) {
                    const int g = i / upg, jb = i - g * upg;
                    const GroupInfo gr = giA[g];
                    if (gr.cost == 0) continue;
                    bool stop = false;
                    for (int h = 0; h < tpu; ++h) {
                        const int s = issued % S;
                        if (vmisc[1] || (issued >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(issued / S - 1) & 1u))) {
                            if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                            vmisc[1] = 1;
                            stop = true;
                            break;
                        }
                        uint8_t* dst = smem + A.off_ring + static_cast<size_t>(s) * A.stage_bytes;
                        const size_t rg = static_cast<size_t>(32 * jb + h * half);
                        mbar_arrive_expect_tx(&full[s], 2 * hb);
                        bulk_g2s(dst, gr.ptr + rg * A.row_bytes, hb, &full[s]);
                        bulk_g2s(dst + hb, gr.ptr + (rg + F) * A.row_bytes, hb, &full[s]);
                        ++issued;
                        __threadfence_block();
                        vmisc[0] = issued;
                    }
                    if (stop) break;
                }
            }
        } else {
            const int cw = warp - 1, ncw = (NT >> 5) - 1, ct = tid - 32, cnt = ncw * 32;
            const uint32_t loff = GT == MOE_CB3 ? lane * 4u : (lane & 15u) * 8u;
            // ---- gate/up tiles, one at a time with all consumer warps (a warp per 256-weight chunk,
            // lane = row; the last warp to finish sums the chunks): SwiGLU in the tile epilogue, q8_1 of
            // h by the tile that completes the unit, then the group's counter
            const int64_t gst = A.out_stride;
            bool multi = false;
            for (int g = 0; g < G; ++g) multi |= giA[g].cost != 0 && giA[g].e1 - giA[g].e0 > kMaxEntriesPerPass;
            const int cwc = A.nch < ncw ? A.nch : ncw;  // chunk warps
            const int ew = ncw - cwc > 4 ? 4 : ncw - cwc;  // epilogue warps
            if (!multi && ew > 0) {
                // Chunk warps only compute (a warp per chunk, lane = row) and arrive on the slot's
                // chunk-done barrier; epilogue warp u % ew takes unit u: per tile it sums the chunk
                // partials, releases the slot, writes the gate/up rows and keeps SwiGLU(gate, up) of its
                // rows; with the unit's 32 h values per entry gathered in its lanes it writes their q8_1
                // block to hq and adds one to the group's counter.
                const int ewi = cw - cwc;  // epilogue warp index (>= 0)
                int q = 0, k = 0;          // tile and unit counters of this CTA
                for (int i = blockIdx.x; i < nunits; i += ngu) {
                    const int g = i / upg, jb = i - g * upg;
                    const GroupInfo gr = giA[g];
                    if (gr.cost == 0) continue;
                    const int ku = k++;
                    const int ne = gr.e1 - gr.e0;
                    int slots[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) slots[e] = entA[gr.e0 + (e < ne ? e : ne - 1)].x;
                    const bool mine_unit = ewi >= 0 && ewi < ew && ku % ew == ewi;
                    float hv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    for (int h = 0; h < tpu; ++h) {
                        const int qq = q++, slot = qq % S;
                        const uint8_t* tile = smem + A.off_ring + static_cast<size_t>(slot) * A.stage_bytes;
                        float* part = reinterpret_cast<float*>(smem + A.off_part + static_cast<size_t>(slot) * A.part_bytes);
                        if (cw < cwc) {
                            if (!vmisc[1] &&
                                !(wait_issued(vmisc, qq) && mbar_wait_bounded(&full[slot], static_cast<uint32_t>(qq / S) & 1u))) {
                                set_err(A.err, MOE_ERR_TIMEOUT);
                                vmisc[1] = 1;
                            }
                            const bool skip = vmisc[1] != 0;
                            for (int c = cw; c < A.nch; c += cwc) {
                                if (!skip && lane < RT) chunk_part<GT>(A, smem, tile, part, ne, c, lane, loff, tabA, slots);
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&cdone[slot]);
                            }
                        } else if (mine_unit) {
                            if (!vmisc[1] &&
                                !(wait_issued(vmisc, qq) && mbar_wait_bounded(&cdone[slot], static_cast<uint32_t>(qq / S) & 1u))) {
                                set_err(A.err, MOE_ERR_TIMEOUT);
                                vmisc[1] = 1;
                            }
                            const bool skip = vmisc[1] != 0;
                            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            if (!skip && lane < RT)
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    if (e < ne) {
                                        float sv = part[e * RT + lane];
                                        for (int cc = 1; cc < A.nch; ++cc)
                                            sv = __fadd_rn(sv, part[(cc * kMaxEntriesPerPass + e) * RT + lane]);
                                        v[e] = sv;
                                    }
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&empty[slot]);  // partials read: the slot is free
                            // gate/up row of tile row `lane`
                            const int rowg = 32 * jb + h * half + (lane < half ? lane : lane - half + F);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (e >= ne) break;
                                if (!skip && lane < RT) A.out[static_cast<int64_t>(gr.e0 + e) * gst + rowg] = v[e];
                                const float uv = __shfl_down_sync(0xffffffffu, v[e], half);
                                // this tile's h for j = h*half + lane (lane < half), moved to lane h*half + lane
                                const float ht = __shfl_up_sync(0xffffffffu, swiglu_rn(v[e], uv), h * half);
                                if (lane >= h * half && lane < (h + 1) * half) hv[e] = ht;
                            }
                        }
                    }
                    if (mine_unit && !vmisc[1]) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e < ne) warp_q8_1(hv[e], L.hq + static_cast<int64_t>(gr.e0 + e) * L.nbj + jb, lane);
                        __syncwarp();
                        if (lane == 0) {
                            __threadfence();
                            atomicAdd(L.sync + g, 1);
                        }
                    }
                }
                qA = q;
            } else {
            int q = 0, k = 0;  // tile and unit counters of this CTA
            for (int i = blockIdx.x; i < nunits; i += ngu) {
                const int g = i / upg, jb = i - g * upg;
                const GroupInfo gr = giA[g];
                if (gr.cost == 0) continue;
                const int ub = k++ % S;  // unit buffer
                float* ux = ubuf + ub * 128;
                const bool single = gr.e1 - gr.e0 <= kMaxEntriesPerPass;
                for (int h = 0; h < tpu; ++h) {
                    const int qq = q++, slot = qq % S;
                    const uint8_t* tile = smem + A.off_ring + static_cast<size_t>(slot) * A.stage_bytes;
                    float* part = reinterpret_cast<float*>(smem + A.off_part + static_cast<size_t>(slot) * A.part_bytes);
                    // gate/up row of tile row `lane`
                    const int rowg = 32 * jb + h * half + (lane < half ? lane : lane - half + F);
                    for (int b0 = gr.e0; b0 < gr.e1; b0 += kMaxEntriesPerPass) {
                        const int ne = gr.e1 - b0 < kMaxEntriesPerPass ? gr.e1 - b0 : kMaxEntriesPerPass;
                        const bool lastb = b0 + kMaxEntriesPerPass >= gr.e1;
                        if (b0 != gr.e0) named_sync(1, cnt);  // the previous batch's partials are summed
                        if (!vmisc[1] &&
                            !(wait_issued(vmisc, qq) && mbar_wait_bounded(&full[slot], static_cast<uint32_t>(qq / S) & 1u))) {
                            set_err(A.err, MOE_ERR_TIMEOUT);
                            vmisc[1] = 1;
                        }
                        const bool skip = vmisc[1] != 0;
                        int slots[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) slots[e] = entA[b0 + (e < ne ? e : ne - 1)].x;
                        for (int c = cw; c < A.nch; c += ncw) {
                            if (!skip && lane < RT) chunk_part<GT>(A, smem, tile, part, ne, c, lane, loff, tabA, slots);
                            __syncwarp();
                            __threadfence_block();
                            int last = 0;
                            if (lane == 0) last = atomicAdd(&misc[64 + 8 * slot], 1) == A.nch - 1;
                            last = __shfl_sync(0xffffffffu, last, 0);
                            if (!last) continue;
                            __threadfence_block();
                            if (!skip)
                                for (int e = 0; e < ne; ++e) {
                                    float v = 0.0f;
                                    if (lane < RT) {
                                        v = part[e * RT + lane];
                                        for (int cc = 1; cc < A.nch; ++cc)
                                            v = __fadd_rn(v, part[(cc * kMaxEntriesPerPass + e) * RT + lane]);
                                        A.out[static_cast<int64_t>(b0 + e) * gst + rowg] = v;
                                    }
                                    const float uv = __shfl_down_sync(0xffffffffu, v, half);
                                    if (single && lane < half) ux[e * 32 + h * half + lane] = swiglu_rn(v, uv);
                                }
                            __syncwarp();
                            if (lane == 0) misc[64 + 8 * slot] = 0;
                            if (!lastb) continue;
                            int done = 0;
                            if (lane == 0) {
                                __threadfence_block();
                                done = atomicAdd(&misc[16 + ub], 1) == tpu - 1;
                            }
                            done = __shfl_sync(0xffffffffu, done, 0);
                            if (done) {
                                // the unit's 32 h values per entry: from the unit buffer, or (groups of more
                                // than 4 entries) from the gate/up rows written in this CTA
                                if (single) __threadfence_block();
                                else __threadfence();
                                if (!skip)
                                    for (int e = gr.e0; e < gr.e1; ++e) {
                                        float hv;
                                        if (single) {
                                            hv = ux[(e - gr.e0) * 32 + lane];
                                        } else {
                                            const float* r = A.out + static_cast<int64_t>(e) * gst + 32 * jb + lane;
                                            hv = swiglu_rn(__ldcg(r), __ldcg(r + F));
                                        }
                                        warp_q8_1(hv, L.hq + static_cast<int64_t>(e) * L.nbj + jb, lane);
                                    }
                                __syncwarp();
                                if (lane == 0) {
                                    misc[16 + ub] = 0;
                                    if (!skip) {
                                        __threadfence();
                                        atomicAdd(L.sync + g, 1);
                                    }
                                }
                            }
                            if (lane == 0) mbar_arrive(&empty[slot]);
                        }
                    }
                }
            }
            qA = q;
            }
        }
    }
    {
        // ---- down phase: this CTA's contiguous, cost-balanced run of (group, 8-row block) pairs in
        // tiles of up to RT rows, through the same ring as the gate/up tiles (numbered after them),
        // so they are prefetched into the slots the last gate/up tiles free
        const int S = A.stages, RT = D.RT, rbpgD = D.rows >> 3, rt8 = RT >> 3;
        const long long d0 = misc[10], d1 = misc[11];
        if (warp == 0) {
            if (lane == 0) {
                int issued = vmisc[0];
                long long cur = d0;
                while (cur < d1) {
                    const Tile t = next_tile(cur, d1, rbpgD, rt8);
                    const GroupInfo gr = giD[t.g];
                    if (gr.cost == 0) continue;
                    const int s = issued % S;
                    if (vmisc[1] || (issued >= S && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(issued / S - 1) & 1u))) {
                        if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                        vmisc[1] = 1;
                        break;
                    }
                    const uint32_t bytes = static_cast<uint32_t>(t.nrows) * static_cast<uint32_t>(D.row_bytes);
                    mbar_arrive_expect_tx(&full[s], bytes);
                    bulk_g2s(smem + A.off_ring + static_cast<size_t>(s) * A.stage_bytes,
                             gr.ptr + static_cast<size_t>(t.row0) * D.row_bytes, bytes, &full[s]);
                    ++issued;
                    __threadfence_block();
                    vmisc[0] = issued;
                }
            }
        } else {
            const int cw = warp - 1, ncw = (NT >> 5) - 1, ct = tid - 32, cnt = ncw * 32;
            int gB0 = 0, gB1 = -1;
            bool multi = false;
            if (d0 < d1) {
                gB0 = static_cast<int>(d0 / rbpgD);
                gB1 = static_cast<int>((d1 - 1) / rbpgD);
                for (int g = gB0; g <= gB1; ++g)
                    multi |= giD[g].cost != 0 && giD[g].e1 - giD[g].e0 > kMaxEntriesPerPass;
            }
            // two: the range spans at most two groups of at most 4 entries, staged once (slots 0-3
            // and 4-7); otherwise a group or batch change waits and restages slots 0-3
            const bool two = d0 < d1 && !multi && gB1 - gB0 <= 1;
            if (two) {
                if (ct == 0)
                    for (int g = gB0; g <= gB1; ++g)
                        if (giD[g].cost && !vmisc[1] && !wait_count(ready + g, upg)) {
                            set_err(A.err, MOE_ERR_TIMEOUT);
                            vmisc[1] = 1;
                        }
                named_sync(1, cnt);
                if (!vmisc[1]) {
                    if (giD[gB0].cost)
                        stage_entries<DT, true>(D, smem, entD, giD[gB0].e0, giD[gB0].e1 - giD[gB0].e0, 0, ct, cnt);
                    if (gB1 != gB0 && giD[gB1].cost)
                        stage_entries<DT, true>(D, smem, entD, giD[gB1].e0, giD[gB1].e1 - giD[gB1].e0,
                                                kMaxEntriesPerPass, ct, cnt);
                }
                named_sync(1, cnt);
            }
            // work items (sub-tile, chunk) are numbered across this CTA's tiles and dealt to the
            // consumer warps in turn; the last warp of a sub-tile sums its chunks
            int q = qA, wbase = 0, cur_g = -1, cur_b0 = -1;
            long long cur = d0;
            while (cur < d1) {
                const Tile t = next_tile(cur, d1, rbpgD, rt8);
                const int g = t.g;
                const GroupInfo gr = giD[g];
                if (gr.cost == 0) continue;
                const int nsb = (t.nrows + 31) >> 5, nbat = (gr.e1 - gr.e0 + kMaxEntriesPerPass - 1) / kMaxEntriesPerPass;
                const int qq = q++, slot = qq % S;
                const uint8_t* tile = smem + A.off_ring + static_cast<size_t>(slot) * A.stage_bytes;
                float* part = reinterpret_cast<float*>(smem + A.off_part + static_cast<size_t>(slot) * A.part_bytes);
                for (int b0 = gr.e0; b0 < gr.e1; b0 += kMaxEntriesPerPass) {
                    const int ne = gr.e1 - b0 < kMaxEntriesPerPass ? gr.e1 - b0 : kMaxEntriesPerPass;
                    if (!two && (g != cur_g || b0 != cur_b0)) {
                        // a new group or batch: wait for its h rows, restage once every warp is done
                        // with the previous ones
                        if (ct == 0 && g != cur_g && !vmisc[1] && !wait_count(ready + g, upg)) {
                            set_err(A.err, MOE_ERR_TIMEOUT);
                            vmisc[1] = 1;
                        }
                        named_sync(1, cnt);
                        if (!vmisc[1]) stage_entries<DT, true>(D, smem, entD, b0, ne, 0, ct, cnt);
                        named_sync(1, cnt);
                        cur_g = g;
                        cur_b0 = b0;
                    }
                    const int s0 = two && g != gB0 ? kMaxEntriesPerPass : 0;
                    const int nitems = nsb * D.nch;
                    const int w0 = wbase + ((cw - wbase) % ncw + ncw) % ncw;
                    wbase += nitems;
                    if (w0 >= wbase) continue;  // no item of this tile for this warp
                    if (!vmisc[1] &&
                        !(wait_issued(vmisc, qq) && mbar_wait_bounded(&full[slot], static_cast<uint32_t>(qq / S) & 1u))) {
                        set_err(A.err, MOE_ERR_TIMEOUT);
                        vmisc[1] = 1;
                    }
                    const bool skip = vmisc[1] != 0;
                    const int slots[4] = {s0, s0 + (ne > 1 ? 1 : 0), s0 + (ne > 2 ? 2 : ne - 1), s0 + (ne > 3 ? 3 : ne - 1)};
                    for (int w = w0; w < wbase; w += ncw) {
                        const int j = w - (wbase - nitems), sb = j / D.nch, c = j - sb * D.nch;
                        const int nr = t.nrows - sb * 32 < 32 ? t.nrows - sb * 32 : 32;
                        if (!skip && lane < nr)
                            chunk_part<DT>(D, smem, tile + static_cast<size_t>(sb) * 32 * D.row_bytes, part + sb * 32, ne, c,
                                           lane, 0, tabD, slots);
                        __syncwarp();
                        __threadfence_block();
                        int last = 0;
                        if (lane == 0) last = atomicAdd(&misc[64 + 8 * slot + sb], 1) == D.nch - 1;
                        last = __shfl_sync(0xffffffffu, last, 0);
                        if (!last) continue;
                        __threadfence_block();
                        if (!skip) reduce_write(D, part + sb * 32, entD, b0, Tile{g, t.row0 + sb * 32, nr}, ne, lane);
                        __syncwarp();
                        if (lane == 0) {
                            misc[64 + 8 * slot + sb] = 0;
                            __threadfence_block();
                            if (atomicAdd(&misc[32 + slot], 1) == nsb * nbat - 1) {
                                misc[32 + slot] = 0;
                                mbar_arrive(&empty[slot]);
                            }
                        }
                    }
                }
            }
        }
    }

    // ---- after an abort: wait (bounded) for this CTA's copies still in flight
    __syncthreads();
    if (tid == 0 && vmisc[1]) {
        const int nq = vmisc[0], S = A.stages;
        for (int qq = nq - S > 0 ? nq - S : 0; qq < nq; ++qq)
            mbar_wait_bounded(&full[qq % S], static_cast<uint32_t>(qq / S) & 1u);
    }
    // ---- exit count; the last CTA zeroes the counters for the next call
    if (tid == 0) {
        __threadfence();
        misc[2] = atomicAdd(L.sync + n, 1) == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (misc[2]) {
        __threadfence();
        for (int i = tid; i <= n; i += NT) L.sync[i] = 0;
    }
}

template <int GT, int DT>
cudaError_t launch_layer_t(const LayerArgs& args, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    LayerArgs a = args;
    a.gu.alpha = Fmt<GT>::ALPHA;
    a.dn.alpha = Fmt<DT>::ALPHA;
    cudaError_t e = cudaFuncSetAttribute(layer_kernel<GT, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(layer_kernel<GT, DT>, dim3(grid), dim3(NT), static_cast<size_t>(smem), s, pdl, a);
}

template <int GT, int DT>
cudaError_t layer_occupancy_t(int NT, int smem, int* ctas) {
    cudaError_t e = cudaFuncSetAttribute(layer_kernel<GT, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, layer_kernel<GT, DT>, NT, smem);
}

}  // namespace moe

// One translation unit per gate/up format: both supported down formats (NL4, Q8_0).
#define MOE_LAYER_TU(NAME, GT)                                                                                  \
    namespace moe {                                                                                             \
    cudaError_t launch_layer_##NAME(const LayerArgs& a, int dt, int grid, int NT, int smem, cudaStream_t s,     \
                                    bool pdl) {                                                                 \
        return dt == MOE_NL4 ? launch_layer_t<GT, MOE_NL4>(a, grid, NT, smem, s, pdl)                           \
                             : launch_layer_t<GT, MOE_Q8_0>(a, grid, NT, smem, s, pdl);                         \
    }                                                                                                           \
    cudaError_t layer_occupancy_##NAME(int dt, int NT, int smem, int* ctas) {                                   \
        return dt == MOE_NL4 ? layer_occupancy_t<GT, MOE_NL4>(NT, smem, ctas)                                   \
                             : layer_occupancy_t<GT, MOE_Q8_0>(NT, smem, ctas);                                 \
    }                                                                                                           \
    }
