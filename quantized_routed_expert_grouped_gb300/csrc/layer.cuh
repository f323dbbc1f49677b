// layer.cuh - the fused layer kernel: one launch runs a layer's whole hot path (routing/grouping,
// activation q8_1, grouped gate/up, SwiGLU + q8_1, grouped down) for one verify window.
//
// What it computes is the composition of the separate steps (#363 "experts: smaller and fewer
// launches for the verify window's PCIe call", "What changes"; #2058 "Verify window: the routed
// experts' gate/up with the group's q8_1 rows in shared memory", "What changed"), with the same
// arithmetic in the same order, so its outputs equal the separate kernels' bit for bit.
//
// How (GB300 design):
//  * Every CTA groups the window's top-k ids itself (one warp: a bitonic sort of (id, lane) keys
//    across the warp when T*k <= 32);
//    CTA 0 also writes the grouping and the activation q8_1 rows to global memory for inspection.
//    The expert pointer tables, like the codebooks, are read before the dependency wait.
//  * One stream of work items for the whole grid, pulled in order from a global counter: first
//    the gate/up units (one 32-value h block of one group, group-major), then the down chunks (a
//    few row tiles of one group, group-major). A CTA's first item is its own index; it fetches the
//    next index while the current item streams. So gate/up and down overlap across the grid,
//    faster CTAs take more items, and no CTA waits for a phase boundary.
//  * Each CTA has one producer warp and 15 consumer warps around a ring of shared-memory slots
//    (1-D bulk copies and full/empty mbarriers). The producer writes a descriptor per ring index
//    (kind, group, rows, entries); the consumer warps all walk the same ring indices.
//  * A gate/up unit is gate rows 32jb .. 32jb+31 and up rows F+32jb .. F+32jb+31 of one expert:
//    two ring tiles (four when rows are long) of 16 gate rows and the matching 16 up rows (two
//    bulk copies into one slot). Chunk warps (a warp per 256-weight chunk, lane = row) only compute
//    and arrive on the slot's chunk-done barrier; an epilogue warp per unit sums the chunk
//    partials, releases the slot, writes the gate/up rows and keeps SwiGLU(gate, up) (product
//    rounded on its own) in its lanes, so the unit's 32 h values per entry end up one per lane: it
//    writes their q8_1 block to hq and a flagged copy of it to the sync array (nine 8-byte pairs
//    of a word and the call's flag, so no fence is needed: a reader takes a pair once its flag is
//    the call's). Every h block is computed once, and no compute warp waits on an epilogue.
//  * The activations are staged as q8_1 by every CTA (one lane quad per block).
//  * Down chunks: the producer copies the chunk's weight tiles into free slots first, then polls
//    (bounded) the flagged copies of the group's q8_1 h rows until every pair carries the call's
//    flag, staging them into one of up to six buffers as they arrive (2-entry batches; a buffer
//    is refilled once every tile that read it has been released), then publishes the tiles. The
//    wait and the staging are one L2 round trip, and the writers issue no fence. A down tile
//    holds up to nsub 32-row sub-tiles; its (sub-tile, 256-weight chunk) work items are dealt to
//    the consumer warps in turn across tiles, and the last warp of a sub-tile sums its chunks
//    and writes the output rows.
//  * The counters and the flagged h copies live in a caller-owned int array that must be zero
//    before the first call; the last CTA to finish (a global exit counter) zeroes the counters
//    and advances the call epoch (the flag is epoch + 1), so every call starts clean and no pair
//    written by an earlier call carries the current flag.
//  * Every wait (mbarriers, the flagged h copies, the ring) has a time limit; on expiry the kernel
//    sets MOE_ERR_TIMEOUT, the producer stops, the consumers walk the published ring indices
//    without computing, the CTA waits (bounded) for its own copies in flight and still takes part
//    in the exit count.
#pragma once

#include "gemv.cuh"
#include "q8_1.cuh"
#include "route.cuh"

namespace moe {

constexpr int kDescRing = 16;  // tile descriptors in flight per CTA (ring indices)
constexpr int kUnitBufs = 4;   // gate/up units in flight per CTA (h buffers in shared memory)

// Advance a sync array's call epoch (the next call's flag is epoch + 1). The epoch never takes
// the value 2^32 - 1, whose flag would be 0, the value of a pair never written: there every pair
// any call on the array has used (word kSyncExt) is zeroed and the epoch restarts at 0, so no
// pair left from the cycle before carries a flag of the new one. One thread; the array's next
// call starts after this grid has completed.
static __device__ __noinline__ void advance_epoch(int32_t* s) {
    uint32_t e = static_cast<uint32_t>(s[kSyncEpoch]) + 1u;
    if (e == 0xFFFFFFFFu) {
        uint64_t* hx = reinterpret_cast<uint64_t*>(s + kSyncHx);
        const int64_t np = s[kSyncExt];
        for (int64_t i = 0; i < np; ++i) hx[i] = 0;
        e = 0;
    }
    s[kSyncEpoch] = static_cast<int32_t>(e);
}

// One 8-byte pair of the flagged h copy: a naturally aligned 64-bit access is single-copy
// atomic, so a reader that sees the flag sees the word written with it.
__device__ __forceinline__ void st_pair(uint64_t* p, uint32_t word, uint32_t flag) {
    const uint64_t v = (static_cast<uint64_t>(flag) << 32) | word;
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_pair(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// A block whose flagged copy was not complete at the first read: wait (bounded) until all nine
// flags equal `flag`, between reads polling the header pair alone, then stage it into `slot`.
// Out of line, since the common case finds the block complete at once (p: its header pair, the
// other pairs nb apart; the staging layout's offsets passed as they are in GemvArgs).
template <int TYPE>
static __device__ __noinline__ bool stage_flagged_wait(uint8_t* smem, int off_actq, int off_act2, int nbp, int nb,
                                                     int slot, int b, const uint64_t* p, uint32_t flag) {
    GemvArgs g;
    g.off_actq = off_actq;
    g.off_act2 = off_act2;
    g.nbp = nbp;
    g.nb = nb;
    const unsigned long long t0 = global_ns();
    for (;;) {
        for (uint32_t j = 0;; ++j) {
            __nanosleep(128);  // (at T = 1 the producers wait longest; 64 ns polled harder for nothing)
            if (static_cast<uint32_t>(ld_pair(p) >> 32) == flag) break;
            if ((j & 15u) == 15u && global_ns() - t0 > kWaitLimitNs) return false;
        }
        uint32_t w[kHxPairs];
        bool ok = true;
#pragma unroll
        for (int k = 0; k < kHxPairs; ++k) {
            const uint64_t v = ld_pair(p + k * nb);
            ok = ok && static_cast<uint32_t>(v >> 32) == flag;
            w[k] = static_cast<uint32_t>(v);
        }
        if (ok) {
            put_staged<TYPE>(g, smem, slot, b, w);
            return true;
        }
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The q8_1 h rows of entries e0 .. e0+ne-1 (ent[e].x; < 0 stages zeros) into slots slot0 ...,
// read from their flagged copies (hx: per row kHxPairs rows of nb pairs, pair k of every block
// side by side, so that one pair of consecutive blocks is one coalesced load across the warp): a
// lane reads each of its blocks until all nine flags equal `flag` (between reads it polls the
// header pair alone), then stages it. False when a block is still missing after kWaitLimitNs.
template <int TYPE>
__device__ __forceinline__ bool stage_flagged(const GemvArgs& a, uint8_t* smem, const int2* ent, const uint64_t* hx,
                                              int e0, int ne, int slot0, uint32_t flag, int lane) {
    for (int i = lane; i < ne * a.nb; i += 32) {
        const int s = i / a.nb, b = i - s * a.nb, row = ent[e0 + s].x;
        uint32_t w[kHxPairs];
        if (row >= 0) {
            const uint64_t* p = hx + static_cast<int64_t>(row) * kHxPairs * a.nb + b;
            bool ok = true;
#pragma unroll
            for (int k = 0; k < kHxPairs; ++k) {
                const uint64_t v = ld_pair(p + k * a.nb);
                ok = ok && static_cast<uint32_t>(v >> 32) == flag;
                w[k] = static_cast<uint32_t>(v);
            }
            if (!ok) {  // not there yet
                if (!stage_flagged_wait<TYPE>(smem, a.off_actq, a.off_act2, a.nbp, a.nb, slot0 + s, b, p, flag))
                    return false;
                continue;
            }
        } else {
#pragma unroll
            for (int k = 0; k < kHxPairs; ++k) w[k] = 0;
        }
        put_staged<TYPE>(a, smem, slot0 + s, b, w);
    }
    return true;
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
// writes): staged words 2j, 2j+1; lane 0 also the (d, aux) pair. qmask: the quad's lanes.
template <int TYPE>
__device__ __forceinline__ void stage_quad(const GemvArgs& a, uint8_t* smem, int slot, int b, int j, const uint32_t w[2],
                                           uint32_t hdr, int S, unsigned qmask) {
    uint32_t c0 = w[0], c1 = w[1];
    if constexpr (TYPE == MOE_NL4) {
        // staged words 2j, 2j+1 interleave code words j and 4+j (nl4_act_perm); code word i is
        // element i & 1 of quad lane i >> 1
        const uint32_t a0 = __shfl_sync(qmask, w[0], j >> 1, 4), a1 = __shfl_sync(qmask, w[1], j >> 1, 4);
        const uint32_t b0 = __shfl_sync(qmask, w[0], 2 + (j >> 1), 4), b1 = __shfl_sync(qmask, w[1], 2 + (j >> 1), 4);
        const uint32_t xa = (j & 1) ? a1 : a0, xb = (j & 1) ? b1 : b0;
        c0 = prmt(xa, xb, 0x5140u);
        c1 = prmt(xa, xb, 0x7362u);
    }
    const int bp = b + (b >> 3);
    *reinterpret_cast<uint2*>(smem + a.off_actq + ((slot * 2 + (j >> 1)) * a.nbp + bp) * 16 + (j & 1) * 8) =
        make_uint2(c0, c1);
    if (j == 0) {
        float aux = 0.0f;
        if constexpr (Fmt<TYPE>::SLOT) {
            aux = __int_as_float(S * -(2 * Fmt<TYPE>::BIAS - 1));
        } else if constexpr (Fmt<TYPE>::CB || TYPE == MOE_NL4) {
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
// (groups by ascending expert id, entries by ascending (t, slot), numbered from 0). The keys
// (id << 5 | lane; invalid ids last) are sorted across the warp by a bitonic network (15
// compare-exchange steps), so lane r holds the entry of rank r; a group starts where the id
// changes. Writes grp_expert, grp_start (G+1), *n_groups, ent_src, ent_dst (shared memory).
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
    const int nv = __popc(__ballot_sync(0xffffffffu, v >= 0));
    uint32_t key = v >= 0 ? (static_cast<uint32_t>(v) << 5) | static_cast<uint32_t>(lane) : 0xFFFFFFFFu;
#pragma unroll
    for (int kk = 2; kk <= 32; kk <<= 1)
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, key, j);
            // ascending within blocks whose kk bit is clear, descending otherwise (all ascending
            // at kk = 32); the lower lane of a pair keeps the smaller key in an ascending block
            const bool keep_min = ((lane & kk) == 0) == ((lane & j) == 0);
            key = keep_min ? min(key, other) : max(key, other);
        }
    const int ex = static_cast<int>(key >> 5), src = static_cast<int>(key & 31u);
    const int prev = __shfl_up_sync(0xffffffffu, ex, 1);
    const bool start = lane < nv && (lane == 0 || prev != ex);
    const unsigned smask = __ballot_sync(0xffffffffu, start);
    if (lane < nv) {
        rsrc[lane] = src / k;
        rdst[lane] = src;
        if (start) {
            const int grp = __popc(smask & ((1u << lane) - 1u));
            rgx[grp] = ex;
            rgs[grp] = lane;
        }
    }
    if (lane == 0) {
        rgs[__popc(smask)] = nv;
        *rng = __popc(smask);
    }
}

// One warp: group tables for both phases (weight pointers from the shared-memory cache when it
// holds them; cost 0 marks a skipped group), the entry tables and the inspection copies (CTA 0).
template <int GT, int DT>
__device__ __forceinline__ void build_tables(const LayerArgs& L, const uint8_t* const* pcA, const uint8_t* const* pcD,
                                             const int* rgx, const int* rgs, const int* rng, const int* rsrc,
                                             const int* rdst, GroupInfo* giA, GroupInfo* giD, int2* entA, int2* entD,
                                             int* misc, int lane) {
    const GemvArgs& A = L.gu;
    const GemvArgs& D = L.dn;
    const int G = *rng, ntot = rgs[G];
    const bool report = blockIdx.x == 0;
    for (int g = lane; g < G; g += 32) {
        const int x = rgx[g], e0 = rgs[g], e1 = rgs[g + 1];
        const uint8_t* pa = pcA ? pcA[x] : static_cast<const uint8_t*>(A.w[x]);
        const uint8_t* pd = pcD ? pcD[x] : static_cast<const uint8_t*>(D.w[x]);
        const bool ok = ((reinterpret_cast<uintptr_t>(pa) | reinterpret_cast<uintptr_t>(pd)) & 15u) == 0;
        if (!ok && report) set_err(A.err, MOE_ERR_ALIGN);
        giA[g] = GroupInfo{pa, x, e0, e1, ok ? 1 : 0};
        giD[g] = GroupInfo{pd, x, e0, e1, ok ? 1 : 0};
    }
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
}

// Pre-built groups of a grouped call (warp 0), checked as the separate kernels check them: the
// count clamped to [0, cap_groups] (MOE_ERR_NGROUPS); a group is skipped when its expert id is out
// of range (MOE_ERR_EXPERT), its entries do not lie in [grp_start[0], cap_entries] in order
// (MOE_ERR_START), its weight pointers are misaligned (MOE_ERR_ALIGN) or one of its entries has a
// source row outside the activation rows or a destination outside the output rows
// (MOE_ERR_ENTRY; the whole group, where the separate kernels skip the entry alone). The tables
// number entries from grp_start[0] (*ebase), like a routed call's from 0. G: n_groups as read after
// the dependency wait. Two rounds of dependent reads: grp_start[0] with the lanes' first groups,
// then every entry of the table's range at once (a lane per entry, in bounds for any index below
// cap_entries), whose rows go into the tables before the groups are checked against them.
template <int GT, int DT>
__device__ __forceinline__ void load_groups(const LayerArgs& L, int G, const uint8_t* const* pcA,
                                            const uint8_t* const* pcD, GroupInfo* giA, GroupInfo* giD, int2* entA,
                                            int2* entD, int* rng, int* ebase, int lane) {
    const GemvArgs& A = L.gu;
    const GemvArgs& D = L.dn;
    const bool report = blockIdx.x == 0;
    if (G < 0 || G > L.g_cap_groups) {
        if (report && lane == 0) set_err(A.err, MOE_ERR_NGROUPS);
        G = G < 0 ? 0 : L.g_cap_groups;
    }
    const int base = G > 0 ? L.g_start[0] : 0;
    int x0 = 0, s0 = 0, s1 = 0;  // the lane's first group (these loads do not wait for base)
    if (lane < G) {
        x0 = L.g_expert[lane];
        s0 = L.g_start[lane];
        s1 = L.g_start[lane + 1];
    }
    if (base >= 0) {
        const int elim = base + L.n < L.g_cap_entries ? base + L.n : L.g_cap_entries;
#pragma unroll 4
        for (int e = base + lane; e < elim; e += 32) {
            entA[e - base] = make_int2(L.g_src[e], e - base);
            entD[e - base] = make_int2(e - base, L.g_dst[e]);
        }
    }
    __syncwarp();
    for (int g = lane; g < G; g += 32) {
        const int x = g == lane ? x0 : L.g_expert[g], e0 = g == lane ? s0 : L.g_start[g],
                  e1 = g == lane ? s1 : L.g_start[g + 1];
        bool ok = true;
        const uint8_t* pa = nullptr;
        const uint8_t* pd = nullptr;
        if (x < 0 || x >= A.n_experts) {
            ok = false;
            if (report) set_err(A.err, MOE_ERR_EXPERT);
        } else if (base < 0 || e0 < base || e1 < e0 || e1 > L.g_cap_entries || e1 - base > L.n) {
            ok = false;
            if (report) set_err(A.err, MOE_ERR_START);
        } else if (e1 == e0) {
            ok = false;
        } else {
            pa = pcA ? pcA[x] : static_cast<const uint8_t*>(A.w[x]);
            pd = pcD ? pcD[x] : static_cast<const uint8_t*>(D.w[x]);
            if ((reinterpret_cast<uintptr_t>(pa) | reinterpret_cast<uintptr_t>(pd)) & 15u) {
                ok = false;
                if (report) set_err(A.err, MOE_ERR_ALIGN);
            } else {
                for (int e = e0 - base; e < e1 - base; ++e) {
                    const int sr = entA[e].x, ds = entD[e].y;
                    if (sr < 0 || sr >= L.T || ds < 0 || ds >= L.g_out_rows) {
                        ok = false;
                        if (report) set_err(A.err, MOE_ERR_ENTRY);
                        break;
                    }
                }
            }
        }
        giA[g] = GroupInfo{pa, x, e0 - base, e1 - base, ok ? 1 : 0};
        giD[g] = GroupInfo{pd, x, e0 - base, e1 - base, ok ? 1 : 0};
    }
    if (lane == 0) {
        *rng = G;
        *ebase = base;
    }
    __syncwarp();
}

__device__ __forceinline__ void bar_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// One warp's partial sums for one 256-weight chunk c of 32 rows at `rows` (lane = row):
// part[(c*kLayerBatch + e)*RT + lane] for the batch's ne (1 or 2) entries, staged in slots[0 .. ne-1].
template <int TYPE>
__device__ __forceinline__ void chunk_part(const GemvArgs& a, const uint8_t* smem, const uint8_t* rows, float* part, int ne,
                                           int c, int lane, uint32_t loff, const uint32_t tab[kTab],
                                           const int slots[kLayerBatch]) {
    if (ne == 1) {
        float acc[1];
        lane_chunk<TYPE, 1>(a, smem, rows, lane, c, loff, tab, slots, acc);
        part[c * kLayerBatch * a.RT + lane] = acc[0];
    } else {
        float acc[2];
        lane_chunk<TYPE, 2>(a, smem, rows, lane, c, loff, tab, slots, acc);
#pragma unroll
        for (int e = 0; e < 2; ++e) part[(c * kLayerBatch + e) * a.RT + lane] = acc[e];
    }
}

// The end of a call, once the CTA's work (if any) is done. The call used the h pairs of its L.n
// entries, the extent an epoch wrap clears. With a sync pair, the call that used the other half
// has completed (this one is past its dependency wait), so CTA 0 resets that half for the call
// after this one and records this call's extent in its own half (read when the next call advances
// this half's epoch). Otherwise an exit count: the last CTA zeroes the counters and advances the
// epoch. Every thread of the CTA calls it.
__device__ __forceinline__ void end_call(const LayerArgs& L, int* misc, int tid) {
    const int32_t ext = L.n * kHxPairs * L.nbj;
    if (L.sync_other) {
        if (blockIdx.x == 0 && tid == 0) {
            L.sync_other[kSyncExit] = 0;
            L.sync_other[kSyncWork] = 0;
            advance_epoch(L.sync_other);
            if (L.sync[kSyncExt] < ext) L.sync[kSyncExt] = ext;
        }
        return;
    }
    if (tid == 0) {
        __threadfence();
        misc[2] = atomicAdd(L.sync + kSyncExit, 1) == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (misc[2] && tid == 0) {
        __threadfence();
        L.sync[kSyncExit] = 0;
        L.sync[kSyncWork] = 0;
        if (L.sync[kSyncExt] < ext) L.sync[kSyncExt] = ext;
        advance_epoch(L.sync);
    }
}

// GIVEN: the grouping and the activation q8_1 come from the caller (moe_expert_grouped_fused)
// instead of routing ids and quantizing x (moe_expert_layer); a template parameter, so that each
// form's kernel carries only its own code.
template <int GT, int DT, bool GIVEN>
__global__ void __launch_bounds__(kMaxThreads, 1) layer_kernel(const LayerArgs L) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const GemvArgs& A = L.gu;
    const GemvArgs& D = L.dn;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NT = blockDim.x;
    const int n = L.n, F = L.F, upg = L.upg, tpu = L.tpu;
    const int SB = A.stages;  // ring slots
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + A.off_bar);
    uint64_t* empty = full + SB;
    uint64_t* dread = empty + SB;         // descriptor d passed by every consumer warp
    uint64_t* ufree = dread + kDescRing;  // unit buffer u free again (its unit's h blocks written)
    uint64_t* pub = ufree + kUnitBufs;    // descriptor d published (or the stream ended there)
    // misc: [0] ring indices published, [1] abort flag, [2] last-CTA flag, [3] the call's flag in
    // the flagged h copies, [5] no more tiles, [12] the first entry of pre-built groups,
    // [6] copies issued, [7] work items published, [8] work items taken, [16 + u] tiles done of the
    // gate/up unit in buffer u, [32 + s] sub-tiles done of slot s, [64 + 8s + b] chunks done of
    // (sub-)tile b of slot s, [128 + 8d ..] descriptor d of ring index q (d = q % kDescRing)
    int* misc = reinterpret_cast<int*>(smem + A.off_misc);
    // gate/up unit buffers: [kUnitBufs][4 entries][32] h values (the CTA's unit k uses k % kUnitBufs)
    float* ubuf = reinterpret_cast<float*>(smem + L.off_unit);
    volatile int* vmisc = misc;
    GroupInfo* giA = reinterpret_cast<GroupInfo*>(smem + A.off_grp);
    GroupInfo* giD = reinterpret_cast<GroupInfo*>(smem + D.off_grp);
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
    // expert pointer tables cached in shared memory (static data: read before the dependency wait)
    const uint8_t** pcA = L.off_ptr ? reinterpret_cast<const uint8_t**>(smem + L.off_ptr) : nullptr;
    const uint8_t** pcD = pcA ? pcA + A.n_experts : nullptr;

    // the call's inputs (routing ids, activation rows, up to NT lines of each) into L2 while the
    // grid before this one finishes: the first reads after the dependency wait then hit L2
    if constexpr (!GIVEN) {
        const uintptr_t xa = reinterpret_cast<uintptr_t>(L.x) & ~uintptr_t(127);
        const uintptr_t xe = reinterpret_cast<uintptr_t>(L.x + static_cast<int64_t>(L.T) * A.K);
        const uintptr_t ia = reinterpret_cast<uintptr_t>(L.ids) & ~uintptr_t(127);
        const uintptr_t ie = reinterpret_cast<uintptr_t>(L.ids + n);
        const uintptr_t xl = xa + static_cast<uintptr_t>(tid) * 128u;
        const uintptr_t il = ia + static_cast<uintptr_t>(NT - 1 - tid) * 128u;
        if (xl < xe) prefetch_l2(reinterpret_cast<const void*>(xl));
        if (il < ie) prefetch_l2(reinterpret_cast<const void*>(il));
    }
    if (tid < 256) misc[tid] = 0;
    if (tid == 0) {
        for (int s = 0; s < SB; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int d = 0; d < kDescRing; ++d) mbar_init(&dread[d], (NT >> 5) - 1);
        for (int u = 0; u < kUnitBufs; ++u) mbar_init(&ufree[u], 1);
        for (int d = 0; d < kDescRing; ++d) mbar_init(&pub[d], 1);
    }
    fence_barrier_init();
    // static data before the dependency wait: codebook replicas, NL4 tables, pointer tables
    if (warp > 0) stage_codebook<GT>(A, smem, tid - 32, NT - 32);
    if (pcA)
        for (int x = tid; x < A.n_experts; x += NT) {
            pcA[x] = static_cast<const uint8_t*>(A.w[x]);
            pcD[x] = static_cast<const uint8_t*>(D.w[x]);
        }
    uint32_t tabA[kTab], tabD[kTab];
    load_table<GT>(A, tabA);
    load_table<DT>(D, tabD);
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    // pre-built groups and none in this call (the same value for every thread): nothing to stage
    // or stream, only the end-of-call words
    int given_ng = 0;  // pre-built groups: n_groups, read once here (also by load_groups)
    if constexpr (GIVEN) {
        given_ng = __ldcg(L.g_ng);
        if (given_ng == 0) {
            end_call(L, misc, tid);
            return;
        }
    }
    uint64_t* hx = reinterpret_cast<uint64_t*>(L.sync + kSyncHx);

    // ---- routing/grouping and tables: one warp when n <= 32, else the whole CTA routes and
    // warp 0 builds the tables
    if (!GIVEN && n > 32) {
        route_cta(L.ids, n, L.k, A.n_experts, 0, sid, sfirst, scount, rgx, rgs, rng, rsrc, rdst, A.err,
                  blockIdx.x == 0);
        __syncthreads();
    }
    int early = 0;  // ring indices of the CTA's first item copied before the tables (warp 0, lane 0)
    // this call's flag in the flagged h copies (the pairs of every earlier call carry a smaller
    // one): read once per CTA, handed to the consumer warps with the tables
    uint32_t flag = 0;
    if (warp == 0) {
        if (lane == 0) flag = 1u + static_cast<uint32_t>(__ldcg(L.sync + kSyncEpoch));
        if (!GIVEN && n <= 32)
            route_warp(L.ids, n, L.k, A.n_experts, rgx, rgs, rng, rsrc, rdst, A.err, blockIdx.x == 0, lane);
        __syncwarp();
        // The CTA's first work item is its own index. When that is a gate/up unit, its first tile
        // needs only the group's expert id, so it is copied now, before the tables are built; the
        // producer publishes it without copying again.
        if (!GIVEN && lane == 0 && static_cast<int>(blockIdx.x) < *rng * upg) {
            const int g = static_cast<int>(blockIdx.x) / upg, jb = static_cast<int>(blockIdx.x) - g * upg;
            const int x = rgx[g];
            const uint8_t* pa = pcA ? pcA[x] : static_cast<const uint8_t*>(A.w[x]);
            const uint8_t* pd = pcD ? pcD[x] : static_cast<const uint8_t*>(D.w[x]);
            if (((reinterpret_cast<uintptr_t>(pa) | reinterpret_cast<uintptr_t>(pd)) & 15u) == 0) {  // as build_tables
                const uint64_t pol = l2_evict_first();
                const int half = A.RT >> 1;
                const uint32_t hb = static_cast<uint32_t>(half) * static_cast<uint32_t>(A.row_bytes);
                // only the first tile: with every CTA copying at once, a smaller first burst lands
                // sooner, and the producer loop copies the unit's other tile a little later
                early = 1;
                for (int h = 0; h < early; ++h) {
                    const size_t rg = static_cast<size_t>(32 * jb + h * half);
                    uint8_t* dst = smem + A.off_ring + static_cast<size_t>(h) * A.stage_bytes;
                    mbar_arrive_expect_tx(&full[h], 2 * hb);
                    bulk_g2s_hint(dst, pa + rg * A.row_bytes, hb, &full[h], pol);
                    bulk_g2s_hint(dst + hb, pa + (rg + F) * A.row_bytes, hb, &full[h], pol);
                }
                vmisc[6] = early;
            }
        }
        if constexpr (GIVEN) load_groups<GT, DT>(L, given_ng, pcA, pcD, giA, giD, entA, entD, rng, &misc[12], lane);
        else build_tables<GT, DT>(L, pcA, pcD, rgx, rgs, rng, rsrc, rdst, giA, giD, entA, entD, misc, lane);
        if (lane == 0) misc[3] = static_cast<int>(flag);
        flag = __shfl_sync(0xffffffffu, flag, 0);
        __threadfence_block();
        bar_arrive(3, NT);  // tables ready
    } else {
        // meanwhile the consumer warps quantize the activations (independent of the grouping)
        const int ct = tid - 32, cnt = NT - 32;
        // ---- activations: x -> q8_1 of all T tokens, staged in slot t; one lane quad per block
        // (pre-built groups: the caller's q8_1 rows, staged as they are)
        if constexpr (GIVEN) {
            for (int i = ct; i < L.T * A.nb; i += cnt) {
                const int r = i / A.nb;
                stage_block<GT>(A, smem, r, r, i - r * A.nb);
            }
        } else {
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
                    stage_quad<GT>(A, smem, t, b, j, w, hdr, Ssum, qmask);
                    if (blockIdx.x == 0 && L.o_xq) put_quad(L.o_xq + i, j, w, hdr);
                }
            }
        }
        named_sync(3, NT);  // with warp 0's arrival: tables ready, activations staged
        flag = static_cast<uint32_t>(vmisc[3]);
    }
    const int G = *rng;
    // global index of the tables' entry 0 (pre-built groups: grp_start[0]), for the scratch rows
    const int ebase = GIVEN ? misc[12] : 0;
    // ---- one stream of work items for the whole grid, taken in order from a global counter:
    // gate/up units (group-major), then down chunks of dchunk tiles of one group (group-major).
    // Each CTA's producer warp pulls items and streams their tiles through the ring, publishing a
    // descriptor per ring index (reused kDescRing indices later, once every consumer warp has
    // passed it). The ring indices' work items (a gate/up tile's 256-weight chunks, a down tile's
    // (sub-tile, chunk) pairs) are numbered in ring order and taken one at a time by whichever
    // consumer warp is free (a shared counter), so a warp busy with an epilogue holds up nobody.
    // The producer warp also stages each down group's q8_1 h rows (4-entry batches) into one of
    // two buffers: a buffer is refilled once every tile that read it has been released.
    const int S = A.stages, RT = A.RT, half = RT >> 1, RTD = D.RT;
    const SmallDiv divS(S);
    const int tpg = (D.rows + RTD - 1) / RTD;
    int dchunk = (2 * G * tpg) / (5 * static_cast<int>(gridDim.x));  // about 2.5 down items per CTA
    dchunk = dchunk < 1 ? 1 : dchunk > 3 ? 3 : dchunk;
    const int nunits = G * upg, cpg = (tpg + dchunk - 1) / dchunk;
    const int nitems = nunits + G * cpg;
    int* work = L.sync + kSyncWork;  // global item counter
    // per ring index q (d = q % kDescRing): [8d] kind (0 gate/up, 1 down), [8d+1] group,
    // [8d+2] jb or first row, [8d+3] h or rows, [8d+4] first entry, [8d+5] entries (<= 4),
    // [8d+6] gate/up: the CTA's unit number, down: first staging slot, [8d+7] first work item
    int* desc = misc + 128;

    if (warp == 0) {
        // lane 0 claims slots, issues the copies and publishes the ring indices; the whole warp
        // stages h rows
        int issued = 0;                          // ring indices published (lane 0)
        int nwork = 0;                           // work items published (lane 0)
        int ku = 0;                              // gate/up units (4-entry batches) issued (lane 0)
        int st_g = -1, st_b0 = -1, st_n = 0;     // staged group and batch, stagings so far
        const int nbuf = D.act_cap / kLayerBatch;  // h buffers, used in turn
        int st_buf = nbuf - 1;                   // buffer of the last staging
        // first ring index of the last, second-last, ... staging (lane 0; kMaxHBufs - 1 of them)
        int st_p0 = 0, st_p1 = 0, st_p2 = 0, st_p3 = 0, st_p4 = 0;
        static_assert(kMaxHBufs == 6, "the staging history holds kMaxHBufs - 1 indices");
        bool stop = false;
        // ring slot j % S free for index j: the tile S indices earlier released (lane 0)
        auto slot_free = [&](int j) -> bool {
            if (vmisc[1]) return false;
            const int jq = divS.div(j), js = j - jq * S;
            if (j >= S && !mbar_wait_bounded(&empty[js], static_cast<uint32_t>(jq - 1) & 1u)) {
                set_err(A.err, MOE_ERR_TIMEOUT);
                vmisc[1] = 1;
                return false;
            }
            return true;
        };
        // descriptor of ring index `issued` (once every consumer warp has passed the one kDescRing
        // indices earlier), then the index and its work items are published (lane 0)
        auto publish = [&](int kind, int g, int a0, int a1, int e0, int ne, int a6, int items) -> bool {
            const int d = issued % kDescRing;
            if (issued >= kDescRing && !mbar_wait_bounded(&dread[d], static_cast<uint32_t>(issued / kDescRing - 1) & 1u)) {
                if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                vmisc[1] = 1;
                return false;
            }
            int* dd = desc + 8 * d;
            dd[0] = kind;
            dd[1] = g;
            dd[2] = a0;
            dd[3] = a1;
            dd[4] = e0;
            dd[5] = ne;
            dd[6] = a6;
            dd[7] = nwork;
            ++issued;
            nwork += items;
            // (mbarrier.arrive releases at CTA scope, the consumers' waits acquire: the descriptor
            // and the counts are ordered before the arrival without a fence, which would also wait
            // for the work counter's atomic still in flight)
            vmisc[0] = issued;
            vmisc[7] = nwork;
            mbar_arrive(&pub[d]);
            return true;
        };
        const uint64_t pol = l2_evict_first();  // the weights are read once per call
        // copy of ring index j's tile into its slot; vmisc[6]: copies issued (lane 0)
        auto copy_tile = [&](int j, const uint8_t* src0, uint32_t b0, const uint8_t* src1, uint32_t b1) {
            const int js = divS.mod(j);
            uint8_t* dst = smem + A.off_ring + static_cast<size_t>(js) * A.stage_bytes;
            mbar_arrive_expect_tx(&full[js], b0 + b1);
            bulk_g2s_hint(dst, src0, b0, &full[js], pol);
            if (b1) bulk_g2s_hint(dst + b0, src1, b1, &full[js], pol);
            vmisc[6] = j + 1;
        };
        const uint32_t hb = static_cast<uint32_t>(half) * static_cast<uint32_t>(A.row_bytes);
        // the first item of CTA b is item b; later ones come from the counter, whose next value is
        // fetched while the current item streams
        // (the counter's value is consumed only at the loop increment, so the atomic's round trip
        // overlaps the item's copies instead of stalling lane 0 before them; with pre-built groups
        // and no item past the first round, as in a small second call, nothing is claimed: 0.26 us
        // less per such call, where the routed form's window lost 0.3 % to the same test)
        int nx = 0;
        const bool claim = !GIVEN || nitems > static_cast<int>(gridDim.x);
        for (int i = blockIdx.x; !stop && i < nitems; i = static_cast<int>(gridDim.x) + __shfl_sync(0xffffffffu, nx, 0)) {
            if (lane == 0) nx = claim ? atomicAdd(work, 1) : nitems;
            if (i < nunits) {
                const int g = i / upg, jb = i - g * upg;
                const GroupInfo gr = giA[g];
                if (gr.cost == 0) continue;
                if (lane == 0)
                    for (int b0 = gr.e0; b0 < gr.e1 && !stop; b0 += kLayerBatch) {
                        const int ne = gr.e1 - b0 < kLayerBatch ? gr.e1 - b0 : kLayerBatch;
                        // unit buffer ku % kUnitBufs free: the unit kUnitBufs earlier has written its h
                        // blocks
                        if (vmisc[1] || (ku >= kUnitBufs &&
                                         !mbar_wait_bounded(&ufree[ku % kUnitBufs],
                                                            static_cast<uint32_t>(ku / kUnitBufs - 1) & 1u))) {
                            if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                            vmisc[1] = 1;
                            stop = true;
                            break;
                        }
                        for (int h = 0; h < tpu; ++h) {
                            const bool pre = issued < early;  // copied before the tables (first item)
                            if (!pre && !slot_free(issued)) {
                                stop = true;
                                break;
                            }
                            const size_t rg = static_cast<size_t>(32 * jb + h * half);
                            if (!pre) copy_tile(issued, gr.ptr + rg * A.row_bytes, hb, gr.ptr + (rg + F) * A.row_bytes, hb);
                            if (!publish(0, g, jb, h, b0, ne, ku, A.nch)) {
                                stop = true;
                                break;
                            }
                        }
                        ++ku;
                    }
                stop = __shfl_sync(0xffffffffu, stop, 0);
            } else {
                const int d = i - nunits, g = d / cpg, c = d - g * cpg;
                const GroupInfo gr = giD[g];
                if (gr.cost == 0) continue;
                const int t0 = c * dchunk, t1 = t0 + dchunk < tpg ? t0 + dchunk : tpg;
                auto tile_src = [&](int t, uint32_t& bytes) {
                    const int row0 = t * RTD, nrows = D.rows - row0 < RTD ? D.rows - row0 : RTD;
                    bytes = static_cast<uint32_t>(nrows) * static_cast<uint32_t>(D.row_bytes);
                    return gr.ptr + static_cast<size_t>(row0) * D.row_bytes;
                };
                for (int b0 = gr.e0; b0 < gr.e1 && !stop; b0 += kLayerBatch) {
                    const int ne = gr.e1 - b0 < kLayerBatch ? gr.e1 - b0 : kLayerBatch;
                    int pre = 0;  // tiles of this batch copied ahead of the h wait (lane 0)
                    if (g != st_g || b0 != st_b0) {
                        int ok = 1;
                        if (lane == 0) {
                            // the weights do not depend on h: copy up to S tiles into free slots first
                            for (int t = t0; t < t1 && pre < S && ok; ++t, ++pre) {
                                ok = slot_free(issued + pre);
                                uint32_t bytes;
                                const uint8_t* src = tile_src(t, bytes);
                                if (ok) copy_tile(issued + pre, src, bytes, nullptr, 0);
                            }
                            // the next buffer free (from staging nbuf on): every ring index before
                            // the first one of staging st_n - nbuf + 1 released (indices before
                            // issued - S are, as their slots were claimed again)
                            if (st_n >= nbuf) {
                                const int lim = nbuf == 2 ? st_p0 : nbuf == 3 ? st_p1 : nbuf == 4 ? st_p2 : nbuf == 5 ? st_p3 : st_p4;
                                for (int j = issued - S > 0 ? issued - S : 0; ok && j < lim; ++j)
                                    ok = mbar_wait_bounded(&empty[divS.mod(j)], static_cast<uint32_t>(divS.div(j)) & 1u);
                            }
                            st_p4 = st_p3;
                            st_p3 = st_p2;
                            st_p2 = st_p1;
                            st_p1 = st_p0;
                            st_p0 = issued;
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        // the batch's h rows, each block staged as soon as its flagged copy is
                        // complete (every unit of the group writes one block per entry)
                        // (the test hook waits for a flag that no call writes)
                        const uint32_t want = L.test_expire ? flag ^ 0x80000000u : flag;
                        ok = __all_sync(0xffffffffu, ok && !vmisc[1] &&
                                                         stage_flagged<DT>(D, smem, entD, hx, b0, ne,
                                                                           kLayerBatch * (st_buf + 1 == nbuf ? 0 : st_buf + 1),
                                                                           want, lane));
                        if (!ok) {
                            if (lane == 0) {
                                if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                                vmisc[1] = 1;
                            }
                            stop = true;
                            break;
                        }
                        __syncwarp();  // every lane's staged blocks before lane 0 publishes
                        st_g = g;
                        st_b0 = b0;
                        ++st_n;
                        st_buf = st_buf + 1 == nbuf ? 0 : st_buf + 1;
                    }
                    const int s0 = kLayerBatch * st_buf;
                    if (lane == 0)
                        for (int t = t0; t < t1; ++t) {
                            if (t - t0 >= pre) {
                                if (!slot_free(issued)) {
                                    stop = true;
                                    break;
                                }
                                uint32_t bytes;
                                const uint8_t* src = tile_src(t, bytes);
                                copy_tile(issued, src, bytes, nullptr, 0);
                            }
                            const int row0 = t * RTD, nrows = D.rows - row0 < RTD ? D.rows - row0 : RTD;
                            if (!publish(1, g, row0, nrows, b0, ne, s0, ((nrows + 31) >> 5) * D.nch)) {
                                stop = true;
                                break;
                            }
                        }
                    stop = __shfl_sync(0xffffffffu, stop, 0);
                }
            }
        }
        if (lane == 0) {
            // no more tiles: the stream ends at ring index vmisc[0]; the consumers waiting for that
            // index are woken by an arrival without a descriptor, made (like a publish) once every
            // consumer warp has passed the index kDescRing earlier
            vmisc[5] = 1;
            const int d = issued % kDescRing;
            if (!vmisc[1] && issued >= kDescRing &&
                !mbar_wait_bounded(&dread[d], static_cast<uint32_t>(issued / kDescRing - 1) & 1u)) {
                set_err(A.err, MOE_ERR_TIMEOUT);
                vmisc[1] = 1;
            }
            mbar_arrive(&pub[d]);  // releases vmisc[5] with it
        }
    } else {
        const uint32_t loff = GT == MOE_CB3 ? lane * 4u : (lane & 15u) * 8u;
        const SmallDiv divN(D.nch);
        const int64_t gst = A.out_stride;
        // the ring index whose work items are [qb, qb + qn), its descriptor (qn < 0: not read yet)
        int q = 0, qb = 0, qn = -1;
        int kind = 0, g = 0, a0 = 0, a1 = 0, e0 = 0, ne = 0, a6 = 0;
        for (;;) {
            int it = 0;
            if (lane == 0) it = atomicAdd(&misc[8], 1);
            it = __shfl_sync(0xffffffffu, it, 0);
            // wait until item `it` is published or the stream ends, passing (and releasing the
            // descriptors of) the ring indices that end at or before it; a wait for a ring index is
            // a blocking mbarrier wait
            bool have = false;
            for (;;) {
                if (qn < 0) {
                    if (!mbar_wait_bounded(&pub[q % kDescRing], static_cast<uint32_t>(q / kDescRing) & 1u)) {
                        if (!vmisc[1]) set_err(A.err, MOE_ERR_TIMEOUT);
                        vmisc[1] = 1;
                        break;
                    }
                    if (vmisc[0] <= q) break;  // the end-of-stream arrival
                    const int* dd = desc + 8 * (q % kDescRing);
                    kind = dd[0];
                    g = dd[1];
                    a0 = dd[2];
                    a1 = dd[3];
                    e0 = dd[4];
                    ne = dd[5];
                    a6 = dd[6];
                    qb = dd[7];
                    qn = kind == 0 ? A.nch : ((a1 + 31) >> 5) * D.nch;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dread[q % kDescRing]);
                }
                if (it < qb + qn) {
                    have = true;
                    break;
                }
                ++q;
                qn = -1;
            }
            if (!have) break;
            const int qs = divS.div(q), slot = q - qs * S, j = it - qb;
            const uint8_t* tile = smem + A.off_ring + static_cast<size_t>(slot) * A.stage_bytes;
            float* part = reinterpret_cast<float*>(smem + A.off_part + static_cast<size_t>(slot) * A.part_bytes);
            if (!vmisc[1] && !mbar_wait_bounded(&full[slot], static_cast<uint32_t>(qs) & 1u)) {
                set_err(A.err, MOE_ERR_TIMEOUT);
                vmisc[1] = 1;
            }
            if (vmisc[1]) break;  // after an abort nothing more is computed (no barrier waits on this warp)
            if (kind == 0) {
                // ---- chunk c = j of gate/up tile h = a1 of unit (g, jb = a0), entries e0 .. e0+ne-1
                const int jb = a0, h = a1, c = j, u = a6 % kUnitBufs;
                const int slots[kLayerBatch] = {entA[e0].x, entA[e0 + (ne > 1 ? 1 : 0)].x};
                if (lane < RT) chunk_part<GT>(A, smem, tile, part, ne, c, lane, loff, tabA, slots);
                __syncwarp();
                __threadfence_block();
                int last = 0;
                if (lane == 0) last = atomicAdd(&misc[64 + 8 * slot], 1) == A.nch - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (!last) continue;
                // the tile's last chunk: sum the partials (fixed chunk order), release the slot, write
                // the gate/up rows and put SwiGLU(gate, up) (product rounded on its own) in the unit
                // buffer
                __threadfence_block();
                float v[kLayerBatch] = {0.0f, 0.0f};
                if (lane < RT)
#pragma unroll
                    for (int e = 0; e < kLayerBatch; ++e)
                        if (e < ne) {
                            float sv = part[e * RT + lane];
                            for (int cc = 1; cc < A.nch; ++cc) sv = __fadd_rn(sv, part[(cc * kLayerBatch + e) * RT + lane]);
                            v[e] = sv;
                        }
                __syncwarp();
                if (lane == 0) {
                    misc[64 + 8 * slot] = 0;
                    mbar_arrive(&empty[slot]);  // partials read: the slot is free
                }
                const int rowg = 32 * jb + h * half + (lane < half ? lane : lane - half + F);
                float* ub = ubuf + u * (kLayerBatch * 32);
#pragma unroll
                for (int e = 0; e < kLayerBatch; ++e) {
                    if (e >= ne) break;
                    if (lane < RT) A.out[static_cast<int64_t>(ebase + e0 + e) * gst + rowg] = v[e];
                    const float uv = __shfl_down_sync(0xffffffffu, v[e], half);
                    if (lane < half) ub[e * 32 + h * half + lane] = swiglu_rn(v[e], uv);
                }
                __syncwarp();
                __threadfence_block();
                // the unit's last tile: q8_1 of its h blocks (one value per lane) to hq and to the
                // flagged copy (pair 0 the header, pair 1 + w code word w = lanes 4w .. 4w+3), the
                // unit buffer free again
                int done = 0;
                if (lane == 0) done = atomicAdd(&misc[16 + u], 1) == tpu - 1;
                done = __shfl_sync(0xffffffffu, done, 0);
                if (!done) continue;
                __threadfence_block();
                for (int e = 0; e < ne; ++e) {
                    uint32_t hdr;
                    int Ssum;
                    const int qv = warp_q8_1_code(ub[e * 32 + lane], hdr, Ssum);
                    moe_q8_1* dst = L.hq + static_cast<int64_t>(ebase + e0 + e) * L.nbj + jb;
                    dst->q[lane] = static_cast<int8_t>(qv);
                    if (lane == 0) *reinterpret_cast<uint32_t*>(dst) = hdr;
                    uint32_t cw = (static_cast<uint32_t>(qv) & 0xFFu) << (8 * (lane & 3));
                    cw |= __shfl_xor_sync(0xffffffffu, cw, 1);
                    cw |= __shfl_xor_sync(0xffffffffu, cw, 2);
                    cw = __shfl_sync(0xffffffffu, cw, lane >= 1 && lane < kHxPairs ? 4 * (lane - 1) : 0);
                    if (lane < kHxPairs)
                        st_pair(hx + (static_cast<int64_t>(e0 + e) * kHxPairs + lane) * L.nbj + jb, lane == 0 ? hdr : cw, flag);
                }
                __syncwarp();
                if (lane == 0) {
                    misc[16 + u] = 0;
                    mbar_arrive(&ufree[u]);
                }
            } else {
                // ---- (sub-tile, chunk) item j of down tile rows a0 .. a0+a1-1 of group g for entries
                // e0 .. e0+ne-1, whose h rows the producer staged in slots a6 .. a6+ne-1
                const int row0 = a0, nrows = a1, s0 = a6;
                const int nsb = (nrows + 31) >> 5, sb = divN.div(j), c = j - sb * D.nch;
                const int nr = nrows - sb * 32 < 32 ? nrows - sb * 32 : 32;
                const int slots[kLayerBatch] = {s0, s0 + (ne > 1 ? 1 : 0)};
                if (lane < nr)
                    chunk_part<DT>(D, smem, tile + static_cast<size_t>(sb) * 32 * D.row_bytes, part + sb * 32, ne, c, lane, 0,
                                   tabD, slots);
                __syncwarp();
                __threadfence_block();
                int last = 0;
                if (lane == 0) last = atomicAdd(&misc[64 + 8 * slot + sb], 1) == D.nch - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (!last) continue;
                __threadfence_block();
                reduce_write<kLayerBatch>(D, part + sb * 32, entD, e0, Tile{g, row0 + sb * 32, nr}, ne, lane);
                __syncwarp();
                if (lane == 0) {
                    misc[64 + 8 * slot + sb] = 0;
                    __threadfence_block();
                    if (atomicAdd(&misc[32 + slot], 1) == nsb - 1) {
                        misc[32 + slot] = 0;
                        mbar_arrive(&empty[slot]);
                    }
                }
            }
        }
    }

    // ---- after an abort: wait (bounded) for this CTA's copies still in flight
    __syncthreads();
    if (tid == 0 && vmisc[1]) {
        const int nq = vmisc[6], S = A.stages;  // copies issued (published or not)
        for (int qq = nq - S > 0 ? nq - S : 0; qq < nq; ++qq)
            mbar_wait_bounded(&full[qq % S], static_cast<uint32_t>(qq / S) & 1u);
    }
    end_call(L, misc, tid);
}

template <int GT, int DT, bool GIVEN>
cudaError_t launch_layer_g(const LayerArgs& args, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    LayerArgs a = args;
    a.gu.alpha = Fmt<GT>::ALPHA;
    a.dn.alpha = Fmt<DT>::ALPHA;
    cudaError_t e =
        cudaFuncSetAttribute(layer_kernel<GT, DT, GIVEN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(layer_kernel<GT, DT, GIVEN>, dim3(grid), dim3(NT), static_cast<size_t>(smem), s, pdl, a);
}

template <int GT, int DT>
cudaError_t launch_layer_t(const LayerArgs& args, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    return args.given ? launch_layer_g<GT, DT, true>(args, grid, NT, smem, s, pdl)
                      : launch_layer_g<GT, DT, false>(args, grid, NT, smem, s, pdl);
}

template <int GT, int DT>
cudaError_t layer_occupancy_t(int NT, int smem, int* ctas) {
    cudaError_t e =
        cudaFuncSetAttribute(layer_kernel<GT, DT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, layer_kernel<GT, DT, false>, NT, smem);
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
