// gemv.cuh - the grouped GEMV kernel behind grouped gate/up and grouped down, for sm_103a.
//
// What it computes (#2058 "Verify window: the routed experts' gate/up with the group's q8_1 rows
// in shared memory", "Why" / "What changed"; #363 "experts: smaller and fewer launches for the
// verify window's PCIe call", "What changes"): for every group g < *n_groups with expert x and
// every entry e of the group, out[o(e)][r] = sum over 32-weight blocks of the block contribution
// of row r of expert x's blob against the entry's q8_1 activation row. Each weight block is read
// from HBM once per group and applied to all of the group's entries.
//
// How (GB300 design, not the pages' kernels):
//  * Work is the flattened list of (group, 8-row block) pairs of this call, split into one
//    contiguous, balanced range per CTA of a persistent grid. A CTA walks its range in tiles of
//    up to RT rows of one expert (contiguous bytes of the blob).
//  * One thread (tid 0) streams tiles into a ring of shared-memory slots with 1-D bulk copies
//    (cp.async.bulk, TMA engine) completing on mbarriers; all threads wait with a time limit.
//  * The group's q8_1 rows (up to 4 entries at a time) are staged once per group in shared
//    memory as 16-byte halves (conflict-free 128-bit loads, padded every 8 blocks) with the
//    scale as fp32 and, for the codebook formats, the exact sum of the codes.
//  * Thread (c, q) owns 256-weight chunk c of R rows q*R..q*R+R-1 of the tile: it decodes each
//    32-weight block once and applies it to every staged entry with dp4a; its per-(row, entry)
//    partial goes to shared memory and a fixed-order sum over the chunks gives the output.
//    The order of every floating-point operation for one (row, entry) depends only on the row's
//    chunk index, so results do not depend on the grid, the tile size or the other entries.
//  * CB2/CB3 grids are stored in shared memory in "x-form" x = (g - 1) / 2 (g odd), replicated
//    per lane ([index][lane] layout: conflict-free lookups). A sign flip of g is then a bit
//    flip of x (~x = -x - 1, so 2*(~x) + 1 = -g), and sum_i s_i g_i q_i = 2 * dp4a(x ^ mask, q)
//    + sum_i q_i, with the per-block code sum taken once per staged activation block.
//  * NL4 codes are looked up in the 16-entry table held in four registers with byte permutes
//    (two 8-entry halves and a per-byte select on the code's top bit).
//  * No tensor cores: at 1-4 entries per group this is a batched GEMV, bound by HBM bandwidth
//    and by the integer decode.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

template <int TYPE>
struct Fmt;
template <>
struct Fmt<MOE_Q8_0> { static constexpr int CHUNK = 272, R = 1, MAXT = 512; static constexpr bool CB = false; };
template <>
struct Fmt<MOE_Q4B> { static constexpr int CHUNK = 160, R = 1, MAXT = 512; static constexpr bool CB = false; };
template <>
struct Fmt<MOE_NL4> { static constexpr int CHUNK = 144, R = 1, MAXT = 512; static constexpr bool CB = false; };
template <>
struct Fmt<MOE_CB2> {
    static constexpr int CHUNK = 70, R = 2, MAXT = 384, NW = 18, IDX = 0, SGN = 8, SUB = 16;
    static constexpr bool CB = true;
};
template <>
struct Fmt<MOE_CB3> {
    static constexpr int CHUNK = 102, R = 2, MAXT = 384, NW = 26, IDX = 0, SGN = 16, SUB = 24;
    static constexpr bool CB = true;
};

__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// ---------------------------------------------------------------- per-format decode

// Bytes 0..3 of the 4-bit sign nibble -> 0xFF where the bit is set (bit i -> msb of byte i by one
// multiply, then a sign-replicating byte permute).
__device__ __forceinline__ uint32_t sign_mask4(uint32_t nib) { return prmt(nib * 0x10204080u, 0u, 0xBA98u); }

// A CB chunk-row (70 or 102 bytes at an even, possibly not 4-aligned address) held as aligned
// words plus the byte-permute selector that realigns a field at logical offset L:
//   L % 4 == 0 -> prmt(raw[L/4], raw[L/4+1], selA), L % 4 == 2 -> same with selA + 0x2222.
template <int TYPE>
struct CBRow {
    uint32_t raw[Fmt<TYPE>::NW];
    uint32_t selA;
    __device__ __forceinline__ void load(const uint8_t* p) {
        const uint32_t mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p)) & 2u;
        const uint8_t* al = p - mis;
#pragma unroll
        for (int i = 0; i < Fmt<TYPE>::NW; ++i) raw[i] = ld32(al + 4 * i);
        selA = mis ? 0x5432u : 0x3210u;
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < Fmt<TYPE>::NW; ++i) raw[i] = 0;
        selA = 0x3210u;
    }
    __device__ __forceinline__ float D() const { return h2f_bits(prmt(raw[0], raw[1], selA)); }
    // word at logical offset 4*i + 2
    __device__ __forceinline__ uint32_t w2(int i) const { return prmt(raw[i], raw[i + 1], selA + 0x2222u); }
};

// Decode 32-weight sub-block j of a CB chunk-row into 8 words of x-form values with the sign
// mask applied (w = x ^ mask) and return ls = 2*sub+1. cbt: this lane's codebook replica.
template <int TYPE>
__device__ __forceinline__ int cb_decode(const CBRow<TYPE>& row, const int j, const uint8_t* cbt, uint32_t W[8]) {
    const uint32_t subw = row.w2(Fmt<TYPE>::SUB);
    const int ls = 2 * static_cast<int>((subw >> (8 * (j >> 1) + 4 * (j & 1))) & 15u) + 1;
    const uint32_t sg = row.w2(Fmt<TYPE>::SGN + j);
    if constexpr (TYPE == MOE_CB3) {
        const uint32_t i0 = row.w2(2 * j), i1 = row.w2(2 * j + 1);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const uint32_t idx = ((w < 4 ? i0 : i1) >> (8 * (w & 3))) & 0xffu;
            const uint32_t g = ld32(cbt + (idx << 7));
            W[w] = g ^ sign_mask4((sg >> (4 * w)) & 15u);
        }
    } else {
        const uint32_t iw = row.w2(j);
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
            const uint32_t idx = (iw >> (8 * gi)) & 0xffu;
            const uint2 g = *reinterpret_cast<const uint2*>(cbt + (idx << 7));
            W[2 * gi] = g.x ^ sign_mask4((sg >> (8 * gi)) & 15u);
            W[2 * gi + 1] = g.y ^ sign_mask4((sg >> (8 * gi + 4)) & 15u);
        }
    }
    return ls;
}

// Block j (32 weights) of a 16-byte-aligned Q8_0 / Q4B / NL4 chunk: 8 weight words matching the
// staged activation words, the weight scale d and (Q4B) the minimum m.
template <int TYPE>
__device__ __forceinline__ void blk_decode(const uint8_t* chunk, const int j, const uint32_t tab[4], uint32_t W[8],
                                           float& d, float& m) {
    if constexpr (TYPE == MOE_Q8_0) {
        const int L = 34 * j;  // j even: L % 4 == 0; j odd: L % 4 == 2
        const uint8_t* p = chunk + (L & ~3);
        uint32_t r[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) r[i] = ld32(p + 4 * i);
        if ((j & 1) == 0) {
            d = h2f_bits(r[0]);
#pragma unroll
            for (int k = 0; k < 8; ++k) W[k] = prmt(r[k], r[k + 1], 0x5432u);
        } else {
            d = h2f_bits(r[0] >> 16);
#pragma unroll
            for (int k = 0; k < 8; ++k) W[k] = r[k + 1];
        }
        m = 0.0f;
    } else if constexpr (TYPE == MOE_Q4B) {
        const uint8_t* p = chunk + 20 * j;
        const uint32_t dm = ld32(p);
        d = h2f_bits(dm);
        m = h2f_bits(dm >> 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t qs = ld32(p + 4 + 4 * k);
            W[k] = qs & 0x0f0f0f0fu;
            W[4 + k] = (qs >> 4) & 0x0f0f0f0fu;
        }
    } else {  // NL4: weight bytes come out in the order [0, 2, 1, 3] of each word (the staged
              // activation words are permuted the same way)
        const int L = 18 * j;
        const uint8_t* p = chunk + (L & ~3);
        uint32_t r[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) r[i] = ld32(p + 4 * i);
        uint32_t qs[4];
        if ((j & 1) == 0) {
            d = h2f_bits(r[0]);
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = prmt(r[k], r[k + 1], 0x5432u);
        } else {
            d = h2f_bits(r[0] >> 16);
#pragma unroll
            for (int k = 0; k < 4; ++k) qs[k] = r[k + 1];
        }
        m = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t Q = qs[k];
            const uint32_t sl = (Q & 0x0707u) | ((Q >> 12) & 0x7070u);          // low codes & 7
            const uint32_t sh = ((Q >> 4) & 0x0707u) | ((Q >> 16) & 0x7070u);   // high codes & 7
            const uint32_t ml = prmt(Q << 4, 0u, 0xB9A8u);                      // low codes >= 8
            const uint32_t mh = prmt(Q, 0u, 0xB9A8u);                           // high codes >= 8
            W[k] = (prmt(tab[0], tab[1], sl) & ~ml) | (prmt(tab[2], tab[3], sl) & ml);
            W[4 + k] = (prmt(tab[0], tab[1], sh) & ~mh) | (prmt(tab[2], tab[3], sh) & mh);
        }
    }
}

// ---------------------------------------------------------------- shared staging

struct Tile {
    int g, row0, nrows;
};

__device__ __forceinline__ Tile next_tile(long long& cur, long long end, int rbpg, int rt8) {
    const int g = static_cast<int>(cur / rbpg);
    const int off = static_cast<int>(cur - static_cast<long long>(g) * rbpg);
    long long n = rbpg - off < rt8 ? rbpg - off : rt8;
    if (n > end - cur) n = end - cur;
    cur += n;
    return Tile{g, off * 8, static_cast<int>(n) * 8};
}

// Group g's expert and entry range; false if the group is skipped (invalid data reported once
// by the calling thread when `report`, or simply empty).
__device__ __forceinline__ bool group_ok(const GemvArgs& a, int g, int& x, int& e0, int& e1, bool report) {
    x = a.grp_expert[g];
    e0 = a.grp_start[g];
    e1 = a.grp_start[g + 1];
    if (x < 0 || x >= a.n_experts) {
        if (report) set_err(a.err, MOE_ERR_EXPERT);
        return false;
    }
    if (e0 < 0 || e1 < e0 || e1 > a.cap_entries) {
        if (report) set_err(a.err, MOE_ERR_START);
        return false;
    }
    if (e1 == e0) return false;
    if (reinterpret_cast<uintptr_t>(a.w[x]) & 15u) {
        if (report) set_err(a.err, MOE_ERR_ALIGN);
        return false;
    }
    return true;
}

// Producer (thread 0): find the next tile of a valid group in [cur, end) and start its copy
// into ring slot `issued % stages`. Returns false when the range is exhausted.
__device__ __forceinline__ bool produce(const GemvArgs& a, uint8_t* smem, uint64_t* bars, long long& cur,
                                        long long end, int& issued) {
    const int rbpg = a.rows >> 3;
    while (cur < end) {
        const Tile t = next_tile(cur, end, rbpg, a.RT >> 3);
        int x, e0, e1;
        if (!group_ok(a, t.g, x, e0, e1, false)) continue;
        const int s = issued % a.stages;
        const uint32_t bytes = static_cast<uint32_t>(t.nrows) * static_cast<uint32_t>(a.row_bytes);
        const uint8_t* src = static_cast<const uint8_t*>(a.w[x]) + static_cast<size_t>(t.row0) * a.row_bytes;
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(smem + static_cast<size_t>(s) * a.stage_bytes, src, bytes, &bars[s]);
        ++issued;
        return true;
    }
    return false;
}

// The codebook in shared memory: CB3 256 x 32 lane replicas of 4 bytes, CB2 256 x 16 replicas of
// 8 bytes, both in x-form and both 32 KB with entry idx at offset idx*128.
template <int TYPE>
__device__ __forceinline__ void stage_codebook(const GemvArgs& a, uint8_t* smem, int tid, int NT) {
    if constexpr (Fmt<TYPE>::CB) {
        uint8_t* cb = smem + a.off_cb;
        bool even = false;
        for (int i = tid; i < 256 * 8; i += NT) {
            const int idx = i >> 3, part = i & 7;
            uint32_t v[2];
#pragma unroll
            for (int h = 0; h < (TYPE == MOE_CB2 ? 2 : 1); ++h) {
                uint32_t w = 0;
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int g = a.codebook[idx * (TYPE == MOE_CB2 ? 8 : 4) + 4 * h + bb];
                    even |= (g & 1) == 0;
                    w |= (static_cast<uint32_t>((g - 1) >> 1) & 0xffu) << (8 * bb);
                }
                v[h] = w;
            }
            uint4 u;
            if constexpr (TYPE == MOE_CB2) u = make_uint4(v[0], v[1], v[0], v[1]);
            else u = make_uint4(v[0], v[0], v[0], v[0]);
            *reinterpret_cast<uint4*>(cb + idx * 128 + part * 16) = u;
        }
        if (even) set_err(a.err, MOE_ERR_CODEBOOK);
    }
}

// Entry bookkeeping for a batch of up to 4 entries (thread 0): misc[4+s] ok, [8+s] activation
// row, [12+s] output row.
__device__ __forceinline__ void setup_entries(const GemvArgs& a, int* misc, int b0, int ne) {
    for (int s = 0; s < kMaxEntriesPerPass; ++s) {
        int ok = 0, in = 0, o = 0;
        if (s < ne) {
            const int e = b0 + s;
            in = a.ent_in ? a.ent_in[e] : e;
            o = a.ent_out ? a.ent_out[e] : e;
            ok = in >= 0 && in < a.n_act_rows && o >= 0 && o < a.out_rows;
            if (!ok) set_err(a.err, MOE_ERR_ENTRY);
        }
        misc[4 + s] = ok;
        misc[8 + s] = in;
        misc[12 + s] = o;
    }
}

template <int TYPE>
__device__ __forceinline__ void stage_act(const GemvArgs& a, uint8_t* smem, const int* misc, int ne, int tid, int NT) {
    int4* q = reinterpret_cast<int4*>(smem + a.off_actq);
    float* dx = reinterpret_cast<float*>(smem + a.off_dx);
    int* aux = reinterpret_cast<int*>(smem + a.off_aux);
    for (int i = tid; i < ne * a.nb; i += NT) {
        const int s = i / a.nb, b = i - s * a.nb, bp = b + (b >> 3);
        uint32_t w[9];
        if (misc[4 + s]) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(a.act + static_cast<int64_t>(misc[8 + s]) * a.nb + b);
#pragma unroll
            for (int k = 0; k < 9; ++k) w[k] = __ldg(src + k);
        } else {
#pragma unroll
            for (int k = 0; k < 9; ++k) w[k] = 0;
        }
        if constexpr (TYPE == MOE_NL4) {
#pragma unroll
            for (int k = 1; k < 9; ++k) w[k] = prmt(w[k], 0u, 0x3120u);
        }
        q[(s * 2 + 0) * a.nbp + bp] = make_int4(w[1], w[2], w[3], w[4]);
        q[(s * 2 + 1) * a.nbp + bp] = make_int4(w[5], w[6], w[7], w[8]);
        dx[s * a.nb + b] = h2f_bits(w[0]);
        if constexpr (Fmt<TYPE>::CB) {
            int S = 0;
#pragma unroll
            for (int k = 1; k < 9; ++k) S = dp4a(w[k], 0x01010101u, S);
            aux[s * a.nb + b] = S;
        } else if constexpr (TYPE == MOE_Q4B) {
            reinterpret_cast<float*>(aux)[s * a.nb + b] = h2f_bits(w[0] >> 16);
        }
    }
}

// ---------------------------------------------------------------- compute

template <int NE>
__device__ __forceinline__ void load_act(const GemvArgs& a, const uint8_t* smem, int b, uint32_t A[NE][8], float dx[NE],
                                         int aux[NE]) {
    const int4* q = reinterpret_cast<const int4*>(smem + a.off_actq);
    const float* dxs = reinterpret_cast<const float*>(smem + a.off_dx);
    const int* auxs = reinterpret_cast<const int*>(smem + a.off_aux);
    const int bp = b + (b >> 3);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const int4 lo = q[(e * 2 + 0) * a.nbp + bp], hi = q[(e * 2 + 1) * a.nbp + bp];
        A[e][0] = lo.x; A[e][1] = lo.y; A[e][2] = lo.z; A[e][3] = lo.w;
        A[e][4] = hi.x; A[e][5] = hi.y; A[e][6] = hi.z; A[e][7] = hi.w;
        dx[e] = dxs[e * a.nb + b];
        aux[e] = auxs[e * a.nb + b];
    }
}

// Thread (c, q): chunk c of rows q*R .. q*R+R-1 of the tile; partials to part[(c*4+e)*RT + row].
template <int TYPE, int NE>
__device__ __forceinline__ void compute_tile(const GemvArgs& a, const uint8_t* tile, const uint8_t* smem, int c, int q,
                                             int nrows, int lane, const uint32_t tab[4], float* part) {
    constexpr int R = Fmt<TYPE>::R;
    float acc[R][NE];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[r][e] = 0.0f;

    if constexpr (Fmt<TYPE>::CB) {
        CBRow<TYPE> rows[R];
        float D[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int row = q * R + r;
            if (row < nrows) rows[r].load(tile + row * a.row_bytes + c * Fmt<TYPE>::CHUNK);
            else rows[r].zero();
            D[r] = rows[r].D();
        }
        const uint8_t* cbt = smem + a.off_cb + (TYPE == MOE_CB3 ? lane * 4 : (lane & 15) * 8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t A[NE][8];
            float dx[NE];
            int sq[NE];
            load_act<NE>(a, smem, c * 8 + j, A, dx, sq);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                uint32_t W[8];
                const int ls = cb_decode<TYPE>(rows[r], j, cbt, W);
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    int d = 0;
#pragma unroll
                    for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[e][w], d);
                    const int isum = 2 * d + sq[e];
                    acc[r][e] = fmaf(static_cast<float>(ls * isum), dx[e], acc[r][e]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int e = 0; e < NE; ++e) acc[r][e] = __fmul_rn(D[r], acc[r][e]);
    } else {
        const int row = q;  // R == 1
        if (row < nrows) {
            const uint8_t* chunk = tile + row * a.row_bytes + c * Fmt<TYPE>::CHUNK;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t A[NE][8];
                float dx[NE];
                int aux[NE];
                load_act<NE>(a, smem, c * 8 + j, A, dx, aux);
                uint32_t W[8];
                float dw, mw;
                blk_decode<TYPE>(chunk, j, tab, W, dw, mw);
#pragma unroll
                for (int e = 0; e < NE; ++e) {
                    int d = 0;
#pragma unroll
                    for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[e][w], d);
                    acc[0][e] = fmaf(__fmul_rn(dw, dx[e]), static_cast<float>(d), acc[0][e]);
                    if constexpr (TYPE == MOE_Q4B) acc[0][e] = fmaf(mw, __int_as_float(aux[e]), acc[0][e]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int row = q * R + r;
        if (row < nrows) {
#pragma unroll
            for (int e = 0; e < NE; ++e) part[(c * kMaxEntriesPerPass + e) * a.RT + row] = acc[r][e];
        }
    }
}

// Fixed-order sum over the chunks, written to the entries' output rows.
__device__ __forceinline__ void reduce_write(const GemvArgs& a, const float* part, const int* misc, const Tile& t,
                                             int ne, int tid, int NT) {
    for (int i = tid; i < ne * t.nrows; i += NT) {
        const int s = i / t.nrows, row = i - s * t.nrows;
        if (!misc[4 + s]) continue;
        float v = 0.0f;
        for (int c = 0; c < a.nch; ++c) v = __fadd_rn(v, part[(c * kMaxEntriesPerPass + s) * a.RT + row]);
        a.out[static_cast<int64_t>(misc[12 + s]) * a.out_stride + t.row0 + row] = v;
    }
}

template <int TYPE>
__device__ __forceinline__ void load_table(const GemvArgs& a, uint32_t tab[4]) {
    if constexpr (TYPE == MOE_NL4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t w = 0;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) w |= (static_cast<uint32_t>(a.codebook[4 * k + bb]) & 0xffu) << (8 * bb);
            tab[k] = w;
        }
    } else {
        tab[0] = tab[1] = tab[2] = tab[3] = 0;
    }
}

template <int TYPE>
__global__ void __launch_bounds__(Fmt<TYPE>::MAXT, 1) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    int* misc = reinterpret_cast<int*>(smem + a.off_misc);
    float* part = reinterpret_cast<float*>(smem + a.off_part);

    if (tid < a.stages) mbar_init(&bars[tid], 1);
    fence_barrier_init();
    __syncthreads();

    if (!a.prefetch_before_wait) pdl_wait();
    int G = *a.n_groups;
    if (G < 0 || G > a.cap_groups) {
        if (blockIdx.x == 0 && tid == 0) set_err(a.err, MOE_ERR_NGROUPS);
        G = G < 0 ? 0 : a.cap_groups;
    }
    const int rbpg = a.rows >> 3;
    const long long total = static_cast<long long>(G) * rbpg;
    const long long rb0 = total * blockIdx.x / gridDim.x, rb1 = total * (blockIdx.x + 1) / gridDim.x;

    long long pcur = rb0;
    int issued = 0;
    if (tid == 0)
        for (int s = 0; s < a.stages; ++s)
            if (!produce(a, smem, bars, pcur, rb1, issued)) break;
    if (a.prefetch_before_wait) pdl_wait();
    pdl_trigger();
    if (rb0 == rb1) return;

    stage_codebook<TYPE>(a, smem, tid, NT);
    uint32_t tab[4];
    load_table<TYPE>(a, tab);

    const int c = tid / a.QR, q = tid - (tid / a.QR) * a.QR;
    const bool active = c < a.nch;
    long long ccur = rb0;
    int k = 0, cur_g = -1, cur_b0 = -1;
    while (ccur < rb1) {
        const Tile t = next_tile(ccur, rb1, rbpg, a.RT >> 3);
        int x, e0, e1;
        if (!group_ok(a, t.g, x, e0, e1, tid == 0)) continue;
        const int slot = k % a.stages;
        const uint32_t parity = static_cast<uint32_t>(k / a.stages) & 1u;
        const uint8_t* tile = smem + static_cast<size_t>(slot) * a.stage_bytes;
        bool waited = false;
        for (int b0 = e0; b0 < e1; b0 += kMaxEntriesPerPass) {
            const int ne = e1 - b0 < kMaxEntriesPerPass ? e1 - b0 : kMaxEntriesPerPass;
            if (t.g != cur_g || b0 != cur_b0) {
                __syncthreads();
                if (tid == 0) setup_entries(a, misc, b0, ne);
                __syncthreads();
                stage_act<TYPE>(a, smem, misc, ne, tid, NT);
                cur_g = t.g;
                cur_b0 = b0;
            }
            bool late = false;
            if (!waited) {
                late = !mbar_wait_bounded(&bars[slot], parity);
                waited = true;
            }
            if (__syncthreads_or(late)) {
                // a staged tile never arrived: report, wait (bounded) for the copies still in
                // flight into this CTA's shared memory, and leave
                if (tid == 0) {
                    set_err(a.err, MOE_ERR_TIMEOUT);
                    for (int kk = k; kk < issued; ++kk)
                        mbar_wait_bounded(&bars[kk % a.stages], static_cast<uint32_t>(kk / a.stages) & 1u);
                }
                __syncthreads();
                return;
            }
            if (active) {
                switch (ne) {
                case 1: compute_tile<TYPE, 1>(a, tile, smem, c, q, t.nrows, lane, tab, part); break;
                case 2: compute_tile<TYPE, 2>(a, tile, smem, c, q, t.nrows, lane, tab, part); break;
                case 3: compute_tile<TYPE, 3>(a, tile, smem, c, q, t.nrows, lane, tab, part); break;
                default: compute_tile<TYPE, 4>(a, tile, smem, c, q, t.nrows, lane, tab, part); break;
                }
            }
            __syncthreads();
            reduce_write(a, part, misc, t, ne, tid, NT);
        }
        __syncthreads();
        if (tid == 0) produce(a, smem, bars, pcur, rb1, issued);
        ++k;
    }
}

// Test hook: isum[r][b] of `rows` rows of one blob against one q8_1 row, by the same decode
// and dot-product code (one thread per (row, chunk), the blob read straight from global memory).
template <int TYPE>
__global__ void __launch_bounds__(256) isum_kernel(const GemvArgs a, const uint8_t* blob, int rows, int32_t* isum) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31;
    int* misc = reinterpret_cast<int*>(smem + a.off_misc);
    if (tid == 0) {
        misc[4] = 1; misc[5] = misc[6] = misc[7] = 0;
        misc[8] = 0;
    }
    __syncthreads();
    stage_codebook<TYPE>(a, smem, tid, NT);
    stage_act<TYPE>(a, smem, misc, 1, tid, NT);
    __syncthreads();
    uint32_t tab[4];
    load_table<TYPE>(a, tab);
    const int i = blockIdx.x * NT + tid;
    if (i >= rows * a.nch) return;
    const int r = i / a.nch, c = i - r * a.nch;
    const uint8_t* chunk = blob + static_cast<size_t>(r) * a.row_bytes + c * Fmt<TYPE>::CHUNK;
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        uint32_t A[1][8];
        float dx[1];
        int aux[1];
        load_act<1>(a, smem, c * 8 + j, A, dx, aux);
        uint32_t W[8];
        int v;
        if constexpr (Fmt<TYPE>::CB) {
            CBRow<TYPE> row;
            row.load(chunk);
            cb_decode<TYPE>(row, j, smem + a.off_cb + (TYPE == MOE_CB3 ? lane * 4 : (lane & 15) * 8), W);
            int d = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[0][w], d);
            v = 2 * d + aux[0];
        } else {
            float dw, mw;
            blk_decode<TYPE>(chunk, j, tab, W, dw, mw);
            int d = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[0][w], d);
            v = d;
        }
        isum[static_cast<size_t>(r) * a.nb + c * 8 + j] = v;
    }
}

// ---------------------------------------------------------------- per-format entry points

template <int TYPE>
cudaError_t launch_gemv_t(const GemvArgs& a, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(gemv_kernel<TYPE>, dim3(grid), dim3(NT), static_cast<size_t>(smem), s, pdl, a);
}

template <int TYPE>
cudaError_t gemv_occupancy_t(int NT, int smem, int* ctas) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, gemv_kernel<TYPE>, NT, smem);
}

template <int TYPE>
cudaError_t launch_isum_t(const int8_t* codebook, int K, const void* blob, int rows, const moe_q8_1* xq,
                          int32_t* isum, cudaStream_t s) {
    GemvArgs a = {};
    a.K = K;
    a.nch = K / 256;
    a.nb = K / 32;
    a.nbp = a.nb + a.nb / 8;
    a.row_bytes = static_cast<int>(a.nch * Fmt<TYPE>::CHUNK);
    a.codebook = codebook;
    a.act = xq;
    a.n_act_rows = 1;
    a.out_rows = 1;
    int off = 0;
    a.off_cb = off;
    off += Fmt<TYPE>::CB ? 32768 : 0;
    a.off_actq = off;
    off += 2 * a.nbp * 16;
    a.off_dx = off;
    off += a.nb * 4;
    a.off_aux = off;
    off += a.nb * 4;
    a.off_misc = off;
    off += 64;
    cudaError_t e = cudaFuncSetAttribute(isum_kernel<TYPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, off);
    if (e != cudaSuccess) return e;
    const int n = rows * a.nch;
    const int grid = (n + 255) / 256;
    return launch_kernel(isum_kernel<TYPE>, dim3(grid > 0 ? grid : 1), dim3(256), static_cast<size_t>(off), s, false,
                         a, static_cast<const uint8_t*>(blob), rows, isum);
}

}  // namespace moe

#define MOE_FORMAT_TU(NAME, TYPE)                                                                            \
    namespace moe {                                                                                          \
    cudaError_t launch_gemv_##NAME(const GemvArgs& a, int grid, int NT, int smem, cudaStream_t s, bool pdl) { \
        return launch_gemv_t<TYPE>(a, grid, NT, smem, s, pdl);                                               \
    }                                                                                                        \
    cudaError_t gemv_occupancy_##NAME(int NT, int smem, int* ctas) { return gemv_occupancy_t<TYPE>(NT, smem, ctas); } \
    cudaError_t launch_isum_##NAME(const int8_t* codebook, int K, const void* blob, int rows,                \
                                   const moe_q8_1* xq, int32_t* isum, cudaStream_t s) {                      \
        return launch_isum_t<TYPE>(codebook, K, blob, rows, xq, isum, s);                                    \
    }                                                                                                        \
    }
