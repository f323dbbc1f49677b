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
//  * Persistent grid. The call's work is the list of (group, 8-row block) pairs; each CTA takes
//    one contiguous range of it, balanced by cost (a row of a group with n entries costs
//    alpha + n, alpha being the decode's share), computed from the device-side group arrays.
//  * Warp specialisation. Warp 0 streams tiles (up to 32 rows of one expert: contiguous bytes of
//    its blob) into a ring of shared-memory slots with 1-D bulk copies (cp.async.bulk, TMA
//    engine); a slot's "full" mbarrier completes on the copy's byte count and its "empty"
//    mbarrier when its consumers have released it. Every wait has a time limit.
//  * The q8_1 rows of the (at most two) groups of a CTA's range are staged once in shared memory
//    as 16-byte halves with (scale, aux) pairs as float2; all lanes of a warp read the same
//    block at the same time (broadcast loads).
//  * Consumer warps form warp-sets; a set owns one tile at a time (lane = row) and its warps
//    split the rows' 256-weight chunks. A lane decodes each 32-weight block of its row's chunk
//    once and applies it to every staged entry with dp4a; the chunk partials go to shared memory
//    and the set's last warp to finish (shared atomic counter after a fence) sums them in chunk
//    order: no barrier between warps. The order of every floating-point operation for one
//    (row, entry) depends only on the row's chunks, so results do not depend on the grid, the
//    tile size or the other entries.
//  * CB2/CB3 grids are held in shared memory (at offset 0) in "x-form" x = (g - 1) / 2 (g odd),
//    replicated per lane ([index][lane]: conflict-free lookups). A sign flip of g is a bit flip
//    of x (2*(~x) + 1 = -g), so sum_i s_i g_i q_i = 2 * dp4a(x ^ mask, q) + sum_i q_i; the
//    per-block code sum is taken once when the activation row is staged. A sign nibble becomes a
//    byte mask by one 32x32->64 multiply (bits to byte msbs) and one sign-replicating permute.
//  * NL4 codes are looked up in the 16-entry table held in four registers with byte permutes
//    taking the codes' nibbles as selectors in place (two 8-entry halves and a per-byte select
//    on the code's top bit, 11 instructions per 8 weights); the staged activation words are
//    permuted once to the resulting nibble order.
//  * No tensor cores: at 1-4 entries per group this is a batched GEMV, bound by HBM bandwidth
//    and by the integer decode.
#pragma once

#include <cuda_fp16.h>

#include <climits>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace moe {

// CHUNK: bytes of one 256-weight chunk (for the slot layouts: its codes; the 8-byte scale
// records follow all of a row's codes). CB: native codebook format (grid staged in shared
// memory). SLOT: transcoded slot layout (BIAS: code bias). ALPHA: decode cost of a row relative to
// one entry's dot products (work balancing). DEC, DOT: warp-instructions per 32-row x 256-weight
// chunk for the decode and per entry for the dot products (measured on the chunk loop alone; a
// cost model for splitting work between phases).
template <int TYPE>
struct Fmt;
template <>
struct Fmt<MOE_Q8_0> {
    static constexpr int CHUNK = 272, ALPHA = 1, DEC = 120, DOT = 148;
    static constexpr bool CB = false, SLOT = false;
};
template <>
struct Fmt<MOE_Q4B> {
    static constexpr int CHUNK = 160, ALPHA = 2, DEC = 200, DOT = 160;
    static constexpr bool CB = false, SLOT = false;
};
template <>
struct Fmt<MOE_NL4> {
    static constexpr int CHUNK = 144, ALPHA = 5, DEC = 574, DOT = 127;
    static constexpr bool CB = false, SLOT = false;
};
template <>
struct Fmt<MOE_CB2> {
    static constexpr int CHUNK = 70, ALPHA = 4, NW = 18, SGN = 8, SUB = 16, DEC = 480, DOT = 150;
    static constexpr bool CB = true, SLOT = false;
};
template <>
struct Fmt<MOE_CB3> {
    static constexpr int CHUNK = 102, ALPHA = 5, NW = 26, SGN = 16, SUB = 24, DEC = 550, DOT = 150;
    static constexpr bool CB = true, SLOT = false;
};
template <>
struct Fmt<MOE_CB3X> {
    static constexpr int CHUNK = 128, ALPHA = 1, BIAS = 8, DEC = 197, DOT = 148;
    static constexpr bool CB = false, SLOT = true;
};
template <>
struct Fmt<MOE_CB2X> {
    static constexpr int CHUNK = 64, ALPHA = 1, BIAS = 2, DEC = 180, DOT = 148;
    static constexpr bool CB = false, SLOT = true;
};

// NL4 table registers: words 0-3 the 16-entry table, words 4-7 the two 8-entry half-tables of the
// single-entry decode (nl4_word2)
constexpr int kTab = 8;
constexpr int kMaxThreads = 512;  // one producer warp + up to 15 consumer warps (<= 128 registers)

__device__ __forceinline__ uint32_t ld32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Ring protocol, consumer side: before waiting on the "full" barrier of the slot of ring tile q,
// wait until the producer has issued tile q (issued[0] > q, written after the copy is requested).
// Several warp-sets share the slots, so a set may reach tile q before the slot's previous tile
// (q - stages, another set's) has landed; the barrier would then still be in that tile's phase,
// whose parity is that of the phase before, and a parity wait would return at once. The producer
// issues tile q only after tile q - stages was released, so once it is issued the slot's barrier
// is in tile q's phase. Gives up (false) after kWaitLimitNs or when the abort flag issued[1] is set.
__device__ __forceinline__ bool wait_issued(const volatile int* issued, int q) {
    if (issued[0] > q) {
        __threadfence_block();
        return true;
    }
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(32);
        if (issued[0] > q) {
            __threadfence_block();
            return true;
        }
        if (issued[1]) return false;
        if ((it & 15u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---------------------------------------------------------------- per-format decode

// Byte mask of sign nibble w of sg (0xFF where the weight is negated). The nibble, isolated,
// times sum_i 2^(7i+c) (c = 7 for even w, 3 for odd w) puts bit i at the msb of byte (w/2 + i)
// of the 64-bit product with no carries (copies 7 bits apart, 4 bits wide); a permute with
// sign replication turns those msbs into the mask.
template <int w>
__device__ __forceinline__ uint32_t sign_mask(uint32_t sg) {
    const uint32_t v = sg & (0xFu << (4 * w));
    const unsigned long long p =
        static_cast<unsigned long long>(v) * ((w & 1) ? 0x01020408ull : 0x10204080ull);
    constexpr uint32_t sel = 0x8888u + 0x1111u * (w >> 1) + 0x3210u;
    return prmt(static_cast<uint32_t>(p), static_cast<uint32_t>(p >> 32), sel);
}

// Shared-memory offset (idx << 7) | loff of index byte k of word iw.
template <int k>
__device__ __forceinline__ uint32_t cb_off(uint32_t iw, uint32_t loff) {
    const uint32_t s = k == 0 ? (iw << 7) : (iw >> (8 * k - 7));
    return (s & 0x7f80u) | loff;
}

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
// mask applied (w = x ^ mask) and return ls = 2*sub+1. tab: the codebook replicas (smem offset
// 0); loff: this lane's replica offset.
template <int TYPE, int j>
__device__ __forceinline__ int cb_decode(const CBRow<TYPE>& row, const uint8_t* tab, uint32_t loff, uint32_t W[8]) {
    const uint32_t subw = row.w2(Fmt<TYPE>::SUB);
    const int ls = 2 * static_cast<int>((subw >> (8 * (j >> 1) + 4 * (j & 1))) & 15u) + 1;
    const uint32_t sg = row.w2(Fmt<TYPE>::SGN + j);
    if constexpr (TYPE == MOE_CB3) {
        const uint32_t i0 = row.w2(2 * j), i1 = row.w2(2 * j + 1);
        W[0] = ld32(tab + cb_off<0>(i0, loff)) ^ sign_mask<0>(sg);
        W[1] = ld32(tab + cb_off<1>(i0, loff)) ^ sign_mask<1>(sg);
        W[2] = ld32(tab + cb_off<2>(i0, loff)) ^ sign_mask<2>(sg);
        W[3] = ld32(tab + cb_off<3>(i0, loff)) ^ sign_mask<3>(sg);
        W[4] = ld32(tab + cb_off<0>(i1, loff)) ^ sign_mask<4>(sg);
        W[5] = ld32(tab + cb_off<1>(i1, loff)) ^ sign_mask<5>(sg);
        W[6] = ld32(tab + cb_off<2>(i1, loff)) ^ sign_mask<6>(sg);
        W[7] = ld32(tab + cb_off<3>(i1, loff)) ^ sign_mask<7>(sg);
    } else {
        const uint32_t iw = row.w2(j);
        uint2 g;
        g = *reinterpret_cast<const uint2*>(tab + cb_off<0>(iw, loff));
        W[0] = g.x ^ sign_mask<0>(sg);
        W[1] = g.y ^ sign_mask<1>(sg);
        g = *reinterpret_cast<const uint2*>(tab + cb_off<1>(iw, loff));
        W[2] = g.x ^ sign_mask<2>(sg);
        W[3] = g.y ^ sign_mask<3>(sg);
        g = *reinterpret_cast<const uint2*>(tab + cb_off<2>(iw, loff));
        W[4] = g.x ^ sign_mask<4>(sg);
        W[5] = g.y ^ sign_mask<5>(sg);
        g = *reinterpret_cast<const uint2*>(tab + cb_off<3>(iw, loff));
        W[6] = g.x ^ sign_mask<6>(sg);
        W[7] = g.y ^ sign_mask<7>(sg);
    }
    return ls;
}

// NL4: one 4-byte code word Q (bytes 4k..4k+3 of a block's codes: low nibbles codes 4k..4k+3,
// high nibbles codes 16+4k..19+4k) -> two weight words in nibble order, wa = weights (4k, 16+4k,
// 4k+1, 17+4k) and wb = (4k+2, 18+4k, 4k+3, 19+4k); the staged activation words are permuted to
// match (nl4_act_perm). Each code's low three bits, as byte-permute selectors (a permute reads
// only the low four nibbles of its selector), pick from the table's two 8-entry halves held in
// registers; a sign-replicating permute spreads each code's top bit over its byte, and that mask
// chooses the half. 11 instructions per 8 weights.
__device__ __forceinline__ void nl4_word(const uint32_t tab[kTab], uint32_t Q, uint32_t& wa, uint32_t& wb) {
    const uint32_t s = Q & 0x77777777u, sb = s >> 16, q4 = Q << 4;
    // top bit of nibble i: Q bit 4i+3 = msb of byte i/2 of (Q << 4) for even i, of Q for odd i
    const uint32_t ma = prmt(q4, Q, 0xD9C8u), mb = prmt(q4, Q, 0xFBEAu);
    const uint32_t la = prmt(tab[0], tab[1], s), ha = prmt(tab[2], tab[3], s);
    const uint32_t lb = prmt(tab[0], tab[1], sb), hb = prmt(tab[2], tab[3], sb);
    wa = (la & ~ma) | (ha & ma);
    wb = (lb & ~mb) | (hb & mb);
}

// NL4 for a single entry, with two byte permutes per four weights and no select: the low
// half-table L (words 4, 5) looked up with the code nibbles as selectors, the high half-table H
// (words 6, 7) with the nibbles xor 8. A permute selector nibble of 8 or more returns the sign of
// the byte it picks, 0 or -1, so per code c one lookup gives the wanted half's byte and the other
// 0 or -1; load_table chooses L and H so that the two always add up to table[c] - 1 (possible for
// every table: the shifted values lie in [-128, 126]). The two words enter the dot products
// separately (dp4a is linear) and the block's exact code sum S adds the 1 back: 11 instructions
// per 8 weights with the dot products, against 13 for nl4_word and its one dp4a per word.
// Outputs are in nl4_word's nibble order: a1 + a2 are weights (4k, 16+4k, 4k+1, 17+4k), b1 + b2
// weights (4k+2, 18+4k, 4k+3, 19+4k).
__device__ __forceinline__ void nl4_word2(const uint32_t tab[kTab], uint32_t Q, uint32_t& a1, uint32_t& a2,
                                          uint32_t& b1, uint32_t& b2) {
    const uint32_t Qx = Q ^ 0x88888888u;
    a1 = prmt(tab[4], tab[5], Q);
    a2 = prmt(tab[6], tab[7], Qx);
    b1 = prmt(tab[4], tab[5], Q >> 16);
    b2 = prmt(tab[6], tab[7], Qx >> 16);
}

// The 8 code words x[0..7] of a q8_1 block in the order nl4_word produces the weights:
// staged word 2k = bytes (x[k].0, x[4+k].0, x[k].1, x[4+k].1), word 2k+1 = (x[k].2, x[4+k].2,
// x[k].3, x[4+k].3).
__device__ __forceinline__ void nl4_act_perm(const uint32_t x[8], uint32_t p[8]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        p[2 * k] = prmt(x[k], x[4 + k], 0x5140u);
        p[2 * k + 1] = prmt(x[k], x[4 + k], 0x7362u);
    }
}

// Block j (32 weights) of a Q8_0 / Q4B chunk in shared memory: 8 weight words matching the
// staged activation words, the weight scale d and (Q4B) the minimum m.
template <int TYPE, int j>
__device__ __forceinline__ void blk_decode_smem(const uint8_t* chunk, uint32_t W[8], float& d, float& m) {
    if constexpr (TYPE == MOE_Q8_0) {
        constexpr int L = 34 * j;  // j even: L % 4 == 0; j odd: L % 4 == 2
        const uint8_t* p = chunk + (L & ~3);
        uint32_t r[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) r[i] = ld32(p + 4 * i);
        if constexpr ((j & 1) == 0) {
            d = h2f_bits(r[0]);
#pragma unroll
            for (int k = 0; k < 8; ++k) W[k] = prmt(r[k], r[k + 1], 0x5432u);
        } else {
            d = h2f_bits(r[0] >> 16);
#pragma unroll
            for (int k = 0; k < 8; ++k) W[k] = r[k + 1];
        }
        m = 0.0f;
    } else {  // Q4B: 20-byte blocks, always 4-aligned
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
    }
}

// Block j of a run of NL4 blocks held in registers (18 bytes each from a 4-byte aligned start):
// its four code words and its scale.
template <int j>
__device__ __forceinline__ void nl4_codes(const uint32_t* raw, uint32_t qs[4], float& d) {
    constexpr int L = 18 * j;
    constexpr int i = L >> 2;
    if constexpr ((j & 1) == 0) {
        d = h2f_bits(raw[i]);
#pragma unroll
        for (int k = 0; k < 4; ++k) qs[k] = prmt(raw[i + k], raw[i + k + 1], 0x5432u);
    } else {
        d = h2f_bits(raw[i] >> 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) qs[k] = raw[i + 1 + k];
    }
}

template <int j>
__device__ __forceinline__ void nl4_decode(const uint32_t* raw, const uint32_t tab[kTab], uint32_t W[8], float& d) {
    uint32_t qs[4];
    nl4_codes<j>(raw, qs, d);
#pragma unroll
    for (int k = 0; k < 4; ++k) nl4_word(tab, qs[k], W[2 * k], W[2 * k + 1]);
}

// The single-entry decode of block j: both permute words per weight word (see nl4_word2).
template <int j>
__device__ __forceinline__ void nl4_decode2(const uint32_t* raw, const uint32_t tab[kTab], uint32_t W1[8], uint32_t W2[8],
                                            float& d) {
    uint32_t qs[4];
    nl4_codes<j>(raw, qs, d);
#pragma unroll
    for (int k = 0; k < 4; ++k) nl4_word2(tab, qs[k], W1[2 * k], W2[2 * k], W1[2 * k + 1], W2[2 * k + 1]);
}

// Sub-block j (32 weights) of a slot chunk: codes -> 8 words of biased values u (one code per
// byte), matching the staged activation words. q: the sub-block's code words (4 for 4-bit
// codes, 2 for 2-bit codes).
template <int TYPE>
__device__ __forceinline__ void slot_decode(const uint32_t* q, uint32_t W[8]) {
    if constexpr (TYPE == MOE_CB3X) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            W[k] = q[k] & 0x0f0f0f0fu;
            W[4 + k] = (q[k] >> 4) & 0x0f0f0f0fu;
        }
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            W[2 * p] = (q[0] >> (2 * p)) & 0x03030303u;
            W[2 * p + 1] = (q[1] >> (2 * p)) & 0x03030303u;
        }
    }
}

// ---------------------------------------------------------------- work split

struct Tile {
    int g, row0, nrows;
};

// rdiv divides by rbpg; qlim: the indices below which its reciprocal is exact (the 64-bit
// division beyond)
__device__ __forceinline__ Tile next_tile(long long& cur, long long end, int rbpg, int rt8, const SmallDiv& rdiv,
                                          long long qlim) {
    const int g = cur < qlim ? rdiv.div(static_cast<int>(cur)) : static_cast<int>(cur / rbpg);
    const int off = static_cast<int>(cur - static_cast<long long>(g) * rbpg);
    long long n = rbpg - off < rt8 ? rbpg - off : rt8;
    if (n > end - cur) n = end - cur;
    cur += n;
    return Tile{g, off * 8, static_cast<int>(n) * 8};
}

// Per-group facts cached in shared memory for the whole launch: expert, entry range, cost per
// 8-row block (0 for a skipped group), and the inclusive prefix of the group costs.
struct GroupInfo {
    const uint8_t* ptr;
    int x, e0, e1, cost;
};

// Flattened (group, 8-row block) index at which the cumulative cost reaches `target`
// (binary search over the cost prefix cum[0..G]).
__device__ __forceinline__ long long locate(const GroupInfo* gi, const long long* cum, int G, int rbpg,
                                            long long target) {
    if (target >= cum[G]) return static_cast<long long>(G) * rbpg;
    int lo = 0, hi = G - 1;  // first g with cum[g+1] > target
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid + 1] > target) hi = mid;
        else lo = mid + 1;
    }
    return static_cast<long long>(lo) * rbpg + (target - cum[lo]) / gi[lo].cost;
}

// ---------------------------------------------------------------- shared staging

// The codebook in shared memory at offset 0: CB3 256 x 32 lane replicas of 4 bytes, CB2 256 x 16
// replicas of 8 bytes, both in x-form and both 32 KB with entry idx at offset idx*128.
// t, nt: this thread's index among nt participating threads (whole warps, warp-aligned).
template <int TYPE>
__device__ __forceinline__ void stage_codebook(const GemvArgs& a, uint8_t* smem, int t, int nt) {
    if constexpr (Fmt<TYPE>::CB) {
        // a warp takes 32 consecutive grid words at a time (one coalesced load), converts them to
        // x-form bytewise and writes whole 128-byte entry rows, lane l word l of a row, so that the
        // replica stores hit 32 different banks: a CB3 entry is one word (32 replicas), a CB2 entry
        // two (16 replicas of the pair, word h of the entry at bytes 4h..4h+3 of each)
        constexpr int kWords = TYPE == MOE_CB2 ? 512 : 256;
        const uint32_t* cbw = reinterpret_cast<const uint32_t*>(a.codebook);
        uint32_t* rows = reinterpret_cast<uint32_t*>(smem);
        const int lane = t & 31;
        bool even = false;
        for (int w0 = t - lane; w0 < kWords; w0 += nt) {
            const uint32_t g = __ldg(cbw + w0 + lane);
            even |= (g & 0x01010101u) != 0x01010101u;
            uint32_t v = 0;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int x = static_cast<int8_t>(g >> (8 * bb));
                v |= (static_cast<uint32_t>((x - 1) >> 1) & 0xffu) << (8 * bb);
            }
            if constexpr (TYPE == MOE_CB3) {
#pragma unroll 8
                for (int j = 0; j < 32; ++j) rows[(w0 + j) * 32 + lane] = __shfl_sync(0xffffffffu, v, j);
            } else {
#pragma unroll 8
                for (int j = 0; j < 16; ++j)
                    rows[((w0 >> 1) + j) * 32 + lane] = __shfl_sync(0xffffffffu, v, 2 * j + (lane & 1));
            }
        }
        if (even) set_err(a.err, MOE_ERR_CODEBOOK);
    }
}

template <int TYPE>
__device__ __forceinline__ void load_table(const GemvArgs& a, uint32_t tab[kTab]) {
    if constexpr (TYPE == MOE_NL4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) tab[k] = __ldg(reinterpret_cast<const uint32_t*>(a.codebook) + k);
        // half-tables of nl4_word2: for j < 8 and the shifted values v = table[j] - 1,
        // w = table[j + 8] - 1, bytes L[j] = v + sH and H[j] = w + sL where sL, sH (0 or 1) are the
        // signs of L[j] and H[j] themselves: then L[j] + (H[j] < 0 ? -1 : 0) = v and
        // H[j] + (L[j] < 0 ? -1 : 0) = w. The first consistent (sL, sH) of (0,0), (0,1), (1,0),
        // (1,1) is taken; one exists for any v, w in [-128, 126].
        const int8_t* t = a.codebook;
        uint32_t lo[2] = {0, 0}, hi[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int v = t[j] - 1, w = t[j + 8] - 1;
            int l = v, h = w;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int sL = c >> 1, sH = c & 1;
                const int l2 = v + sH, h2 = w + sL;
                if ((l2 < 0) == (sL != 0) && (h2 < 0) == (sH != 0) && l2 >= -128 && h2 >= -128 && l2 <= 127 && h2 <= 127) {
                    l = l2;
                    h = h2;
                    break;
                }
            }
            lo[j >> 2] |= (static_cast<uint32_t>(l) & 0xFFu) << (8 * (j & 3));
            hi[j >> 2] |= (static_cast<uint32_t>(h) & 0xFFu) << (8 * (j & 3));
        }
        tab[4] = lo[0];
        tab[5] = lo[1];
        tab[6] = hi[0];
        tab[7] = hi[1];
    } else {
#pragma unroll
        for (int k = 0; k < kTab; ++k) tab[k] = 0;
    }
}

// Staged activations: slot i of the shared-memory act region holds one q8_1 row as 16-byte code
// halves (q[(i*2 + h)*nbp + bp], bp = b + b/8: conflict-free 128-bit loads) and (d, aux) pairs
// (q2[i*nb + b]); aux = exact code sum S times the format's factor (CB and NL4: S, slots:
// -(2 bias - 1) S), s (Q4B) or 0. Row `src` < 0 stages zeros; rows are read through the read-only path.
template <int TYPE>
__device__ __forceinline__ void put_staged(const GemvArgs& a, uint8_t* smem, int slot, int b, uint32_t w[9]);

template <int TYPE>
__device__ __forceinline__ void stage_block(const GemvArgs& a, uint8_t* smem, int slot, int src, int b) {
    uint32_t w[9];
    if (src >= 0) {
        const uint32_t* p = reinterpret_cast<const uint32_t*>(a.act + static_cast<int64_t>(src) * a.nb + b);
#pragma unroll
        for (int k = 0; k < 9; ++k) w[k] = __ldg(p + k);
    } else {
#pragma unroll
        for (int k = 0; k < 9; ++k) w[k] = 0;
    }
    put_staged<TYPE>(a, smem, slot, b, w);
}

// Block b of a q8_1 row held as nine words w (header, then code words) into slot `slot`.
template <int TYPE>
__device__ __forceinline__ void put_staged(const GemvArgs& a, uint8_t* smem, int slot, int b, uint32_t w[9]) {
    int4* q = reinterpret_cast<int4*>(smem + a.off_actq);
    float2* q2 = reinterpret_cast<float2*>(smem + a.off_act2);
    const int bp = b + (b >> 3);
    if constexpr (TYPE == MOE_NL4) {
        uint32_t p[8];
        nl4_act_perm(w + 1, p);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[1 + k] = p[k];
    }
    q[(slot * 2 + 0) * a.nbp + bp] = make_int4(w[1], w[2], w[3], w[4]);
    q[(slot * 2 + 1) * a.nbp + bp] = make_int4(w[5], w[6], w[7], w[8]);
    float aux = 0.0f;
    if constexpr (Fmt<TYPE>::CB || Fmt<TYPE>::SLOT) {
        int S = 0;
#pragma unroll
        for (int k = 1; k < 9; ++k) S = dp4a(w[k], 0x01010101u, S);
        // CB: sum s g q = 2 dot(x ^ mask, q) + S; slots: = 2 dot(u, q) - (2 bias - 1) S
        if constexpr (Fmt<TYPE>::SLOT) S *= -(2 * Fmt<TYPE>::BIAS - 1);
        aux = __int_as_float(S);
    } else if constexpr (TYPE == MOE_Q4B) {
        aux = h2f_bits(w[0] >> 16);
    } else if constexpr (TYPE == MOE_NL4) {
        int S = 0;  // the exact code sum, for the single-entry decode's shift
#pragma unroll
        for (int k = 1; k < 9; ++k) S = dp4a(w[k], 0x01010101u, S);
        aux = __int_as_float(S);
    }
    q2[slot * a.nb + b] = make_float2(h2f_bits(w[0]), aux);
}

// All n rows of the activation matrix into slots 0..n-1.
template <int TYPE>
__device__ __forceinline__ void stage_all(const GemvArgs& a, uint8_t* smem, int n, int t, int nt) {
    for (int i = t; i < n * a.nb; i += nt) {
        const int r = i / a.nb;
        stage_block<TYPE>(a, smem, r, r, i - r * a.nb);
    }
}

// The activation rows of entries e0 .. e0+ne-1 (ent[e].x, -1 when invalid) into slots slot0 ...
template <int TYPE>
__device__ __forceinline__ void stage_entries(const GemvArgs& a, uint8_t* smem, const int2* ent, int e0, int ne,
                                              int slot0, int t, int nt) {
    for (int i = t; i < ne * a.nb; i += nt) {
        const int s = i / a.nb;
        stage_block<TYPE>(a, smem, slot0 + s, ent[e0 + s].x, i - s * a.nb);
    }
}

template <int NE>
__device__ __forceinline__ void load_act(const GemvArgs& a, const uint8_t* smem, int b, const int slots[NE],
                                         uint32_t A[NE][8], float dx[NE], float aux[NE]) {
    const int4* q = reinterpret_cast<const int4*>(smem + a.off_actq);
    const float2* q2 = reinterpret_cast<const float2*>(smem + a.off_act2);
    const int bp = b + (b >> 3);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const int4 lo = q[(slots[e] * 2 + 0) * a.nbp + bp], hi = q[(slots[e] * 2 + 1) * a.nbp + bp];
        A[e][0] = lo.x; A[e][1] = lo.y; A[e][2] = lo.z; A[e][3] = lo.w;
        A[e][4] = hi.x; A[e][5] = hi.y; A[e][6] = hi.z; A[e][7] = hi.w;
        const float2 v = q2[slots[e] * a.nb + b];
        dx[e] = v.x;
        aux[e] = v.y;
    }
}

// ---------------------------------------------------------------- compute

// Two independent dp4a chains (even and odd words) halve the dependent latency.
__device__ __forceinline__ int dot8(const uint32_t W[8], const uint32_t A[8]) {
    int d0 = 0, d1 = 0;
#pragma unroll
    for (int w = 0; w < 8; w += 2) {
        d0 = dp4a(W[w], A[w], d0);
        d1 = dp4a(W[w + 1], A[w + 1], d1);
    }
    return d0 + d1;
}

// One lane's row of chunk c (256 weights) against NE staged entries: chunk partials acc[e].
// All lanes of a warp read the same activation block at the same time (broadcast loads).
template <int TYPE, int NE, int j>
__device__ __forceinline__ void cb_block(const GemvArgs& a, const uint8_t* smem, const CBRow<TYPE>& row, int c,
                                         uint32_t loff, const int* slots, float acc[NE]) {
    uint32_t A[NE][8];
    float dx[NE], sq[NE];
    load_act<NE>(a, smem, c * 8 + j, slots, A, dx, sq);
    uint32_t W[8];
    const int ls = cb_decode<TYPE, j>(row, smem, loff, W);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        const int isum = 2 * dot8(W, A[e]) + __float_as_int(sq[e]);
        acc[e] = fmaf(static_cast<float>(ls * isum), dx[e], acc[e]);
    }
}

// Block j (0..3) of a 72-byte run of four NL4 blocks held in raw[18]; b: its block index in the row.
template <int NE, int j>
__device__ __forceinline__ void nl4_block(const GemvArgs& a, const uint8_t* smem, const uint32_t raw[18],
                                          const uint32_t tab[kTab], int b, const int* slots, float acc[NE]) {
    uint32_t A[NE][8];
    float dx[NE], aux[NE];
    load_act<NE>(a, smem, b, slots, A, dx, aux);
    float dw;
    if constexpr (NE == 1) {
        uint32_t W1[8], W2[8];
        nl4_decode2<j>(raw, tab, W1, W2, dw);
        int d0 = 0, d1 = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            d0 = dp4a(W1[w], A[0][w], d0);
            d1 = dp4a(W2[w], A[0][w], d1);
        }
        const int isum = d0 + d1 + __float_as_int(aux[0]);
        acc[0] = fmaf(__fmul_rn(dw, dx[0]), static_cast<float>(isum), acc[0]);
    } else {
        uint32_t W[8];
        nl4_decode<j>(raw, tab, W, dw);
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = fmaf(__fmul_rn(dw, dx[e]), static_cast<float>(dot8(W, A[e])), acc[e]);
    }
}

template <int TYPE, int NE, int j>
__device__ __forceinline__ void plain_block(const GemvArgs& a, const uint8_t* smem, const uint8_t* chunk,
                                            const uint32_t* raw, const uint32_t tab[kTab], int c, const int* slots,
                                            float acc[NE]) {
    uint32_t A[NE][8];
    float dx[NE], aux[NE];
    load_act<NE>(a, smem, c * 8 + j, slots, A, dx, aux);
    uint32_t W[8];
    float dw, mw = 0.0f;
    if constexpr (TYPE == MOE_NL4) nl4_decode<j>(raw, tab, W, dw);
    else blk_decode_smem<TYPE, j>(chunk, W, dw, mw);
#pragma unroll
    for (int e = 0; e < NE; ++e) {
        acc[e] = fmaf(__fmul_rn(dw, dx[e]), static_cast<float>(dot8(W, A[e])), acc[e]);
        if constexpr (TYPE == MOE_Q4B) acc[e] = fmaf(mw, aux[e], acc[e]);
    }
}

// Sub-block j of a slot chunk (j may be a run-time index: the CB3X chunk loop is kept rolled two
// sub-blocks at a time, which keeps the hot code small enough for the instruction caches).
template <int TYPE, int NE>
__device__ __forceinline__ void slot_block(const GemvArgs& a, const uint8_t* smem, const uint32_t* q, uint32_t subw,
                                           int c, int j, const int* slots, float acc[NE]) {
    uint32_t A[NE][8];
    float dx[NE], aux[NE];
    load_act<NE>(a, smem, c * 8 + j, slots, A, dx, aux);
    const int ls = 2 * static_cast<int>((subw >> (8 * (j >> 1) + 4 * (j & 1))) & 15u) + 1;
    if constexpr (TYPE == MOE_CB3X) {
        // The low nibbles (weights 4k..4k+3 of word k) go into dp4a as they are; the high ones
        // (weights 16+4k..) stay in place as 16 x code, through the unsigned-by-signed dp4a, and
        // the sum's factor 16 comes off with one shift (exact: it is a multiple of 16), so no
        // nibble is shifted down: 2 (low + high) = 2 low + high16 / 8.
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            lo[k] = q[k] & 0x0f0f0f0fu;
            hi[k] = q[k] & 0xf0f0f0f0u;
        }
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            int dl = 0, dh = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dl = dp4a(lo[k], A[e][k], dl);
                dh = dp4a_us(hi[k], A[e][4 + k], dh);
            }
            const int isum = 2 * dl + (dh >> 3) + __float_as_int(aux[e]);
            acc[e] = fmaf(static_cast<float>(ls * isum), dx[e], acc[e]);
        }
    } else {
        uint32_t W[8];
        slot_decode<TYPE>(q, W);
#pragma unroll
        for (int e = 0; e < NE; ++e) {
            const int isum = 2 * dot8(W, A[e]) + __float_as_int(aux[e]);
            acc[e] = fmaf(static_cast<float>(ls * isum), dx[e], acc[e]);
        }
    }
}

// The code words of 16 bytes at p (16-byte aligned when `al16`, else 8-byte aligned).
__device__ __forceinline__ void ld16(const uint8_t* p, bool al16, uint32_t q[4]) {
    if (al16) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
    } else {
        const uint2 v0 = *reinterpret_cast<const uint2*>(p), v1 = *reinterpret_cast<const uint2*>(p + 8);
        q[0] = v0.x; q[1] = v0.y; q[2] = v1.x; q[3] = v1.y;
    }
}

template <int TYPE, int NE>
__device__ __forceinline__ void slot_chunk(const GemvArgs& a, const uint8_t* smem, const uint8_t* rowp, int c,
                                           const int* slots, float acc[NE]) {
    const uint2 sc = *reinterpret_cast<const uint2*>(rowp + a.nch * Fmt<TYPE>::CHUNK + c * 8);
    const float D = h2f_bits(sc.x);
    const uint8_t* codes = rowp + c * Fmt<TYPE>::CHUNK;
    const bool al16 = (a.row_bytes & 15) == 0;
    uint32_t q[4];
    if constexpr (TYPE == MOE_CB3X) {  // 16 bytes per sub-block
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
            ld16(codes + 16 * j, al16, q);
            slot_block<TYPE, NE>(a, smem, q, sc.y, c, j, slots, acc);
        }
    } else {  // 8 bytes per sub-block: two sub-blocks per 16-byte load
        ld16(codes + 0, al16, q); slot_block<TYPE, NE>(a, smem, q, sc.y, c, 0, slots, acc);
        slot_block<TYPE, NE>(a, smem, q + 2, sc.y, c, 1, slots, acc);
        ld16(codes + 16, al16, q); slot_block<TYPE, NE>(a, smem, q, sc.y, c, 2, slots, acc);
        slot_block<TYPE, NE>(a, smem, q + 2, sc.y, c, 3, slots, acc);
        ld16(codes + 32, al16, q); slot_block<TYPE, NE>(a, smem, q, sc.y, c, 4, slots, acc);
        slot_block<TYPE, NE>(a, smem, q + 2, sc.y, c, 5, slots, acc);
        ld16(codes + 48, al16, q); slot_block<TYPE, NE>(a, smem, q, sc.y, c, 6, slots, acc);
        slot_block<TYPE, NE>(a, smem, q + 2, sc.y, c, 7, slots, acc);
    }
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = __fmul_rn(D, acc[e]);
}

template <int TYPE, int NE>
__device__ __forceinline__ void lane_chunk(const GemvArgs& a, const uint8_t* smem, const uint8_t* tile, int row, int c,
                                           uint32_t loff, const uint32_t tab[kTab], const int* slots, float acc[NE]) {
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[e] = 0.0f;
    const uint8_t* chunk = tile + row * a.row_bytes + c * Fmt<TYPE>::CHUNK;
    if constexpr (Fmt<TYPE>::SLOT) {
        slot_chunk<TYPE, NE>(a, smem, tile + row * a.row_bytes, c, slots, acc);
    } else if constexpr (Fmt<TYPE>::CB) {
        CBRow<TYPE> rr;
        rr.load(chunk);
        const float D = rr.D();
        cb_block<TYPE, NE, 0>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 1>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 2>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 3>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 4>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 5>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 6>(a, smem, rr, c, loff, slots, acc);
        cb_block<TYPE, NE, 7>(a, smem, rr, c, loff, slots, acc);
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[e] = __fmul_rn(D, acc[e]);
    } else if constexpr (TYPE == MOE_NL4) {
        // two rounds of four 18-byte blocks (72 bytes, 8-byte aligned), the loop kept rolled so the
        // hot code stays small enough for the instruction caches
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            uint32_t raw[18];
#pragma unroll
            for (int k = 0; k < 9; ++k) {
                const uint2 v = *reinterpret_cast<const uint2*>(chunk + 72 * p + 8 * k);
                raw[2 * k] = v.x;
                raw[2 * k + 1] = v.y;
            }
            nl4_block<NE, 0>(a, smem, raw, tab, c * 8 + 4 * p, slots, acc);
            nl4_block<NE, 1>(a, smem, raw, tab, c * 8 + 4 * p + 1, slots, acc);
            nl4_block<NE, 2>(a, smem, raw, tab, c * 8 + 4 * p + 2, slots, acc);
            nl4_block<NE, 3>(a, smem, raw, tab, c * 8 + 4 * p + 3, slots, acc);
        }
    } else {
        const uint32_t raw[1] = {0};
        plain_block<TYPE, NE, 0>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 1>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 2>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 3>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 4>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 5>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 6>(a, smem, chunk, raw, tab, c, slots, acc);
        plain_block<TYPE, NE, 7>(a, smem, chunk, raw, tab, c, slots, acc);
    }
}

// The warp's chunks (c = wi, wi + WPS, ...) of the tile's rows (lane = row) -> chunk partials
// part[(c*4 + e)*RT + row].
template <int TYPE, int NE>
__device__ __forceinline__ void warp_chunks(const GemvArgs& a, const uint8_t* smem, const uint8_t* tile, float* part,
                                            int wi, int lane, uint32_t loff, const uint32_t tab[kTab], const int* slots) {
    for (int c = wi; c < a.nch; c += a.WPS) {
        float acc[NE];
        lane_chunk<TYPE, NE>(a, smem, tile, lane, c, loff, tab, slots, acc);
#pragma unroll
        for (int e = 0; e < NE; ++e) part[(c * kMaxEntriesPerPass + e) * a.RT + lane] = acc[e];
    }
}

template <int TYPE>
__device__ __forceinline__ void compute_batch(const GemvArgs& a, const uint8_t* smem, const uint8_t* tile, float* part,
                                              int ne, int wi, int lane, int nrows, uint32_t loff, const uint32_t tab[kTab],
                                              const int slots[4]) {
    if (lane >= nrows) return;
    // batches of 3 entries run the 4-entry code (the fourth slot repeats the third; its result
    // is never read)
    if (ne == 1) warp_chunks<TYPE, 1>(a, smem, tile, part, wi, lane, loff, tab, slots);
    else if (ne == 2) warp_chunks<TYPE, 2>(a, smem, tile, part, wi, lane, loff, tab, slots);
    else warp_chunks<TYPE, 4>(a, smem, tile, part, wi, lane, loff, tab, slots);
}

// Fixed-order sum over the chunks (c = 0 .. nch-1) of each (row, entry), written to the entry's
// output row.
// STRIDE: entries per chunk in the partials layout (part[(c*STRIDE + e)*RT + row]).
template <int STRIDE = kMaxEntriesPerPass>
__device__ __forceinline__ void reduce_write(const GemvArgs& a, const float* part, const int2* ent, int b0,
                                             const Tile& t, int ne, int lane) {
    if (lane >= t.nrows) return;
    for (int e = 0; e < ne; ++e) {
        const int2 en = ent[b0 + e];
        if (en.x < 0) continue;
        float s = part[e * a.RT + lane];
        for (int c = 1; c < a.nch; ++c) s = __fadd_rn(s, part[(c * STRIDE + e) * a.RT + lane]);
        a.out[static_cast<int64_t>(en.y) * a.out_stride + t.row0 + lane] = s;
    }
}

template <int TYPE>
__global__ void __launch_bounds__(kMaxThreads, 1) gemv_kernel(const GemvArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NT = blockDim.x;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
    uint64_t* empty = full + a.stages;
    // misc: [0] tiles issued, [1] abort flag, [2] n_groups, [64 + s] arrivals at ring slot s (the
    // last warp of a tile sums its chunk partials)
    int* misc = reinterpret_cast<int*>(smem + a.off_misc);
    GroupInfo* gi = reinterpret_cast<GroupInfo*>(smem + a.off_grp);
    long long* cum = reinterpret_cast<long long*>(gi + a.cap_groups);
    int2* ent = reinterpret_cast<int2*>(smem + a.off_ent);  // per entry: (act row or -1, out row)
    const int S = a.stages;
    const SmallDiv sdiv(S);
    const int rbpg = a.rows >> 3, rt8 = a.RT >> 3;
    // (the 2^31 - 1 cap keeps the index's int conversion exact)
    const SmallDiv rdiv(rbpg);
    const long long qlim = rbpg > 1 ? (0xFFFFFFFFll / (rbpg - 1) < 0x7FFFFFFFll ? 0xFFFFFFFFll / (rbpg - 1) : 0x7FFFFFFFll)
                                    : 0x7FFFFFFFll;
    // the whole activation matrix fits in the act region: staged once, indexed by act row
    const bool all_rows = a.n_act_rows <= a.act_cap;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], a.WPS + 1);
            misc[64 + s] = 0;
        }
        misc[0] = 0;
        misc[1] = 0;
    }
    fence_barrier_init();
    // static data first (before the dependency wait): the codebook replicas and the NL4 table
    if (warp > 0) stage_codebook<TYPE>(a, smem, tid - 32, NT - 32);
    uint32_t tab[kTab];
    load_table<TYPE>(a, tab);
    if (!a.prefetch_before_wait) pdl_wait();

    // One round of independent loads: the group count, every group slot and every entry slot (the
    // arrays hold cap_groups / cap_entries items whatever *n_groups is), and, for gate/up, the
    // activation rows (inputs after the wait).
    if (tid == 0) misc[2] = *a.n_groups;
    for (int g = tid; g < a.cap_groups; g += NT)
        gi[g] = GroupInfo{nullptr, a.grp_expert[g], a.grp_start[g], a.grp_start[g + 1], 0};
    for (int e = tid; e < a.cap_entries; e += NT) {
        const int in = a.ent_in ? a.ent_in[e] : e;
        const int o = a.ent_out ? a.ent_out[e] : e;
        const bool ok = in >= 0 && in < a.n_act_rows && o >= 0 && o < a.out_rows;
        ent[e] = make_int2(ok ? in : -1, o);
    }
    if (all_rows && !a.prefetch_before_wait) stage_all<TYPE>(a, smem, a.n_act_rows, tid, NT);
    __syncthreads();
    int G = misc[2];
    if (G < 0 || G > a.cap_groups) {
        if (blockIdx.x == 0 && tid == 0) set_err(a.err, MOE_ERR_NGROUPS);
        G = G < 0 ? 0 : a.cap_groups;
    }
    // validate the groups (one per thread), fetch their weight pointers, cost them
    for (int g = tid; g < G; g += NT) {
        GroupInfo v = gi[g];
        bool ok = true;
        const bool rep = blockIdx.x == 0;
        if (v.x < 0 || v.x >= a.n_experts) {
            ok = false;
            if (rep) set_err(a.err, MOE_ERR_EXPERT);
        } else if (v.e0 < 0 || v.e1 < v.e0 || v.e1 > a.cap_entries) {
            ok = false;
            if (rep) set_err(a.err, MOE_ERR_START);
        } else if (v.e1 == v.e0) {
            ok = false;
        } else {
            v.ptr = static_cast<const uint8_t*>(a.w[v.x]);
            if (reinterpret_cast<uintptr_t>(v.ptr) & 15u) {
                ok = false;
                if (rep) set_err(a.err, MOE_ERR_ALIGN);
            } else if (rep) {
                for (int e = v.e0; e < v.e1; ++e)
                    if (ent[e].x < 0) set_err(a.err, MOE_ERR_ENTRY);
            }
        }
        v.cost = ok ? a.alpha + (v.e1 - v.e0) : 0;
        gi[g] = v;
    }
    __syncthreads();
    if (warp == 0) {
        long long run = 0;
        if (lane == 0) cum[0] = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            long long v = g < G ? static_cast<long long>(gi[g].cost) * rbpg : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (g < G) cum[g + 1] = run + v;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
    const long long tot = cum[G];
    const long long rb0 = locate(gi, cum, G, rbpg, tot * blockIdx.x / gridDim.x);
    const long long rb1 = locate(gi, cum, G, rbpg, tot * (blockIdx.x + 1) / gridDim.x);

    // producer: the first S tiles may start before the dependency wait (down kernel)
    long long pcur = rb0;
    int issued = 0;
    const uint64_t pol = l2_evict_first();  // the weights are read once per call
    auto produce_one = [&](bool wait_empty) -> int {  // 1 issued, 0 range exhausted, -1 timeout
        while (pcur < rb1) {
            const Tile t = next_tile(pcur, rb1, rbpg, rt8, rdiv, qlim);
            const GroupInfo g = gi[t.g];
            if (g.cost == 0) continue;
            const int iq = sdiv.div(issued), s = issued - iq * S;
            if (wait_empty && issued >= S) {
                if (!mbar_wait_bounded(&empty[s], static_cast<uint32_t>(iq - 1) & 1u)) return -1;
            }
            const uint32_t bytes = static_cast<uint32_t>(t.nrows) * static_cast<uint32_t>(a.row_bytes);
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s_hint(smem + a.off_ring + static_cast<size_t>(s) * a.stage_bytes,
                          g.ptr + static_cast<size_t>(t.row0) * a.row_bytes, bytes, &full[s], pol);
            ++issued;
            __threadfence_block();
            *reinterpret_cast<volatile int*>(misc) = issued;
            return 1;
        }
        return 0;
    };
    if (tid == 0)
        for (int s = 0; s < S; ++s)
            if (produce_one(false) != 1) break;
    if (a.prefetch_before_wait) pdl_wait();
    pdl_trigger();
    if (rb0 == rb1) return;

    if (warp == 0) {
        if (lane == 0) {
            for (;;) {
                if (*reinterpret_cast<volatile int*>(misc + 1)) break;
                const int rc = produce_one(true);
                if (rc == 0) break;
                if (rc < 0) {
                    set_err(a.err, MOE_ERR_TIMEOUT);
                    *reinterpret_cast<volatile int*>(misc + 1) = 1;
                    break;
                }
            }
        }
        return;
    }

    // consumers: warp-set `set` takes the CTA's tiles set, set + TP, ...; within a set, warp wi
    // takes chunks wi, wi + WPS, ... of every row of the tile (lane = row)
    const int cw = warp - 1;
    const int set = cw / a.WPS, wi = cw - set * a.WPS;
    const int ct = tid - 32, cnt = a.CW * 32;
    const uint32_t loff = TYPE == MOE_CB3 ? lane * 4u : (lane & 15u) * 8u;

    // Activations: staged already (gate/up) or now, after the wait (down), when they all fit;
    // otherwise a range spanning at most two groups of at most 4 entries each has both groups'
    // rows staged here. Any other range, and any range holding a group of more than 4 entries,
    // is walked by warp-set 0 alone with barriers between entry batches, restaging (unless all
    // rows are staged) at every group or batch change.
    const int gA = static_cast<int>(rb0 / rbpg), gB = static_cast<int>((rb1 - 1) / rbpg);
    const int neA = gi[gA].e1 - gi[gA].e0, neB = gi[gB].e1 - gi[gB].e0;
    // A group of more than kMaxEntriesPerPass entries takes several entry batches per tile; those
    // run on the barrier path (the last-warp path keeps one batch's partials per slot).
    bool multi = false;
    for (int g = gA; g <= gB; ++g) multi |= gi[g].cost != 0 && gi[g].e1 - gi[g].e0 > kMaxEntriesPerPass;
    const bool two = !all_rows && !multi && gB - gA <= 1;
    const bool fast = !multi && (all_rows || two);
    if (all_rows && a.prefetch_before_wait) {
        stage_all<TYPE>(a, smem, a.n_act_rows, ct, cnt);
        named_sync(1, cnt);
    } else if (two) {
        if (gi[gA].cost) stage_entries<TYPE>(a, smem, ent, gi[gA].e0, neA, 0, ct, cnt);
        if (gB != gA && gi[gB].cost) stage_entries<TYPE>(a, smem, ent, gi[gB].e0, neB, kMaxEntriesPerPass, ct, cnt);
        named_sync(1, cnt);
    } else if (!fast && set != 0) {
        return;
    }
    const int TPe = fast ? a.TP : 1;
    const SmallDiv tdiv(TPe);
    const int scnt = a.WPS * 32, st = ct - set * scnt;  // thread index within the set

    long long ccur = rb0;
    int k = 0, cur_g = -1, cur_b0 = -1;
    bool aborted = false;
    while (ccur < rb1) {
        const Tile t = next_tile(ccur, rb1, rbpg, rt8, rdiv, qlim);
        const GroupInfo g = gi[t.g];
        if (g.cost == 0) continue;
        const int kk = k++;
        if (tdiv.mod(kk) != set) continue;
        const int kq = sdiv.div(kk), slot = kk - kq * S;
        const uint32_t parity = static_cast<uint32_t>(kq) & 1u;
        const uint8_t* tile = smem + a.off_ring + static_cast<size_t>(slot) * a.stage_bytes;
        float* part = reinterpret_cast<float*>(smem + a.off_part + static_cast<size_t>(slot) * a.part_bytes);
        if (!aborted && !(wait_issued(misc, kk) && mbar_wait_bounded(&full[slot], parity))) {
            aborted = true;
            set_err(a.err, MOE_ERR_TIMEOUT);
            *reinterpret_cast<volatile int*>(misc + 1) = 1;
        }
        if (*reinterpret_cast<volatile int*>(misc + 1)) aborted = true;
        // entry batches: one for a group of up to 4 entries
        for (int b0 = g.e0; b0 < g.e1; b0 += kMaxEntriesPerPass) {
            const int ne = g.e1 - b0 < kMaxEntriesPerPass ? g.e1 - b0 : kMaxEntriesPerPass;
            int slots[4];
            if (all_rows) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = ent[b0 + (e < ne ? e : ne - 1)].x;
                    slots[e] = r < 0 ? 0 : r;
                }
            } else {
                const int s0 = two && t.g != gA ? kMaxEntriesPerPass : 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) slots[e] = s0 + (e < ne ? e : ne - 1);
            }
            if (!fast && !all_rows && (t.g != cur_g || b0 != cur_b0)) {
                named_sync(1, scnt);
                stage_entries<TYPE>(a, smem, ent, b0, ne, 0, st, scnt);
                named_sync(1, scnt);
                cur_g = t.g;
                cur_b0 = b0;
            }
            if (!aborted) compute_batch<TYPE>(a, smem, tile, part, ne, wi, lane, t.nrows, loff, tab, slots);
            if (fast) {
                // release the weights, then the set's last warp sums the chunk partials
                __syncwarp();
                __threadfence_block();
                int last = 0;
                if (lane == 0) {
                    mbar_arrive(&empty[slot]);
                    last = atomicAdd(&misc[64 + slot], 1) == a.WPS - 1;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence_block();
                    if (!aborted) reduce_write(a, part, ent, b0, t, ne, lane);
                    __syncwarp();
                    if (lane == 0) {
                        misc[64 + slot] = 0;
                        mbar_arrive(&empty[slot]);
                    }
                }
            } else {
                named_sync(1, scnt);
                if (wi == 0 && !aborted) reduce_write(a, part, ent, b0, t, ne, lane);
                named_sync(1, scnt);
            }
        }
        if (!fast) {
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[slot]);
                if (wi == 0) mbar_arrive(&empty[slot]);
            }
        }
    }
    if (aborted && ct == 0) {
        // wait (bounded) for the copies still in flight into this CTA's shared memory
        const int n = *reinterpret_cast<volatile int*>(misc);
        for (int q = n - S > 0 ? n - S : 0; q < n; ++q)
            mbar_wait_bounded(&full[q % S], static_cast<uint32_t>(q / S) & 1u);
    }
}

// Test hook: isum[r][b] of `rows` rows of one blob against one q8_1 row, by the same decode
// and dot-product code (one thread per (row, chunk), the blob read straight from global memory).
template <int TYPE>
__global__ void __launch_bounds__(256) isum_kernel(const GemvArgs a, const uint8_t* blob, int rows, int32_t* isum) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31;
    stage_codebook<TYPE>(a, smem, tid, NT);
    stage_all<TYPE>(a, smem, 1, tid, NT);
    __syncthreads();
    uint32_t tab[kTab];
    load_table<TYPE>(a, tab);
    const int i = blockIdx.x * NT + tid;
    if (i >= rows * a.nch) return;
    const int r = i / a.nch, c = i - r * a.nch;
    const uint8_t* chunk = blob + static_cast<size_t>(r) * a.row_bytes + c * Fmt<TYPE>::CHUNK;
    const uint32_t loff = TYPE == MOE_CB3 ? lane * 4u : (lane & 15u) * 8u;
    int32_t out[8];
    if constexpr (Fmt<TYPE>::SLOT) {
        const uint8_t* rowp = blob + static_cast<size_t>(r) * a.row_bytes;
        const uint8_t* codes = rowp + c * Fmt<TYPE>::CHUNK;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            constexpr int qb = TYPE == MOE_CB3X ? 16 : 8;
            uint32_t q[4];
            for (int k = 0; k < qb / 4; ++k) q[k] = ld32(codes + j * qb + 4 * k);
            uint32_t A[1][8];
            float dx[1], aux[1];
            const int slot0[1] = {0};
            load_act<1>(a, smem, c * 8 + j, slot0, A, dx, aux);
            uint32_t W[8];
            slot_decode<TYPE>(q, W);
            out[j] = 2 * dot8(W, A[0]) + __float_as_int(aux[0]);
        }
    } else if constexpr (Fmt<TYPE>::CB) {
        CBRow<TYPE> row;
        row.load(chunk);
        auto one = [&](auto jc) {
            constexpr int j = decltype(jc)::value;
            uint32_t A[1][8];
            float dx[1], aux[1];
            const int slot0[1] = {0};
            load_act<1>(a, smem, c * 8 + j, slot0, A, dx, aux);
            uint32_t W[8];
            cb_decode<TYPE, j>(row, smem, loff, W);
            int d = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[0][w], d);
            out[j] = 2 * d + __float_as_int(aux[0]);
        };
        one(std::integral_constant<int, 0>{}); one(std::integral_constant<int, 1>{});
        one(std::integral_constant<int, 2>{}); one(std::integral_constant<int, 3>{});
        one(std::integral_constant<int, 4>{}); one(std::integral_constant<int, 5>{});
        one(std::integral_constant<int, 6>{}); one(std::integral_constant<int, 7>{});
    } else {
        uint32_t raw[36];
        if constexpr (TYPE == MOE_NL4) {
#pragma unroll
            for (int k = 0; k < 36; ++k) raw[k] = ld32(chunk + 4 * k);
        }
        auto one = [&](auto jc) {
            constexpr int j = decltype(jc)::value;
            uint32_t A[1][8];
            float dx[1], aux[1];
            const int slot0[1] = {0};
            load_act<1>(a, smem, c * 8 + j, slot0, A, dx, aux);
            uint32_t W[8];
            float dw, mw;
            if constexpr (TYPE == MOE_NL4) nl4_decode<j>(raw, tab, W, dw);
            else blk_decode_smem<TYPE, j>(chunk, W, dw, mw);
            int d = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) d = dp4a(W[w], A[0][w], d);
            if constexpr (TYPE == MOE_NL4) {
                // the single-entry decode must give the same sum (else a value no sum takes)
                uint32_t W1[8], W2[8];
                nl4_decode2<j>(raw, tab, W1, W2, dw);
                int d2 = __float_as_int(aux[0]);
#pragma unroll
                for (int w = 0; w < 8; ++w) d2 = dp4a(W2[w], A[0][w], dp4a(W1[w], A[0][w], d2));
                if (d2 != d) d = INT_MIN;
            }
            out[j] = d;
        };
        one(std::integral_constant<int, 0>{}); one(std::integral_constant<int, 1>{});
        one(std::integral_constant<int, 2>{}); one(std::integral_constant<int, 3>{});
        one(std::integral_constant<int, 4>{}); one(std::integral_constant<int, 5>{});
        one(std::integral_constant<int, 6>{}); one(std::integral_constant<int, 7>{});
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) isum[static_cast<size_t>(r) * a.nb + c * 8 + j] = out[j];
}

// ---------------------------------------------------------------- per-format entry points

template <int TYPE>
cudaError_t launch_gemv_t(const GemvArgs& args, int grid, int NT, int smem, cudaStream_t s, bool pdl) {
    GemvArgs a = args;
    a.alpha = Fmt<TYPE>::ALPHA;
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
    a.row_bytes = static_cast<int>(a.nch * (Fmt<TYPE>::CHUNK + (Fmt<TYPE>::SLOT ? 8 : 0)));
    a.codebook = codebook;
    a.act = xq;
    a.n_act_rows = 1;
    a.out_rows = 1;
    int off = Fmt<TYPE>::CB ? 32768 : 0;  // codebook at offset 0
    a.off_actq = off;
    off += 2 * a.nbp * 16;
    a.off_act2 = off;
    off += a.nb * 8;
    a.off_misc = off;
    off += 128;
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
