// qsa.cu - QSA decode block scores for a verify window of T <= 4 queries.
//
// What it computes (#2059 "QSA decode: the window's block scores with the queries in registers
// and six shuffles per block", "What changed" and "Bit for bit"): for each query t (4 heads of
// 128 fp32 values) and each key block b (one pooled key of 128 int8 codes, fp32 scale):
//   lane l of a warp owns the slice 4l..4l+3 of every head: p_l = q0*k0, then three fused
//   multiply-adds for the slice's next dims; a head's 32 lane partials are summed with the warp
//   sum's pairings (level j = 16, 8, 4, 2, 1 adds lane l's value and lane (l xor j)'s);
//   r_h = max(dot_h * scale_b, 0); score = ((r_0 + r_1) + r_2) + r_3, and +1e9 on the tail
//   block (the last one). Every operation is one fp32 rounding, in that order, so the scores
//   are the same bits as the CPU oracle's.
//
// How (GB300 design, not the page's kernel):
//  * A warp takes a chunk of NB key blocks (NB * T' * 4 = 64 values, T' = T rounded up to 1, 2
//    or 4) and reads each block's 128 bytes once for all queries: a 4-byte asynchronous copy
//    (cp.async) per lane per block into the warp's ring of shared-memory stages, issued 4 KB of
//    keys ahead of the arithmetic so that DRAM latency is hidden (a lane reads back only the
//    words it copied itself, so waiting for its own copies is enough). The queries' slices stay in registers for the whole kernel, as head pairs
//    (q_h, q_h+1) so that one packed fp32x2 fused multiply-add (fma.rn.f32x2) computes two
//    heads' products per instruction; the key value is converted exactly (a byte permute into
//    2^23 + (k + 128), then one subtraction) and used in both halves.
//  * The pairings need every lane's partial of a value. The first level (lane l with lane l xor
//    16) is one shuffle exchange: lanes 16-31 take the chunk's blocks in swapped halves, so the
//    first half of every lane's steps gives the values it keeps and the second half the ones its
//    partner keeps, sent over and added (the same two operands as the definition's, and fp32
//    addition commutes). Each lane then writes its 16 kept pair sums into a padded shared-memory
//    tile (row = value pair, column = lane mod 16; 144-byte rows keep the 8-byte writes and the
//    16-byte reads free of bank conflicts), and lane j reads row j and adds it up in the pairing
//    order (levels 8, 4, 2, 1) with packed fp32x2 additions. Packed arithmetic rounds each half
//    on its own, so nothing changes in the bits.
//  * The lanes holding heads 0-1 and 2-3 of one (block, query) meet with two shuffles for the
//    head-order sum; the score is stored by the even lane.
//  * Bound: instruction issue and the fp32 pipe at T = 3-4 (about 100 warp-instructions per block:
//    32 packed multiply-adds, the key conversion, the exchange, 4 shared-memory writes and the
//    reduction), not HBM (132 bytes per block).
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kQsaWarps = 4;          // warps per CTA (a 4.6 KB tile each)
constexpr int kQsaRow = 18;           // float2 per shared-memory row (16 lane pairs + 16 bytes of padding)
constexpr int kQsaRows = 32;          // value pairs per chunk
constexpr float kQsaTail = 1e9f;      // added to the tail block's score
constexpr float kByteBias = 8388736.0f;  // 2^23 + 128

__device__ __forceinline__ unsigned long long pk(float2 v) {
    return (static_cast<unsigned long long>(__float_as_uint(v.y)) << 32) | __float_as_uint(v.x);
}
__device__ __forceinline__ float2 upk(unsigned long long v) {
    return make_float2(__uint_as_float(static_cast<uint32_t>(v)), __uint_as_float(static_cast<uint32_t>(v >> 32)));
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d = pk(c);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(pk(a)), "l"(pk(b)));
    return upk(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
    return upk(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a)), "l"(pk(b)));
    return upk(d);
}

// Byte i of w (an int8 code, w already xor 0x80808080) as an exact fp32, in both halves.
template <int i>
__device__ __forceinline__ float2 key2(uint32_t wx) {
    const float f = __uint_as_float(prmt(wx, 0x4B000000u, 0x7440u + i));  // 2^23 + k + 128
    return add2(make_float2(f, f), make_float2(-kByteBias, -kByteBias));
}

// Asynchronous 4-byte copy global -> shared (cp.async; src_bytes 0 fills zeros without reading).
__device__ __forceinline__ void cp4(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Chunks of key blocks per stage ring of each warp: D stages of NB blocks (4 KB of keys).
template <int TQ>
struct QsaGeom {
    static constexpr int NB = 16 / TQ;    // key blocks per chunk (64 values = 32 pairs)
    static constexpr int D = 32 / NB;     // chunks in flight per warp
    static constexpr int kTile = kQsaRows * kQsaRow * 8;        // reduction tile bytes
    static constexpr int kKeys = D * NB * 128;                  // key ring bytes
    static constexpr int kScale = D * 16 * 4;                   // scale ring bytes (NB <= 16 per stage)
    static constexpr int kWarp = kTile + kKeys + kScale;
};

// The lane's copies of chunk ch into stage st: word `lane` of each of the chunk's blocks, and
// (lanes < NB) the blocks' scales; blocks past the end are zero-filled without a read.
template <int TQ>
__device__ __forceinline__ void issue_chunk(uint8_t* ring, float* sring, const int8_t* keys, const float* scale,
                                            long long n_blocks, long long ch, int st, int lane) {
    constexpr int NB = QsaGeom<TQ>::NB;
    const long long b0 = ch * NB;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const bool in = b0 + b < n_blocks;
        cp4(ring + (st * NB + b) * 128 + 4 * lane, keys + (in ? (b0 + b) * 128 + 4 * lane : 0), in ? 4u : 0u);
    }
    if (lane < NB) {
        const bool in = b0 + lane < n_blocks;
        cp4(sring + st * 16 + lane, scale + (in ? b0 + lane : 0), in ? 4u : 0u);
    }
}

// TQ: queries held (1, 2 or 4; the T actual ones first, the rest zero and never stored).
template <int TQ>
__global__ void __launch_bounds__(kQsaWarps * 32) qsa_kernel(const float* __restrict__ q, int T,
                                                             const int8_t* __restrict__ keys,
                                                             const float* __restrict__ scale, long long n_blocks,
                                                             float* __restrict__ scores) {
    using G = QsaGeom<TQ>;
    constexpr int NB = G::NB, D = G::D;
    extern __shared__ __align__(16) uint8_t qsa_smem[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint8_t* wbase = qsa_smem + wid * G::kWarp;
    float2(*tl)[kQsaRow] = reinterpret_cast<float2(*)[kQsaRow]>(wbase);
    uint8_t* ring = wbase + G::kTile;
    float* sring = reinterpret_cast<float*>(wbase + G::kTile + G::kKeys);
    const long long n_chunks = (n_blocks + NB - 1) / NB;
    const long long warps = static_cast<long long>(gridDim.x) * kQsaWarps;
    const long long ch0 = static_cast<long long>(blockIdx.x) * kQsaWarps + wid;
    // D chunks of the warp's sequence in flight before any arithmetic (one commit group each;
    // empty groups past the end keep the count uniform)
#pragma unroll
    for (int i = 0; i < D; ++i) {
        const long long ch = ch0 + i * warps;
        if (ch < n_chunks) issue_chunk<TQ>(ring, sring, keys, scale, n_blocks, ch, i, lane);
        cp_commit();
    }
    // the lane's slices of every query and head pair: qp[t][hp][i] = (q[t][2hp][4l+i], q[t][2hp+1][4l+i])
    float2 qp[TQ][2][4];
#pragma unroll
    for (int t = 0; t < TQ; ++t)
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (t < T) {
                a = __ldg(reinterpret_cast<const float4*>(q + (t * 4 + 2 * hp) * 128) + lane);
                b = __ldg(reinterpret_cast<const float4*>(q + (t * 4 + 2 * hp + 1) * 128) + lane);
            }
            qp[t][hp][0] = make_float2(a.x, b.x);
            qp[t][hp][1] = make_float2(a.y, b.y);
            qp[t][hp][2] = make_float2(a.z, b.z);
            qp[t][hp][3] = make_float2(a.w, b.w);
        }
    // lanes 16-31 take the chunk's blocks in swapped halves (step b: block b xor NB/2)
    const int hb = lane >= 16 ? NB / 2 : 0;
    int st = 0;
    for (long long ch = ch0; ch < n_chunks; ch += warps) {
        const long long b0 = ch * NB;
        cp_wait<D - 1>();  // this lane's copies of chunk ch have landed (it reads only those)
        uint32_t kw[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            kw[b] = *reinterpret_cast<const uint32_t*>(ring + (st * NB + (b ^ hb)) * 128 + 4 * lane);
        // ---- the lane's partials, step b: block b (lanes 0-15) or block b xor NB/2 (lanes 16-31).
        // Pairing level 16 (slice l with slice l xor 16) by one exchange: the first NB/2 steps
        // give the blocks the lane keeps, the last NB/2 the ones its partner keeps, sent to it
        // and added (the same two operands as the definition's; fp32 addition commutes)
        float2 kp[NB / 2][TQ][2];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const uint32_t wx = kw[b] ^ 0x80808080u;
            const float2 k0 = key2<0>(wx), k1 = key2<1>(wx), k2 = key2<2>(wx), k3 = key2<3>(wx);
#pragma unroll
            for (int t = 0; t < TQ; ++t)
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) {
                    float2 p = mul2(qp[t][hp][0], k0);
                    p = fma2(qp[t][hp][1], k1, p);
                    p = fma2(qp[t][hp][2], k2, p);
                    p = fma2(qp[t][hp][3], k3, p);
                    if (b < NB / 2) {
                        kp[b][t][hp] = p;
                    } else {
                        const float2 r = make_float2(__shfl_xor_sync(0xffffffffu, p.x, 16),
                                                     __shfl_xor_sync(0xffffffffu, p.y, 16));
                        kp[b - NB / 2][t][hp] = add2(kp[b - NB / 2][t][hp], r);
                    }
                }
        }
        // the kept sums: pair row (block * TQ + t) * 2 + hp of the lane's blocks, column = lane % 16
#pragma unroll
        for (int b = 0; b < NB / 2; ++b)
#pragma unroll
            for (int t = 0; t < TQ; ++t)
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) tl[((b + hb) * TQ + t) * 2 + hp][lane & 15] = kp[b][t][hp];
        __syncwarp();  // every lane's sums (and scale copies) before the reduction reads them
        // ---- lane j sums pair row j over the 16 columns in the warp sum's order: level 8 adds
        // columns c and c + 8, then 4, 2, 1 on the results
        float2 x[16];
        const float4* row = reinterpret_cast<const float4*>(tl[lane]);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = row[i];
            x[2 * i] = make_float2(v.x, v.y);
            x[2 * i + 1] = make_float2(v.z, v.w);
        }
        // ---- lane j: (block, query) m = j / 2, heads 2(j & 1) and 2(j & 1) + 1
        const int m = lane >> 1, b = m / TQ, t = m - b * TQ;
        const long long blk = b0 + b;
        const float sc = sring[st * 16 + b];
        __syncwarp();  // the tile and the stage are rewritten below / by the next chunk
        // refill this stage with the chunk D steps ahead (an empty group past the end)
        {
            const long long nx = ch + D * warps;
            if (nx < n_chunks) issue_chunk<TQ>(ring, sring, keys, scale, n_blocks, nx, st, lane);
            cp_commit();
        }
        st = st + 1 == D ? 0 : st + 1;
#pragma unroll
        for (int j = 8; j >= 1; j >>= 1)
#pragma unroll
            for (int c = 0; c < j; ++c) x[c] = add2(x[c], x[c + j]);
        const float s0 = __fmul_rn(x[0].x, sc), s1 = __fmul_rn(x[0].y, sc);
        const float r0 = s0 > 0.0f ? s0 : 0.0f, r1 = s1 > 0.0f ? s1 : 0.0f;
        const float r2 = __shfl_down_sync(0xffffffffu, r0, 1), r3 = __shfl_down_sync(0xffffffffu, r1, 1);
        if ((lane & 1) == 0 && t < T && blk < n_blocks) {
            float s = __fadd_rn(__fadd_rn(__fadd_rn(r0, r1), r2), r3);
            if (blk == n_blocks - 1) s = __fadd_rn(s, kQsaTail);
            scores[static_cast<long long>(t) * n_blocks + blk] = s;
        }
    }
    cp_wait<0>();  // no copy outstanding at exit
}

template <int TQ>
cudaError_t launch_qsa_t(const float* q, int T, const int8_t* keys, const float* scale, long long n_blocks,
                         float* scores, cudaStream_t s) {
    using G = QsaGeom<TQ>;
    const long long chunks = (n_blocks + G::NB - 1) / G::NB;
    const int smem = kQsaWarps * G::kWarp;
    // resident CTAs on the whole device: set up once per device (attribute + occupancy query)
    constexpr int kMaxDev = 64;
    static std::atomic<long long> slots[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    long long cap = slots[dev].load(std::memory_order_relaxed);
    if (cap <= 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qsa_kernel<TQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qsa_kernel<TQ>, kQsaWarps * 32, smem);
        if (e != cudaSuccess) return e;
        cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
        slots[dev].store(cap, std::memory_order_relaxed);
    }
    const long long need = (chunks + kQsaWarps - 1) / kQsaWarps;
    const int grid = static_cast<int>(need < cap ? need : cap);
    qsa_kernel<TQ><<<grid, kQsaWarps * 32, smem, s>>>(q, T, keys, scale, n_blocks, scores);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* scale, long long n_blocks,
                                    float* scores, cudaStream_t s) {
    if (T == 1) return launch_qsa_t<1>(q, T, keys, scale, n_blocks, scores, s);
    if (T == 2) return launch_qsa_t<2>(q, T, keys, scale, n_blocks, scores, s);
    return launch_qsa_t<4>(q, T, keys, scale, n_blocks, scores, s);
}

}  // namespace moe
