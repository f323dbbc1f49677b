// q8_1.cuh - the device q8_1 block quantizer and the fp32 SwiGLU it is fused with.
//
// One warp quantizes one block of 32 values, lane i holding value i:
//   amax = max |x_i| (exact), d = amax / 127 (IEEE divide), q_i = round-half-away(x_i / d)
//   (q = 0 when d == 0), S = sum q_i (exact int), stored d16 = fp16_rn(d), s16 = fp16_rn(d * S).
// The same body serves the activation quantizer and the fused SwiGLU + q8_1 kernel, as in
// #363 "experts: smaller and fewer launches for the verify window's PCIe call", "What changes"
// ("the quantizer body ... factored out into a device function").
// Explicit _rn intrinsics keep every rounding where it is written (no contraction, no FTZ).
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

// e^x in fp32 by Cody-Waite range reduction (W. J. Cody, W. Waite, "Software Manual for the
// Elementary Functions", 1980) and a degree-7 Taylor polynomial:
//   k = nearest integer to x*log2(e);  r = (x - k*ln2_hi) - k*ln2_lo,  |r| <= ln2/2,
//   with ln2_hi = 45426/65536 (16 significant bits, so k*ln2_hi is exact for |k| < 256) and
//   ln2_lo = fp32(ln2 - ln2_hi);  e^r = 1 + r + r^2/2! + ... + r^7/7! by Horner (truncation
//   below 1e-8 relative);  e^x = (e^r * 2^k1) * 2^k2 with k1 = k/2 (exact), k2 = k - k1.
// Above 88.76 the result is +inf, below -104 it is 0 (under half the least subnormal).
__device__ __forceinline__ float pow2_int(int n) {  // 2^n, -126 <= n <= 127
    return __int_as_float((n + 127) << 23);
}

__device__ __forceinline__ float exp_cw(float x) {
    if (x != x) return x;
    if (x > 88.76f) return __int_as_float(0x7f800000);
    if (x < -104.0f) return 0.0f;
    const float kLog2e = (float)1.4426950408889634;
    const float kLn2Hi = 0.693145751953125f;
    const float kLn2Lo = (float)(0.6931471805599453 - 0.693145751953125);
    const float k = rintf(__fmul_rn(x, kLog2e));
    const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(k, kLn2Hi)), __fmul_rn(k, kLn2Lo));
    float p = (float)(1.0 / 5040.0);
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 720.0));
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 120.0));
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 24.0));
    p = __fadd_rn(__fmul_rn(p, r), (float)(1.0 / 6.0));
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const int ki = static_cast<int>(k), k1 = ki / 2, k2 = ki - k1;
    return __fmul_rn(__fmul_rn(p, pow2_int(k1)), pow2_int(k2));
}

// silu(g) = g / (1 + e^-g); h = fp32(silu(g) * u), the product rounded on its own.
__device__ __forceinline__ float swiglu_rn(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g)));
    return __fmul_rn(s, u);
}

// The q8_1 block of the warp's 32 values (lane i holds v): returns the lane's code; every lane
// receives the header word d16 | s16 << 16 and the exact code sum S.
__device__ __forceinline__ int warp_q8_1_code(float v, uint32_t& hdr, int& S) {
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const int q = d == 0.0f ? 0 : static_cast<int>(roundf(__fdiv_rn(v, d)));
    S = q;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    const uint32_t d16 = __half_as_ushort(__float2half_rn(d));
    const uint32_t s16 = __half_as_ushort(__float2half_rn(__fmul_rn(d, static_cast<float>(S))));
    hdr = d16 | (s16 << 16);
    return q;
}

// Quantize the warp's 32 values (lane i holds v) into one q8_1 block at dst.
__device__ __forceinline__ void warp_q8_1(float v, moe_q8_1* dst, int lane) {
    uint32_t hdr;
    int S;
    const int q = warp_q8_1_code(v, hdr, S);
    dst->q[lane] = static_cast<int8_t>(q);
    if (lane == 0) *reinterpret_cast<uint32_t*>(dst) = hdr;
}

}  // namespace moe
