/* oracle.c - plain, slow CPU oracle for the grouped routed-expert decode.
 *
 * TEST INFRASTRUCTURE, NOT THE PRODUCT: only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg use it. It shares nothing with the CUDA path. Build it with
 * -ffp-contract=off (no fused multiply-add) and without fast-math.
 *
 * What it follows (see oracle.h for the byte layouts, which are this project's own):
 *  - #2058 "Verify window: the routed experts' gate/up with the group's q8_1 rows in shared
 *    memory", "Why": a group's gate/up weights are decoded once and applied to each of the
 *    group's 1-4 q8_1 entries; "Bit for bit": entries of a group are independent.
 *  - #363 "experts: smaller and fewer launches for the verify window's PCIe call", "What
 *    changes": SwiGLU and the q8_1 quantization run over the call's own entries
 *    [grp_start[0], grp_start[n_groups]); the SwiGLU product is rounded to fp32 on its own
 *    before the q8_1 block sums; "Exactness": a second call's entries start past 0 and its
 *    destinations are scattered.
 * Readings where the pages are silent (each one is listed with its reason in the design
 * notes): q8_1 is d = amax/127 (fp32 divide), q = round-half-away(x/d), s = fp16(d * sum q);
 * the block contributions below; exp by Cody-Waite reduction and a Taylor polynomial;
 * groups ordered by ascending expert id, entries by ascending (t, slot).
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against something
 * other than itself (numpy's binary16 conversion, fp64 exp, brute-force fp64 dot products of
 * dequantized operands, hand-built blocks with known weights, closed forms, invariants),
 * and tests/test_oracle_mutants.py rebuilds it with planted mistakes (ORC_PLANT_*) to show
 * the pins catch them.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ binary16 */

float orc_h2f(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24); /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25); /* (1 + man/1024) * 2^(ex-15) */
    return (float)(sign ? -v : v);
}

uint16_t orc_f2h(float f) {
    double x = f;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return sign | 0x7e00;
    double a = fabs(x);
    if (a >= 65520.0) return sign | 0x7c00; /* halfway to 2^16 and above round to inf */
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1; /* 2^ex <= a < 2^(ex+1) */
    double quantum = ex < -14 ? ldexp(1.0, -24) : ldexp(1.0, ex - 10);
    double r = rint(a / quantum); /* exact scaling, then nearest integer, ties to even */
    double v = r * quantum;
    if (v < ldexp(1.0, -14)) return sign | (uint16_t)r; /* subnormal */
    frexp(v, &e);
    ex = e - 1;
    uint32_t man = (uint32_t)(v / ldexp(1.0, ex - 10)) - 1024;
    return sign | (uint16_t)(((ex + 15) << 10) | man);
}

/* ------------------------------------------------------------------ exp, SwiGLU */

/* e^x in fp32 by Cody and Waite's range reduction (W. J. Cody, W. Waite, "Software Manual
 * for the Elementary Functions", 1980): x = k*ln2 + r with k = nearest integer to x*log2(e)
 * and ln2 split into a 16-significant-bit high part (so k*ln2_hi is exact for |k| <= 256)
 * and the fp32 remainder; then e^r by its Taylor series 1 + r + r^2/2! + ... + r^7/7!
 * (Horner), whose truncation error for |r| <= ln2/2 is below 1e-8 relative; then the exact
 * scaling by 2^k, split in two factors so that only the final product can round. */
static float pow2i(int n) { /* 2^n for -126 <= n <= 127 */
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)(n + 127) << 23;
    return c.f;
}

float orc_expf(float x) {
    const float log2e = (float)1.4426950408889634;    /* log2(e) */
    const float ln2_hi = 0.693145751953125f;          /* 45426 * 2^-16 */
    const float ln2_lo = (float)(0.6931471805599453 - 0.693145751953125);
    if (x != x) return x;
    if (x > 88.76f) return INFINITY; /* e^88.76 > FLT_MAX */
    if (x < -104.0f) return 0.0f;    /* e^-104 is below half the smallest subnormal */
    float k = rintf(x * log2e);
    float r = (x - k * ln2_hi) - k * ln2_lo;
    float p = (float)(1.0 / 5040.0);
    p = p * r + (float)(1.0 / 720.0);
    p = p * r + (float)(1.0 / 120.0);
    p = p * r + (float)(1.0 / 24.0);
#ifndef ORC_PLANT_EXP_TERM
    p = p * r + (float)(1.0 / 6.0);
#else
    p = p * r + (float)(1.0 / 5.0);
#endif
    p = p * r + 0.5f;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    int ki = (int)k, k1 = ki / 2, k2 = ki - k1;
    return (p * pow2i(k1)) * pow2i(k2);
}

float orc_silu(float g) { return g / (1.0f + orc_expf(-g)); }

/* #363 "What changes": the product is rounded on its own (one fp32 multiply). */
float orc_swiglu(float g, float u) { return orc_silu(g) * u; }

/* ------------------------------------------------------------------ q8_1 */

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }

static void q8_1_block(const float* x, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    int S = 0;
    for (int i = 0; i < 32; i++) {
        int q = 0;
        if (d != 0.0f) {
#ifndef ORC_PLANT_ROUND_EVEN
            q = (int)roundf(x[i] / d); /* nearest, halfway cases away from zero */
#else
            q = (int)rintf(x[i] / d);
#endif
        }
        out[4 + i] = (uint8_t)(int8_t)q;
        S += q;
    }
    uint16_t d16 = orc_f2h(d);
#ifndef ORC_PLANT_S_FROM_D16
    uint16_t s16 = orc_f2h(d * (float)S);
#else
    uint16_t s16 = orc_f2h(orc_h2f(d16) * (float)S);
#endif
    wr16(out, d16);
    wr16(out + 2, s16);
}

void orc_quantize_q8_1(const float* x, int64_t n, uint8_t* out) {
    for (int64_t b = 0; b < n / 32; b++) q8_1_block(x + 32 * b, out + 36 * b);
}

/* ------------------------------------------------------------------ weight formats */

int64_t orc_row_bytes(int type, int K) {
    if (K <= 0 || K % 32) return 0;
    switch (type) {
    case ORC_Q8_0: return (int64_t)(K / 32) * 34;
    case ORC_Q4B: return (int64_t)(K / 32) * 20;
    case ORC_NL4: return (int64_t)(K / 32) * 18;
    case ORC_CB2: return K % 256 ? 0 : (int64_t)(K / 256) * 70;
    case ORC_CB3: return K % 256 ? 0 : (int64_t)(K / 256) * 102;
    case ORC_CB3X: return K % 256 ? 0 : (int64_t)(K / 256) * (128 + 8);
    case ORC_CB2X: return K % 256 ? 0 : (int64_t)(K / 256) * (64 + 8);
    }
    return 0;
}

/* ---- transcoded slots: codes of the K weights, then one 8-byte scale record per 256 weights */

static int slot_bits(int type) { return type == ORC_CB3X ? 4 : 2; }
static int slot_bias(int type) { return type == ORC_CB3X ? 8 : 2; }

/* Code u of weight n of a slot row. */
static int slot_code(int type, const uint8_t* row, int n) {
    int c = n / 256, j = (n % 256) / 32, i = n % 32;
    if (type == ORC_CB3X) {
        const uint8_t* sb = row + c * 128 + j * 16;
#ifndef ORC_PLANT_SLOT_ORDER
        return i < 16 ? (sb[i] & 15) : (sb[i - 16] >> 4);
#else
        return (sb[i / 2] >> (4 * (i & 1))) & 15;
#endif
    }
    const uint8_t* sb = row + c * 64 + j * 8;
    return (sb[i % 8] >> (2 * (i / 8))) & 3;
}

static const uint8_t* slot_scale(int type, const uint8_t* row, int K, int n) {
    int code_bytes = type == ORC_CB3X ? 128 : 64;
    return row + (K / 256) * code_bytes + (n / 256) * 8;
}

/* 4-bit code j (0..31) of a 16-byte nibble array. */
static int nib_code(const uint8_t* qs, int j) {
#ifndef ORC_PLANT_NIBBLE_ORDER
    return j < 16 ? (qs[j] & 15) : (qs[j - 16] >> 4);
#else
    return (qs[j / 2] >> (4 * (j & 1))) & 15;
#endif
}

/* Sub-scale multiplier ls_j = 2*sub_j + 1 of 32-weight sub-block j of a CB super-block. */
static int cb_ls(const uint8_t* sub, int j) {
#ifndef ORC_PLANT_SUB_NIBBLE
    int s = (sub[j >> 1] >> (4 * (j & 1))) & 15;
#else
    int s = (sub[j >> 1] >> (4 * (1 - (j & 1)))) & 15;
#endif
#ifndef ORC_PLANT_LS
    return 2 * s + 1;
#else
    return s;
#endif
}

static int sign_bit(uint8_t s, int p) {
#ifndef ORC_PLANT_SIGN_ORDER
    return (s >> p) & 1;
#else
    return (s >> (7 - p)) & 1;
#endif
}

/* Signed grid value of weight n (0..255) of a CB super-block starting at sb. */
static int cb_value(int type, const uint8_t* sb, const int8_t* cb, int n) {
    int g, neg;
    if (type == ORC_CB2) {
        const uint8_t *idx = sb + 2, *sign = sb + 34;
        g = cb[idx[n / 8] * 8 + n % 8];
        neg = sign_bit(sign[n / 8], n % 8);
    } else {
        const uint8_t *idx = sb + 2, *sign = sb + 66;
        g = cb[idx[n / 4] * 4 + n % 4];
        neg = sign_bit(sign[n / 8], n % 8);
    }
    return neg ? -g : g;
}

static const uint8_t* cb_sub(int type, const uint8_t* sb) { return sb + (type == ORC_CB2 ? 66 : 98); }

void orc_int_weights(int type, const uint8_t* row, int K, const int8_t* cb, int32_t* v) {
    for (int n = 0; n < K; n++) {
        int b = n / 32, i = n % 32;
        switch (type) {
        case ORC_Q8_0: v[n] = (int8_t)row[34 * b + 2 + i]; break;
        case ORC_Q4B: v[n] = nib_code(row + 20 * b + 4, i); break;
        case ORC_NL4: v[n] = cb[nib_code(row + 18 * b + 2, i)]; break;
        case ORC_CB2: v[n] = cb_value(type, row + 70 * (n / 256), cb, n % 256); break;
        case ORC_CB3: v[n] = cb_value(type, row + 102 * (n / 256), cb, n % 256); break;
        case ORC_CB3X:
        case ORC_CB2X: v[n] = 2 * (slot_code(type, row, n) - slot_bias(type)) + 1; break;
        }
    }
}

void orc_dequant_row(int type, const uint8_t* row, int K, const int8_t* cb, double* w) {
    int32_t* v = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    orc_int_weights(type, row, K, cb, v);
    for (int n = 0; n < K; n++) {
        int b = n / 32;
        switch (type) {
        case ORC_Q8_0: w[n] = (double)orc_h2f(rd16(row + 34 * b)) * v[n]; break;
        case ORC_Q4B:
            w[n] = (double)orc_h2f(rd16(row + 20 * b)) * v[n] + (double)orc_h2f(rd16(row + 20 * b + 2));
            break;
        case ORC_NL4: w[n] = (double)orc_h2f(rd16(row + 18 * b)) * v[n]; break;
        case ORC_CB2:
        case ORC_CB3: {
            const uint8_t* sb = row + (type == ORC_CB2 ? 70 : 102) * (n / 256);
            w[n] = (double)orc_h2f(rd16(sb)) * cb_ls(cb_sub(type, sb), (n % 256) / 32) * v[n];
            break;
        }
        case ORC_CB3X:
        case ORC_CB2X: {
            const uint8_t* sc = slot_scale(type, row, K, n);
            w[n] = (double)orc_h2f(rd16(sc)) * cb_ls(sc + 4, (n % 256) / 32) * v[n];
            break;
        }
        }
    }
    free(v);
}

void orc_block_isum(int type, const uint8_t* row, int K, const int8_t* cb, const uint8_t* xq,
                    int32_t* isum) {
    int32_t* v = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    orc_int_weights(type, row, K, cb, v);
    for (int b = 0; b < K / 32; b++) {
        int32_t s = 0;
        for (int i = 0; i < 32; i++) s += v[32 * b + i] * (int32_t)(int8_t)xq[36 * b + 4 + i];
        isum[b] = s;
    }
    free(v);
}

/* Block contribution c_b of weight block b against q8_1 block b, summed over b in fp64:
 *   Q8_0, NL4 : c = d_w * d_x * isum
 *   Q4B       : c = d_w * d_x * isum + m_w * s_x   (q8_1 carries s = d * sum q for this term)
 *   CB2, CB3  : c = D * d_x * (ls_j * isum_j)      (per 32-weight sub-block j) */
double orc_row_dot(int type, const uint8_t* row, int K, const int8_t* cb, const uint8_t* xq) {
    int nb = K / 32;
    int32_t* isum = (int32_t*)malloc(sizeof(int32_t) * (size_t)nb);
    orc_block_isum(type, row, K, cb, xq, isum);
    double acc = 0.0;
    for (int b = 0; b < nb; b++) {
        double dx = orc_h2f(rd16(xq + 36 * b)), sx = orc_h2f(rd16(xq + 36 * b + 2));
        switch (type) {
        case ORC_Q8_0: acc += (double)orc_h2f(rd16(row + 34 * b)) * dx * isum[b]; break;
        case ORC_NL4: acc += (double)orc_h2f(rd16(row + 18 * b)) * dx * isum[b]; break;
        case ORC_Q4B:
            acc += (double)orc_h2f(rd16(row + 20 * b)) * dx * isum[b];
#ifndef ORC_PLANT_Q4B_MIN
            acc += (double)orc_h2f(rd16(row + 20 * b + 2)) * sx;
#endif
            break;
        case ORC_CB2:
        case ORC_CB3: {
            const uint8_t* sb = row + (type == ORC_CB2 ? 70 : 102) * (b / 8);
            acc += (double)orc_h2f(rd16(sb)) * dx * ((double)cb_ls(cb_sub(type, sb), b % 8) * isum[b]);
            break;
        }
        case ORC_CB3X:
        case ORC_CB2X: {
            const uint8_t* sc = slot_scale(type, row, K, 32 * b);
            acc += (double)orc_h2f(rd16(sc)) * dx * ((double)cb_ls(sc + 4, b % 8) * isum[b]);
            break;
        }
        }
    }
    free(isum);
    return acc;
}

int orc_transcode_row(int src_type, const uint8_t* src, int K, const int8_t* cb, int dst_type, uint8_t* dst) {
    int bits = slot_bits(dst_type), bias = slot_bias(dst_type), lim = (1 << bits) - 1, bad = 0;
    int code_bytes = dst_type == ORC_CB3X ? 128 : 64;
    int32_t* v = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    orc_int_weights(src_type, src, K, cb, v);
    memset(dst, 0, (size_t)orc_row_bytes(dst_type, K));
    for (int n = 0; n < K; n++) {
        int u = (v[n] - 1) / 2 + bias; /* v odd: exact */
        if ((v[n] & 1) == 0 || u < 0 || u > lim) { bad = -1; u = 0; }
        int c = n / 256, j = (n % 256) / 32, i = n % 32;
        if (dst_type == ORC_CB3X) {
            uint8_t* sb = dst + c * 128 + j * 16;
            if (i < 16) sb[i] |= (uint8_t)u;
            else sb[i - 16] |= (uint8_t)(u << 4);
        } else {
            uint8_t* sb = dst + c * 64 + j * 8;
            sb[i % 8] |= (uint8_t)(u << (2 * (i / 8)));
        }
    }
    for (int c = 0; c < K / 256; c++) {
        const uint8_t* sb = src + (src_type == ORC_CB2 ? 70 : 102) * c;
        uint8_t* sc = dst + (K / 256) * code_bytes + 8 * c;
        sc[0] = sb[0];
        sc[1] = sb[1];
        memcpy(sc + 4, cb_sub(src_type, sb), 4);
    }
    free(v);
    return bad;
}

/* ------------------------------------------------------------------ grouped steps */

int orc_grouped_gemv(int type, const int8_t* cb, int K, int rows, const uint8_t* const* w,
                     int n_experts, const int32_t* grp_expert, const int32_t* grp_start,
                     int n_groups, const uint8_t* act, const int32_t* ent_in,
                     const int32_t* ent_out, double* out, int64_t out_stride) {
    int64_t rb = orc_row_bytes(type, K), ab = (int64_t)(K / 32) * 36;
    int bad = 0;
    for (int g = 0; g < n_groups; g++) {
        int x = grp_expert[g];
        if (x < 0 || x >= n_experts) { bad = -1; continue; }
        for (int e = grp_start[g]; e < grp_start[g + 1]; e++) {
#ifndef ORC_PLANT_ENTRY_ROW
            int in = ent_in ? ent_in[e] : e;
#else
            int in = e;
#endif
            int o = ent_out ? ent_out[e] : e;
            for (int r = 0; r < rows; r++)
                out[(int64_t)o * out_stride + r] = orc_row_dot(type, w[x] + (int64_t)r * rb, K, cb, act + (int64_t)in * ab);
        }
    }
    return bad;
}

void orc_swiglu_q8_1(const float* gu, int F, int e0, int e1, uint8_t* hq) {
    float* h = (float*)malloc(sizeof(float) * (size_t)F);
    for (int e = e0; e < e1; e++) {
        const float* row = gu + (int64_t)e * 2 * F;
        for (int j = 0; j < F; j++) h[j] = orc_swiglu(row[j], row[F + j]);
        orc_quantize_q8_1(h, F, hq + (int64_t)e * (F / 32) * 36);
    }
    free(h);
}

int orc_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base,
                    int32_t* grp_expert, int32_t* grp_start, int32_t* n_groups,
                    int32_t* ent_src, int32_t* ent_dst) {
    int n = T * k, m = 0, dropped = 0;
    int* key = (int*)malloc(sizeof(int) * (size_t)(n + 1));
    int* pos = (int*)malloc(sizeof(int) * (size_t)(n + 1));
    /* entries in (t, slot) order, then a stable insertion sort by expert id */
    for (int t = 0; t < T; t++)
        for (int s = 0; s < k; s++) {
            int x = topk_ids[t * k + s];
            if (x < 0 || x >= n_experts) { dropped++; continue; }
            key[m] = x;
#ifndef ORC_PLANT_ROUTE_ORDER
            pos[m] = t * k + s;
#else
            pos[m] = s * T + t;
#endif
            m++;
        }
    for (int i = 1; i < m; i++) {
        int kx = key[i], px = pos[i], j = i - 1;
        while (j >= 0 && (key[j] > kx || (key[j] == kx && pos[j] > px))) {
            key[j + 1] = key[j]; pos[j + 1] = pos[j]; j--;
        }
        key[j + 1] = kx; pos[j + 1] = px;
    }
    int G = 0;
    for (int i = 0; i < m; i++) {
        int e = entry_base + i;
        if (i == 0 || key[i] != key[i - 1]) {
            grp_expert[G] = key[i];
            grp_start[G] = e;
            G++;
        }
#ifndef ORC_PLANT_ROUTE_ORDER
        ent_src[e] = pos[i] / k;
        ent_dst[e] = pos[i];
#else
        ent_src[e] = pos[i] % T;
        ent_dst[e] = (pos[i] % T) * k + pos[i] / T;
#endif
    }
    grp_start[G] = entry_base + m;
    *n_groups = G;
    free(key);
    free(pos);
    return dropped;
}

/* ------------------------------------------------------------------ router and combine */

/* The k largest logits by repeated selection: a logit ranks above another when it is larger,
 * or equal with the lower expert id. */
int orc_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, double* weights) {
    if (k <= 0 || k > E || T < 0) return -1;
    char* taken = (char*)calloc((size_t)E, 1);
    if (!taken) return -1;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
#ifdef ORC_PLANT_TIE_HIGH
                if (best < 0 || l[e] >= l[best]) best = e;
#else
                if (best < 0 || l[e] > l[best]) best = e;
#endif
            }
            taken[best] = 1;
            topk_ids[(int64_t)t * k + j] = best;
        }
        double sum = 0.0;
#ifdef ORC_PLANT_SOFTMAX_ALL
        for (int e = 0; e < E; ++e) sum += exp((double)l[e]);
#else
        for (int j = 0; j < k; ++j) sum += exp((double)l[topk_ids[(int64_t)t * k + j]]);
#endif
        for (int j = 0; j < k; ++j) weights[(int64_t)t * k + j] = exp((double)l[topk_ids[(int64_t)t * k + j]]) / sum;
    }
    free(taken);
    return 0;
}

void orc_combine(const float* out, int64_t out_stride, const int32_t* topk_ids, const double* weights, int T,
                 int k, int E, int n_embd, double* y) {
    for (int t = 0; t < T; ++t) {
        for (int n = 0; n < n_embd; ++n) {
            double acc = 0.0;
#ifdef ORC_PLANT_COMBINE_SLOT
            for (int j = 0; j + 1 < k; ++j) {
#else
            for (int j = 0; j < k; ++j) {
#endif
                const int x = topk_ids[(int64_t)t * k + j];
                if (x < 0 || x >= E) continue;
                acc += weights[(int64_t)t * k + j] * (double)out[((int64_t)t * k + j) * out_stride + n];
            }
            y[(int64_t)t * n_embd + n] = acc;
        }
    }
}

/* ------------------------------------------------------------------ QSA decode block scores */

/* #2059 "QSA decode: the window's block scores with the queries in registers and six shuffles
 * per block", "What changed" and "Bit for bit": the queries' head slices sit 4 floats per lane
 * of a warp, a head's lane products are reduced with the warp sum's pairings (xor 16, 8, 4, 2,
 * 1), the relus of the heads are summed in head order, and the tail block gets +1e9. The
 * arithmetic is fp32 (this file is built without contraction: fmaf below is the one fused step,
 * named on purpose). */
static float qsa_lane_partial(const float* qh, const int8_t* kb, int lane) {
#ifdef ORC_PLANT_QSA_LANE_INTERLEAVE
    const int d[4] = {lane, lane + 32, lane + 64, lane + 96};
#else
    const int d[4] = {4 * lane, 4 * lane + 1, 4 * lane + 2, 4 * lane + 3};
#endif
#ifdef ORC_PLANT_QSA_NO_FMA
    float p = qh[d[0]] * (float)kb[d[0]];
    for (int i = 1; i < 4; ++i) p = p + qh[d[i]] * (float)kb[d[i]];
#else
    float p = qh[d[0]] * (float)kb[d[0]];
    for (int i = 1; i < 4; ++i) p = fmaf(qh[d[i]], (float)kb[d[i]], p);
#endif
    return p;
}

static float qsa_head_dot(const float* qh, const int8_t* kb) {
    float v[ORC_QSA_LANES];
    for (int l = 0; l < ORC_QSA_LANES; ++l) v[l] = qsa_lane_partial(qh, kb, l);
#ifdef ORC_PLANT_QSA_TREE_SEQ
    float s = v[0];
    for (int l = 1; l < ORC_QSA_LANES; ++l) s = s + v[l];
    return s;
#else
    /* level j replaces every lane's value by its own plus lane (l xor j)'s; after level 1 every
     * lane holds the same sum */
    for (int j = ORC_QSA_LANES / 2; j >= 1; j /= 2) {
        float w[ORC_QSA_LANES];
        for (int l = 0; l < ORC_QSA_LANES; ++l) w[l] = v[l] + v[l ^ j];
        memcpy(v, w, sizeof v);
    }
    return v[0];
#endif
}

void orc_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* scale, int64_t n_blocks,
                          float* scores) {
    for (int t = 0; t < T; ++t) {
        for (int64_t b = 0; b < n_blocks; ++b) {
            const int8_t* kb = keys + b * ORC_QSA_DIM;
            float r[ORC_QSA_HEADS];
            for (int h = 0; h < ORC_QSA_HEADS; ++h) {
                const float s = qsa_head_dot(q + ((int64_t)t * ORC_QSA_HEADS + h) * ORC_QSA_DIM, kb) * scale[b];
                r[h] = s > 0.0f ? s : 0.0f;
            }
#ifdef ORC_PLANT_QSA_HEAD_ORDER
            float sc = ((r[3] + r[2]) + r[1]) + r[0];
#else
            float sc = ((r[0] + r[1]) + r[2]) + r[3];
#endif
#ifdef ORC_PLANT_QSA_TAIL_FIRST
            if (b == 0) sc = sc + 1e9f;
#else
            if (b == n_blocks - 1) sc = sc + 1e9f;
#endif
            scores[(int64_t)t * n_blocks + b] = sc;
        }
    }
}
