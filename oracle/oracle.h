/* oracle.h - CPU oracle for the grouped routed-expert decode of the verify window.
 *
 * TEST INFRASTRUCTURE, NOT THE PRODUCT. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. It shares no code, header, table or
 * constant with the CUDA path; both follow the same written format definitions.
 *
 * Sources (web pages of one inference engine):
 *  [P1] #2058 "Verify window: the routed experts' gate/up with the group's q8_1 rows in
 *       shared memory", sections "Why", "What changed", "Bit for bit".
 *  [P2] #363 "experts: smaller and fewer launches for the verify window's PCIe call",
 *       sections "What changes", "Exactness".
 * The pages name the quantised formats but print no byte layout; the five formats below
 * (Q8_0, Q4B, NL4, CB2, CB3) are this project's own synthetic definitions.
 *
 * All byte layouts are little-endian; fp16 fields are IEEE binary16 bit patterns.
 *   q8_1 (36 B per 32 values) : u16 d, u16 s, i8 q[32]            ([P1] "Why": 36-byte blocks)
 *   Q8_0 (34 B per 32 weights): u16 d, i8 q[32]                    w = d*q
 *   Q4B  (20 B per 32 weights): u16 d, u16 m, u8 qs[16]            w = d*code + m
 *   NL4  (18 B per 32 weights): u16 d, u8 qs[16]                   w = d*table[code]
 *       code j = qs[j] & 15 for j < 16, qs[j-16] >> 4 for j >= 16
 *   CB2  (70 B per 256 weights): u16 D, u8 idx[32], u8 sign[32], u8 sub[4]
 *       weight n: group i = n/8, p = n%8: +-grid2[idx[i]][p], bit p of sign[i] negates
 *   CB3  (102 B per 256 weights): u16 D, u8 idx[64], u8 sign[32], u8 sub[4]
 *       weight n: group i = n/4, p = n%4: +-grid3[idx[i]][p], bit n%8 of sign[n/8] negates
 *   CB2/CB3 sub-block j (32 weights): sub_j = (sub[j>>1] >> 4*(j&1)) & 15, ls_j = 2*sub_j+1,
 *       w = D * ls_j * (+-grid value)
 * Transcoded slot layouts (load-time re-encodings of CB2/CB3 holding the same integers): each
 * weight's signed odd value v = +-grid is stored as u = (v - 1)/2 + bias, so v = 2*(u - bias) + 1.
 * A row of K weights is K/256 code chunks followed by K/256 scale records of 8 bytes
 * (u16 D, u16 0, u8 sub[4]):
 *   CB3X: 128 B of 4-bit codes per 256 weights, bias 8 (|v| <= 15). In 32-weight sub-block j
 *         (16 bytes): byte i, low nibble = weight i, high nibble = weight 16 + i.
 *   CB2X:  64 B of 2-bit codes per 256 weights, bias 2 (|v| <= 3). In sub-block j (8 bytes):
 *         bits 2p..2p+1 of byte i = weight 8p + i.
 * Rows of the native formats are K/32 blocks (K/256 super-blocks) packed without padding.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_Q8_0 = 1, ORC_Q4B = 2, ORC_NL4 = 3, ORC_CB2 = 4, ORC_CB3 = 5, ORC_CB3X = 6, ORC_CB2X = 7 };

/* IEEE binary16 <-> binary32, round to nearest even (subnormals kept). */
float orc_h2f(uint16_t h);
uint16_t orc_f2h(float f);

/* exp, silu and the SwiGLU product in fp32 (round to nearest, no fused multiply-add). */
float orc_expf(float x);
float orc_silu(float g);
float orc_swiglu(float g, float u);

/* Bytes of one row of K weights in the given format (0 if K is not a valid length). */
int64_t orc_row_bytes(int type, int K);

/* q8_1 of n values (n % 32 == 0): out receives n/32 blocks of 36 bytes. */
void orc_quantize_q8_1(const float* x, int64_t n, uint8_t* out);

/* Transcode one row of CB2/CB3 (src_type) into the slot layout dst_type (CB3X or CB2X).
 * Returns 0, or -1 when a value does not fit the slot's code range (row left unspecified). */
int orc_transcode_row(int src_type, const uint8_t* src, int K, const int8_t* cb, int dst_type, uint8_t* dst);

/* Dequantize one row to fp64 (w[K]); cb is the codebook (CB2 256x8, CB3 256x4, NL4 16). */
void orc_dequant_row(int type, const uint8_t* row, int K, const int8_t* cb, double* w);

/* Integer weight codes of one row (the values the integer dot products use):
 * Q8_0 q, Q4B code, NL4 table[code], CB2/CB3 +-grid value. */
void orc_int_weights(int type, const uint8_t* row, int K, const int8_t* cb, int32_t* v);

/* Per 32-block integer sums isum[b] = sum_i v_i * q_i of one row against one q8_1 row. */
void orc_block_isum(int type, const uint8_t* row, int K, const int8_t* cb, const uint8_t* xq,
                    int32_t* isum);

/* One row against one q8_1 row by the block-contribution formula, summed in fp64. */
double orc_row_dot(int type, const uint8_t* row, int K, const int8_t* cb, const uint8_t* xq);

/* Grouped GEMV (gate/up and down): for every group g < n_groups with expert x = grp_expert[g]
 * and every entry e in [grp_start[g], grp_start[g+1]): out[o(e)*out_stride + r] =
 * row_dot(W_x row r, act row i(e)) for r < rows, with i(e) = ent_in ? ent_in[e] : e and
 * o(e) = ent_out ? ent_out[e] : e. act holds rows of K/32 q8_1 blocks. Returns 0, or -1 on
 * an expert id out of range (nothing written for that group). */
int orc_grouped_gemv(int type, const int8_t* cb, int K, int rows, const uint8_t* const* w,
                     int n_experts, const int32_t* grp_expert, const int32_t* grp_start,
                     int n_groups, const uint8_t* act, const int32_t* ent_in,
                     const int32_t* ent_out, double* out, int64_t out_stride);

/* SwiGLU + q8_1 over entries [e0, e1): gu rows are [gate F | up F] fp32, hq rows F/32 blocks. */
void orc_swiglu_q8_1(const float* gu, int F, int e0, int e1, uint8_t* hq);

/* Routing/grouping of topk_ids[T][k]: groups by ascending expert id, entries inside a group by
 * ascending (t, slot); entries numbered from entry_base. Outputs: grp_expert[G],
 * grp_start[G+1], *n_groups, ent_src[e] = t, ent_dst[e] = t*k + slot (indexed by global e).
 * Ids outside [0, n_experts) are dropped and counted in the return value. */
int orc_route_group(const int32_t* topk_ids, int T, int k, int n_experts, int entry_base,
                    int32_t* grp_expert, int32_t* grp_start, int32_t* n_groups,
                    int32_t* ent_src, int32_t* ent_dst);

/* The steps either side of the grouped call (the pages do not define the router; this is the
 * plainest reading, and "the combined output" of #3455's parity check for the combine):
 * router: for each token t, the k largest of logits[t][0..E) (ties: the lower expert id first)
 * in descending order -> topk_ids[t][0..k); weights[t][j] = e^(l_j) / sum over the k selected
 * of e^(l_i), in fp64 (libm exp). Returns -1 if k > E or k <= 0. */
int orc_router_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, double* weights);

/* combine: y[t][n] = sum over j < k with 0 <= topk_ids[t][j] < E of weights[t][j] * out[t*k+j][n],
 * in fp64 (rows of n_embd values, out_stride apart). */
void orc_combine(const float* out, int64_t out_stride, const int32_t* topk_ids, const double* weights, int T,
                 int k, int E, int n_embd, double* y);

/* QSA decode block scores (#2059 "QSA decode: the window's block scores with the queries in
 * registers and six shuffles per block"): queries q[T][4 heads][128] fp32, one pooled key per
 * block, keys[n_blocks][128] int8 with an fp32 scale[n_blocks] (> 0). For query t and block b,
 * head h: lane l (0..31) takes the slice 4l..4l+3, p_l = q0*k0, then p_l = fma(q_i, k_i, p_l)
 * for i = 1, 2, 3 (k exact in fp32); the 32 partials are summed with the warp sum's pairings
 * (level j = 16, 8, 4, 2, 1: p_l <- p_l + p_(l xor j)); r_h = max(dot_h * scale_b, 0);
 * scores[t][b] = ((r_0 + r_1) + r_2) + r_3, plus 1e9 for the tail block b = n_blocks - 1.
 * All fp32, one rounding per operation. */
#define ORC_QSA_HEADS 4
#define ORC_QSA_DIM 128
#define ORC_QSA_LANES 32
void orc_qsa_block_scores(const float* q, int T, const int8_t* keys, const float* scale, int64_t n_blocks,
                          float* scores);

#ifdef __cplusplus
}
#endif
#endif
