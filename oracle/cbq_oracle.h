/*
 * cbq_oracle.h -- CPU oracle for the codebook-4bit quantized matvec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package
 * entry module and the CPU-baseline leg of the benchmark may load this code.
 * The product path (the CUDA library) never calls it, shares no code with it
 * and has no CPU fallback.
 *
 * What it computes, in the order the pages describe it:
 *   - the 4-bit codebook weight format registered as new quant types
 *     ("feat(ds4): add DSpark speculative runtime + optimizations" #496,
 *     summary: "ROCmFP4/ROCmFPX quant types + CPU reference conversions");
 *   - activation quantization to per-32 int8 plus an fp32 scale, and the
 *     per-block integer dot of the MMVQ vecdot ("... MMVQ vecdot, MMVF ..."
 *     in the same summary);
 *   - the quantized matvec over 1..n activation columns (MMVQ with ne1 > 1
 *     columns; MMVQ_MAX_MOE_BATCH_SIZE in the same summary);
 *   - the routed-expert mul_mat_id with the SwiGLU split and the
 *     router-weighted combine ("DS4 SwiGLU split op plumbing for the fused
 *     FFN matvec paths"; "DFLASH_DS4_FFN_RAW_MMID / DFLASH_DS4_FFN_FUSED_COMBINE
 *     accumulation reorder" in "fix(ds4): keep ROCmFPX generation byte-safe"
 *     #494; "configured routed-expert top-k" in "feat(ds4): add DSpark
 *     speculative decoding").
 *
 * Format (the pages print no layout; these are the plain readings used
 * throughout this library):
 *   - one block = 32 weights along K = 18 bytes: bytes 0-1 an IEEE binary16
 *     scale dw (little-endian), bytes 2-17 the 16 index bytes qs;
 *   - qs byte j (0..15) holds the index of element j in its low nibble and of
 *     element j+16 in its high nibble (the "get_int"/"get_low_int" pair of the
 *     codebook-16 expander in "fix(ggml): make ROCmFP4 codebook
 *     self-contained on CUDA" feeds the two 16-element halves);
 *   - weight i = dw * codebook[index_i] with the 16-level int8 codebook below;
 *   - a matrix W of M rows x K columns is stored row-major as M x (K/32)
 *     blocks.
 *
 * Precision: activation quantization is fp32 (its rule fixes fp32: d =
 * max|x|/127 in fp32, q = round-half-to-even(x/d)); every accumulation of the
 * matvec and of the MoE is fp64; the MoE intermediate a = silu(g)*u is
 * rounded to fp32 before it is requantized, because the down projection takes
 * it through the same fp32 quantization rule.
 *
 * Parity pins (see the tests): fp16 decoding against numpy over all 65536
 * patterns; quantization against hand-worked fixtures and exact-rational
 * nearest/tie-to-even properties; block dots against the per-entry table,
 * one-hot positions and a hand-worked block; the matvec against an fp64
 * dequantize-then-dot; scale linearity, sign symmetry and zero scales; the MoE
 * against its k=1 reduction, the silu odd-part identity and token independence;
 * the weight converter against numpy's binary16 rounding, hand-worked blocks
 * (ties, a negative maximum, a zero block), an exact round trip of weights on
 * the codebook grid and an exact-rational nearest-level search; the sinkhorn
 * normalisation against the closed forms of a rank-one matrix (uniform after
 * one step) and of the 2 x 2 limit, the fixed point of a doubly stochastic
 * input, invariance to a constant added to a row, permutation equivariance
 * and the column sums.
 */
#ifndef CBQ_ORACLE_H
#define CBQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_QK 32          /* weights per block */
#define ORACLE_BLOCK_BYTES 18 /* 2-byte fp16 scale + 16 index bytes */

/* The 16-level int8 codebook of the 4-bit format, indexed by a nibble. */
extern const int8_t oracle_codebook[16];

/* IEEE 754 binary16 -> binary32, exact for every pattern (NaN stays NaN). */
float oracle_half_to_float(uint16_t h);

/* Index (0..15) of element i (0..31) of one 18-byte block. */
int oracle_block_index(const uint8_t *blk, int i);

/* The 32 weights of one block in fp64: dw * codebook[index_i]. */
void oracle_dequantize_block(const uint8_t *blk, double out[32]);

/* Activation quantization of n columns x[c][K] (K % 32 == 0):
 * per 32-block amax = max|x|, d = amax/127 (fp32), q = rint(x/d) clamped to
 * [-127,127], and q = 0 where d == 0.  Outputs qx[c][K] and dx[c][K/32]. */
void oracle_quantize_act(const float *x, int64_t K, int n, int8_t *qx, float *dx);

/* Per-block int32 dots s[c][r][b] = sum_i codebook[idx(r,b,i)] * qx[c][32b+i]. */
void oracle_block_dots(const uint8_t *W, int64_t M, int64_t K,
                       const int8_t *qx, int n, int32_t *s);

/* y[c][r] = sum_b dw(r,b) * dx[c][b] * s[c][r][b], accumulated in fp64. */
void oracle_matvec_q(const uint8_t *W, int64_t M, int64_t K,
                     const int8_t *qx, const float *dx, int n, double *y);

/* Same, for the selected rows rows[0..nrows) only: y[c][i] for row rows[i]. */
void oracle_matvec_q_rows(const uint8_t *W, int64_t M, int64_t K,
                          const int8_t *qx, const float *dx, int n,
                          const int64_t *rows, int64_t nrows, double *y);

/* Quantize x then matvec: the whole dense hot path. */
void oracle_matvec(const uint8_t *W, int64_t M, int64_t K,
                   const float *x, int n, double *y);

/* Tolerance base of each output: bound[c][r] = sum_i |w_i * xhat_i| with
 * xhat_i = qx_i * dx (the activation the integer pipeline sees). */
void oracle_matvec_bound(const uint8_t *W, int64_t M, int64_t K,
                         const int8_t *qx, const float *dx, int n, double *bound);
void oracle_matvec_bound_rows(const uint8_t *W, int64_t M, int64_t K,
                              const int8_t *qx, const float *dx, int n,
                              const int64_t *rows, int64_t nrows, double *bound);

/* silu(z) = z / (1 + exp(-z)) in fp64. */
double oracle_silu(double z);

/* Routed-expert FFN for n_tok tokens, top-k slots each.
 *   gate_up: E experts, each 2F rows x H columns (rows 0..F-1 gate, F..2F-1 up)
 *   down:    E experts, each H rows x F columns
 *   h[t][H], ids[t][k], wts[t][k]
 * For every token t and slot j (in slot order) with e = ids[t][j] in [0,E):
 *   qh,dh = quantize(h_t); g,u = gate/up rows . (qh,dh) in fp64;
 *   a = fp32( swiglu ? silu(g)*u : g*u ); qa,da = quantize(a);
 *   o = down_e . (qa,da) in fp64;  y_t += wts[t][j] * o  (fp64).
 * A slot whose id is outside [0,E) contributes nothing and counts in the
 * return value (the number of such slots).
 * Optional outputs (NULL to skip), all indexed by slot p = t*k + j:
 *   a_out[p][F] (fp32), qa_out[p][F] (int8), da_out[p][F/32] (fp32).
 * y[t][H] is fp64. */
int oracle_moe(const uint8_t *gate_up, const uint8_t *down, int E, int64_t H, int64_t F,
               const float *h, int n_tok, const int32_t *ids, const float *wts, int k,
               int swiglu, double *y, float *a_out, int8_t *qa_out, float *da_out);

/* Routed layer plus one shared expert that every token passes through with
 * router weight 1 (the DS4 FFN block's always-on expert; the pages name the
 * routed layer only, so the shared expert is read as one more expert of the
 * same shape, applied to every token after its routed slots):
 *   y_t = sum_j wts[t][j] * o_{ids[t][j]}(h_t)  +  o_sh(h_t)
 * where o_sh is the per-slot computation of oracle_moe with the weights
 * sh_gate_up (2F x H) and sh_down (H x F).  The routed sum is formed first
 * and the shared output added to it (fp64).  Returns the number of routed
 * slots whose id is outside [0,E). */
int oracle_moe_shared(const uint8_t *gate_up, const uint8_t *down, int E, int64_t H, int64_t F,
                      const uint8_t *sh_gate_up, const uint8_t *sh_down,
                      const float *h, int n_tok, const int32_t *ids, const float *wts, int k,
                      int swiglu, double *y);

/* The down projection + combine alone, from given per-slot quantized
 * intermediates qa[p][F], da[p][F/32] (p = t*k + j).  Also returns the
 * tolerance base ybound[t][H] = sum_j |wts| * sum_i |wd_i * ahat_i|. */
int oracle_moe_down_combine(const uint8_t *down, int E, int64_t H, int64_t F,
                            int n_tok, const int32_t *ids, const float *wts, int k,
                            const int8_t *qa, const float *da,
                            double *y, double *ybound);

/* Routed-expert selection from router logits (the "configured routed-expert
 * top-k" of "feat(ds4): add DSpark speculative decoding"; the pages give no
 * formula, the plain reading is used): for every token t, ids[t][0..k) are
 * the indices of the k largest logits[t][0..E) in descending order, equal
 * logits ordered by the lower index first; wts[t][j] is the softmax over the
 * k selected logits, computed in fp64 (exp(l_j - l_max) / sum).
 * 1 <= k <= E. */
void oracle_router_topk(const float *logits, int n_tok, int E, int k, int32_t *ids, double *wts);

/* IEEE 754 binary32 -> binary16, rounded to nearest, ties to even; values of
 * magnitude 65520 and above (and infinities) give infinity, NaN a quiet NaN. */
uint16_t oracle_float_to_half(float f);

/* The weight converter: fp32 weights to the 4-bit codebook format (the
 * "CPU reference conversions" of the quant types in "feat(ds4): add DSpark
 * speculative runtime + optimizations" #496; the pages give no rule, this is
 * the plain reading).  For one block of 32 weights w[0..32):
 *   m = the weight of largest magnitude (the first one among equal
 *       magnitudes); if m == 0 the block is all zero bytes;
 *   dw = binary16(m / -127): the fp32 division, then rounding to nearest
 *       even -- -127 is the codebook level of largest magnitude, so m lands
 *       on it;
 *   index_i = the j minimising |w_i - dw * codebook[j]| (distances exact in
 *       fp64), the lowest j among equal distances;
 * packed as the format says (dw little-endian in bytes 0-1, element i's index
 * in the low nibble of byte 2+i for i < 16, in the high nibble of byte
 * 2+i-16 otherwise).  |m| must stay below 127 * 65520 (a finite scale). */
void oracle_quantize_weights_block(const float *w, uint8_t *blk);

/* A row-major M x K fp32 matrix (K % 32 == 0) to M x (K/32) blocks. */
void oracle_quantize_weights(const float *w, int64_t M, int64_t K, uint8_t *blocks);

/* Sinkhorn normalisation of the hyper-connection mixing matrices (the
 * "register-resident sinkhorn kernel" of the fused DS4 hyper-connection op,
 * GGML_OP_DS4_HC, in "feat(ds4): add DSpark speculative runtime +
 * optimizations" #496; its NHC = 4 specialisation in "fix(ds4): keep ROCmFPX
 * generation byte-safe" #494; the pages give neither the iteration count nor
 * the update, the plain reading of a Sinkhorn normalisation is used).  For
 * each of the n row-major nhc x nhc matrices c of logits:
 *   P = exp(c - max(c)), in fp64 (the shift multiplies P by a positive
 *       constant, which the first normalisation removes);
 *   `iters` times: divide every row of P by its sum, then every column by
 *       its sum (sums in index order);
 * out = P after the last column step (its columns sum to 1).
 * nhc >= 1, iters >= 0 (0 gives exp(c - max c) itself). */
void oracle_hc_sinkhorn(const float *logits, int64_t n, int nhc, int iters, double *out);

#ifdef __cplusplus
}
#endif

#endif /* CBQ_ORACLE_H */
