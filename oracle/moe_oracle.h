/*
 * CPU oracle for the forward pass of one Mixture-of-Experts layer, and for its
 * backward pass with the top-K choice held fixed.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, plain reference the CUDA library
 * is checked against. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no code, header, table or helper with the
 * CUDA library, and the CUDA library never calls it.
 *
 * bf16 values travel as their raw 16-bit patterns (uint16_t). Every array is
 * dense row-major; sizes are in elements.
 *
 * Sources (page title, section):
 *   "混合专家模型(MoE)架构优化与SonicMoE实践" (SonicMoE page)
 *       §1    X in R^{T x d}; the router scores E experts per token and keeps the
 *             best K; then Gather, a two-layer expert MLP (GEMM), and Scatter back
 *             to the tokens' positions; H = SiLU(W1 X) held at 2 bytes/element.
 *       §2.2  SwiGLU fused into the GEMM epilogue; intermediates grouped by expert;
 *             the backward pass (dH, and the routing-score gradient dS fused
 *             into it) exists, its formulas are not printed: the backward here is
 *             the chain rule of the forward definition.
 *       §3.1  expert_frequency_estimation: per-expert counts as a loop over t, k.
 *       §3.2  the kept routing scores are renormalised (softmax renormalisation).
 *   "Triton优化MoE模型：topk_gating算子融合实战" (top-k gating page)
 *       §2.1  flow: logits -> softmax -> top-k -> output.
 *       §2.2  max-subtracted softmax over a token's expert scores, then top-2.
 *       §4.1  subtract the maximum before exp for numerical stability.
 *   "稀疏矩阵乘法（SpMM）在MoE中的应用：利用Triton内核加速稀疏专家的计算" (SpMM page)
 *       §2    CSR row offsets (an exclusive prefix sum of per-row counts).
 *       §6    the outputs of the selected experts are combined with their weights.
 *
 * Readings where the pages are silent (each is stated where it is used):
 *   - router logits are fp32: per (token, expert), one fused multiply-add chain
 *     over j = 0..d-1 ascending from +0.0f when E > 32; with E <= 32 one such
 *     chain over each block of 1024 consecutive j, the block sums added in
 *     ascending block order; then + bias[e] as a single fp32 add;
 *   - top-K is chosen on the logits (softmax is strictly increasing, so the same
 *     set), ties go to the lower expert index, output in descending order;
 *   - probabilities and weights are computed in double, rounded once to fp32;
 *   - the gated branch is W1 (SiLU), the linear branch W3, no biases;
 *   - H is rounded to bf16 (2 bytes/element); Z and Y sums stay in double until
 *     the single final bf16 rounding of Y;
 *   - rows of one expert are ordered by ascending token index.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Round a double to the nearest bf16 (ties to even) and return its bits. */
uint16_t oracle_bf16_from_double(double v);
/* Exact value of a bf16 bit pattern. */
double oracle_bf16_to_double(uint16_t b);

/* L[t,e] = fp32 fma chain over j ascending of X[t,j]*Wr[j,e] (with E <= 32,
 * one chain per 1024-step block of j, block sums added in ascending order),
 * + bias[e]. */
void oracle_router_logits(const uint16_t *X, const float *Wr, const float *bias,
                          int64_t T, int d, int E, float *L);

/* Top-K of each logit row (ties: lower index first), softmax in double, weights
 * renormalised over the K kept experts when renorm != 0. idx/w are [T,K]. */
void oracle_topk_softmax(const float *L, int64_t T, int E, int K, int renorm,
                         int32_t *idx, float *w);

/* counts[e] = number of (t,k) with idx[t,k] == e (plain double loop). */
void oracle_expert_counts(const int32_t *idx, int64_t T, int K, int E, int32_t *counts);

/* offsets[E+1] (exclusive prefix sum of counts); rows of expert e occupy
 * offsets[e]..offsets[e+1]-1 in ascending token order. perm_token[p] = t,
 * perm_slot[p] = t*K+k, row_of_slot[t*K+k] = p. */
void oracle_permute(const int32_t *idx, int64_t T, int E, int K,
                    int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                    int32_t *row_of_slot);

/* Fixed-size row blocks per expert: for every expert with rows, ceil(count/M)
 * blocks {expert, first row, rows (<= M), 0} in expert order. Writes at most
 * max_tiles entries of tiles[.][4] and returns the number of blocks. */
int oracle_tile_schedule(const int32_t *offsets, int E, int M, int32_t *tiles, int max_tiles);

/* H[p,:] = bf16( SiLU(x W1[e]) * (x W3[e]) ), x = X[perm_token[p]], for the rows
 * p of each expert e; sums in double over d ascending. W1/W3 are [E,d,n]. */
void oracle_gate_up(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                    const int32_t *perm_token, const int32_t *offsets,
                    int E, int d, int n, uint16_t *H);
/* The pre-activations of the same rows, unrounded: A1[p,:] = x W1[e] and
 * A3[p,:] = x W3[e] in double ([R,n] each), the two products gate_up rounds
 * SiLU(A1)*A3 from. A training forward keeps them for the backward pass. */
void oracle_gate_up_pre(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                        const int32_t *perm_token, const int32_t *offsets, int E, int d, int n,
                        double *A1, double *A3);

/* Z[p,:] = w[perm_slot[p]] * (H[p,:] W2[e]) in double; W2 is [E,n,d]. */
void oracle_down(const uint16_t *H, const uint16_t *W2, const float *topk_w,
                 const int32_t *perm_slot, const int32_t *offsets,
                 int E, int n, int d, double *Z);

/* Y[t,:] = bf16( sum over k ascending of Z[row_of_slot[t*K+k],:] ), double sum. */
void oracle_combine(const double *Z, const int32_t *row_of_slot, int64_t T, int K,
                    int d, uint16_t *Y);
/* Same with bf16 Z rows (used to check the combine step on its own). */
void oracle_combine_bf16(const uint16_t *Z, const int32_t *row_of_slot, int64_t T,
                         int K, int d, uint16_t *Y);

/* The layer for a list of tokens, straight from the definition, token by token:
 * route the token, run each selected expert's SwiGLU MLP on it, weight and sum.
 * Outputs per listed token: Y rows [n_tok,d], idx/w rows [n_tok,K]. */
void oracle_forward_tokens(const uint16_t *X, const float *Wr, const float *bias,
                           const uint16_t *W1, const uint16_t *W3, const uint16_t *W2,
                           int64_t T, int d, int E, int K, int n, int renorm,
                           const int64_t *tokens, int64_t n_tok,
                           uint16_t *Y_rows, int32_t *idx_rows, float *w_rows);

/* ---- Token Rounding (SonicMoE page, §3 "令牌舍入路由"): a routing mode whose
 * per-expert row counts are multiples of the tile size M, so no tile is padded.
 *
 * Inputs: the router logits L [T,E] and the plain top-K choice idx [T,K] made
 * from them (oracle_topk_softmax). Steps:
 *   1. f_e = the number of (t,k) with idx[t,k] == e (§3.1, expert frequency).
 *   2. c_e = f_e rounded to the nearest multiple of M, halves up:
 *      M * floor((f_e + floor(M/2)) / M) (§3.2's rounding kernel; §3.1 allows
 *      either the rounded-up or the rounded-down multiple and this picks the
 *      nearer). If that exceeds T (an expert can take each token at most once)
 *      the rounded-down multiple is used.
 *   3. The second sort (§3.1): for expert e, order all T tokens by (token chose
 *      e in its top-K first, then L[t,e] descending, then t ascending) and keep
 *      the first c_e. Rounding down drops the chosen tokens with the lowest
 *      scores for e; rounding up adds the unchosen tokens with the highest.
 *   4. Rows are grouped by expert, ascending t inside an expert:
 *      offsets = exclusive prefix sum of c, perm_token[p] = t of row p,
 *      row_map[t,e] = the row of (t,e), -1 when t is not kept by e.
 *   5. Weights (§3.2, softmax renormalisation after rounding): p = softmax(L[t,:])
 *      in double; row_w[row_map[t,e]] = p_e / (sum of p over the experts that
 *      kept t) when renorm != 0, else p_e; rounded once to fp32.
 * The score compared in step 3 is the logit, the same fp32 value that decided
 * the top-K: for one token it orders experts exactly as p does.
 * Returns the number of rows R' = offsets[E], or -1 (and writes no rows) when R'
 * would exceed cap, the length of perm_token and row_w. counts_out is [E]. */
int64_t oracle_token_rounding(const float *L, const int32_t *idx, int64_t T, int E, int K,
                              int M, int renorm, int64_t cap, int32_t *counts_out,
                              int32_t *offsets, int32_t *perm_token, int32_t *row_map,
                              float *row_w);

/* Y[t,:] = bf16( sum over e ascending with row_map[t,e] >= 0 of Z[row_map[t,e],:] ),
 * double sum; a token no expert kept gets zeros. row_map is [T,E]. */
void oracle_combine_rows(const double *Z, const int32_t *row_map, int64_t T, int E, int d,
                         uint16_t *Y);
/* Same with bf16 Z rows (used to check the combine step on its own). */
void oracle_combine_rows_bf16(const uint16_t *Z, const int32_t *row_map, int64_t T, int E,
                              int d, uint16_t *Y);

/* The layer output for a list of tokens under a given expert assignment, token
 * by token: Y[t] = bf16( sum over e ascending with row_map[t,e] >= 0 of
 * row_w[row_map[t,e]] * SwiGLU-MLP_e(X[t]) ). */
void oracle_forward_assigned(const uint16_t *X, const uint16_t *W1, const uint16_t *W3,
                             const uint16_t *W2, int64_t T, int d, int E, int n,
                             const int32_t *row_map, const float *row_w,
                             const int64_t *tokens, int64_t n_tok, uint16_t *Y_rows);

/* Threads the OpenMP loops use (1 when built without OpenMP). */
int oracle_num_threads(void);

/* Backward of the layer with the top-K choice idx [T,K] held fixed (routing
 * is not differentiable; the weights are). oracle_forward_fixed computes, in
 * double, Y [T,d] of the layer with that choice and without the bf16 roundings
 * of H and Y (the roundings pass gradients through unchanged); oracle_backward
 * returns the gradient of sum(Y * dY) with respect to X (dX [T,d]), Wr (dWr
 * [d,E]), bias (dbias [E], may be NULL), W1 and W3 (dW1, dW3 [E,d,n]) and W2
 * (dW2 [E,n,d]). All inputs and outputs are double (bf16 and fp32 tensors
 * widen exactly). Single-threaded: sized for tests. */
void oracle_forward_fixed(const double *X, const double *Wr, const double *bias,
                          const double *W1, const double *W3, const double *W2,
                          const int32_t *idx, int64_t T, int d, int E, int K, int n, int renorm,
                          double *Y);
void oracle_backward(const double *X, const double *Wr, const double *bias,
                     const double *W1, const double *W3, const double *W2,
                     const int32_t *idx, const double *dY, int64_t T, int d, int E, int K, int n,
                     int renorm, double *dX, double *dWr, double *dbias, double *dW1,
                     double *dW3, double *dW2);
/* The same gradient's per-row quantities in grouped row order (perm_slot [T*K]
 * as oracle_permute writes it): dS [T*K] (the routing weights' gradients),
 * dA1, dA3 [T*K,n] (the gradients of x W1[e] and x W3[e]), dXg [T*K,d] (each
 * row's share of dX) and dL [T,E] (the logits' gradient). Summed as the
 * comment at its definition says, they give oracle_backward's dX, dW1, dW3,
 * dWr and dbias. */
void oracle_backward_rows(const double *X, const double *Wr, const double *bias,
                          const double *W1, const double *W3, const double *W2,
                          const int32_t *idx, const int32_t *perm_slot, const double *dY,
                          int64_t T, int d, int E, int K, int n, int renorm, double *dS,
                          double *dA1, double *dA3, double *dXg, double *dL);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
