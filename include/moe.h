/*
 * moe.h - C ABI of libmoe.so: the forward pass of one Mixture-of-Experts layer
 * on an NVIDIA GB300 (sm_103a).
 *
 * The layer (page "混合专家模型(MoE)架构优化与SonicMoE实践", §1): tokens
 * X[T,d] are scored against E experts by a router, each token keeps its best K
 * experts, rows are gathered per expert, each expert applies a two-layer SwiGLU
 * MLP (W1/W3 [E,d,n] up, W2 [E,n,d] down), and the weighted expert outputs are
 * scattered back and summed per token:
 *
 *   L[t,:]  = X[t,:] Wr (+ bias)                       router logits, fp32
 *   idx, w  = top-K of softmax(L[t,:]), renormalised  (ties -> lower index)
 *   H[p,:]  = SiLU(x W1[e]) * (x W3[e])                x = X[t_p], bf16 out
 *   Z[p,:]  = w_p * (H[p,:] W2[e])                     bf16 out
 *   Y[t,:]  = sum_k Z[row_of_slot[t*K+k],:]            ascending k, fp32 sum, bf16 out
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless a parameter says "host". The caller
 *     owns every buffer, including the workspace; the library allocates no
 *     device memory and keeps no state besides a per-device cache of the SM
 *     count and architecture check (and the built-in scratch array of
 *     moe_permute_noalloc, below).
 *   - bf16 data travels as raw 16-bit patterns (moe_bf16). Matrices are dense
 *     and row-major. Integer outputs are int32.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work on it and return; none waits for the GPU (except
 *     moe_sync_check, moe_forward_host and moe_forward_host_stream, which say so).
 *   - Argument and shape errors are reported synchronously, before anything is
 *     enqueued. A failed launch returns MOE_ERR_CUDA. Problems the kernels
 *     detect on the device (an expert index out of range, a stalled pipeline
 *     that gave up after its time limit) set bits in the workspace's error word,
 *     which moe_sync_check reads.
 *   - Supported shapes: 1 <= T, 1 <= E <= 256, 1 <= K <= min(E, 8);
 *     d % 256 == 0 and n % 128 == 0 for the expert GEMMs (d % 8 == 0 for the
 *     router and combine alone); T*K*max(d,n) < 2^31. Anything else returns
 *     MOE_ERR_UNSUPPORTED_SHAPE.
 *   - The kernels are built for sm_103a only; any other device returns MOE_ERR_ARCH.
 *   - Every kernel is launched with programmatic dependent launch: it may start
 *     while the previous kernel on the stream finishes, and waits for that
 *     kernel's results before reading global memory. Results do not depend on it.
 *   - Environment variables that choose between kernels for the same step (for
 *     tests and measurements; unset is the default choice). Routing results are
 *     bit-identical either way; GEMM outputs may differ within rounding:
 *       MOE_PDL=0             launch without programmatic dependent launch (read
 *                             once per process);
 *       MOE_GEMM_CTA_PAIR=0/1 expert GEMMs on single CTAs / on CTA pairs;
 *       MOE_GEMM_FUSED=1      both expert GEMMs in one launch where n <= 2048
 *                             (default: two launches; see moe_expert_mlp);
 *       MOE_FUSED_GAP_ROUNDS=g rounds the fused launch keeps between a
 *                             gate/up round and the down rounds reading it
 *                             (default 2);
 *       MOE_ROUTER_PAIRS=4..8 router logits (E > 32) on the one-block-per-SM
 *                             kernel with that many token pairs per scheduler;
 *                             0: on the 4 x 8 register-tile kernel.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad flag */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set above */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,/* ws_bytes < moe_workspace_bytes(...) */
    MOE_ERR_ARCH = 4,               /* current device is not sm_103 */
    MOE_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_TIMEOUT = 6,     /* a kernel wait hit its time limit (error word) */
    MOE_ERR_DEVICE_CHECK = 7        /* a kernel found bad input data (error word) */
} moe_status_t;

/* Bits of the device error word (first 4 bytes of the workspace). */
#define MOE_DEVERR_TIMEOUT      0x1u  /* a pipeline wait gave up after its time limit */
#define MOE_DEVERR_BAD_EXPERT   0x2u  /* a top-K index outside [0, E) was skipped */
#define MOE_DEVERR_COUNT_MISMATCH 0x4u /* counts[] disagreed with the recount of topk_idx */
#define MOE_DEVERR_REPEATED_EXPERT 0x8u /* a token listed one expert twice; the repeat was skipped */

/* Human-readable name of a status code (static string). */
const char *moe_status_string(int status);

/* Version of this ABI (major*100 + minor). 101 added the Token Rounding calls. */
int moe_abi_version(void);

/* Bytes of workspace the calls below need for this layer shape; 0 for an
 * invalid shape. The workspace holds, 256-byte aligned: the device error word,
 * counts[E], offsets[E+1], tile_base[E+1], the grouping scratch
 * (ceil(T/32)*E counters and T*K ranks), perm_token/perm_slot/row_of_slot [T*K],
 * topk_idx/topk_w [T*K] for moe_forward, the tile list [T*K/128+E][4], the
 * gathered rows Xg [T*K,d] bf16 (used by the CTA-pair gate/up GEMM), H [T*K,n]
 * bf16, Z [T*K,d] bf16 and the router logits [T,E] fp32 (moe_forward).
 * Before first use the caller zeroes it once (moe_workspace_init). */
size_t moe_workspace_bytes(int T, int d, int E, int K, int n);

/* Zero the workspace's error word, control words and the one-kernel
 * grouping's block flags: its first min(ws_bytes, 512) bytes (enqueued on
 * `stream`). */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Router from activations (page "Triton优化MoE模型：topk_gating算子融合实战",
 * §2.1-§2.2, and the SonicMoE page §1, §3.2).
 *   X       [T,d] bf16      token activations
 *   Wr      [d,E] fp32      router weights
 *   bias    [E] fp32 or NULL  added to every token's logits
 *   renorm  1: weights renormalised over the K kept experts; 0: raw softmax probs
 * Outputs: logits [T,E] fp32 (the router scores; also the call's scratch),
 *          topk_idx [T,K] int32 (descending score; ties -> lower index),
 *          topk_w [T,K] fp32, counts [E] int32 (tokens routed to each expert;
 *          the call zeroes it first).
 * Logits are fp32 fused multiply-add chains over j ascending from +0, then
 * + bias[e]: with E > 32 one chain over j = 0..d-1; with E <= 32 one chain per
 * block of 1024 consecutive j, the block sums added in ascending block order.
 * Bit-identical to that sequential definition. With E <= 32, E % 4 == 0, a
 * 16-byte-aligned Wr and d <= 32768: a memset of counts and ONE kernel
 * (logits and selection). Otherwise two kernels (logits, then softmax and
 * top-K) and, unless E <= 16 and T <= 2048, a memset of counts. */
moe_status_t moe_route(const moe_bf16 *X, const float *Wr, const float *bias,
                       int T, int d, int E, int K, int renorm, float *logits,
                       int32_t *topk_idx, float *topk_w, int32_t *counts, void *stream);

/* Router from given logits [T,E] fp32 (softmax + top-K + counts only). Same
 * outputs as moe_route. */
moe_status_t moe_route_logits(const float *logits, int T, int E, int K, int renorm,
                              int32_t *topk_idx, float *topk_w, int32_t *counts,
                              void *stream);

/* Group the routed slots by expert (SonicMoE page §1 Gather, §2.2 grouping by
 * expert, §3.1 per-expert counts; SpMM page §2 CSR row offsets).
 *   topk_idx [T,K] int32, each row K distinct experts (as the router writes
 *   it); counts [E] int32 or NULL (when given it is checked against a recount
 *   on the device; a mismatch sets MOE_DEVERR_COUNT_MISMATCH).
 * Outputs: offsets [E+1]; rows of expert e are offsets[e]..offsets[e+1]-1 in
 *   ascending token order; perm_token [T*K] (token of each grouped row),
 *   perm_slot [T*K] (t*K+k of each row), row_of_slot [T*K] (inverse of
 *   perm_slot; -1 for a slot whose index was out of range, which sets
 *   MOE_DEVERR_BAD_EXPERT, or repeats an expert listed earlier in its token's
 *   row, which sets MOE_DEVERR_REPEATED_EXPERT; such slots get no row and the
 *   rows in use end at offsets[E] < T*K);
 *   tiles [(T*K)/128 + E][4] int32 = {expert, first row, rows<=128, 0}, expert
 *   order, and num_tiles [1] (tile_base[E]). ws: workspace of this shape.
 * Kernels: for T <= 65536 ONE (each block counts its run of 32-token chunks
 * per expert, publishes the counts with a flag and, behind bounded waits on
 * every block's flag, takes the offsets from the expert totals and its start
 * within each expert from the blocks before it, then scatters); otherwise three
 * (rank, scan, scatter). The result is the same either way. */
moe_status_t moe_permute(const int32_t *topk_idx, const int32_t *counts,
                         int T, int E, int K,
                         int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                         int32_t *row_of_slot, int32_t *tiles, int32_t *num_tiles,
                         void *ws, size_t ws_bytes, void *stream);

/* moe_permute for callers that cannot allocate device memory. The pages have
 * no counterpart of this call: it exists for code that is given only its inputs
 * and outputs and may not call cudaMalloc, e.g. a plugin inside an inference
 * engine that owns all device memory, or a serving loop whose memory was
 * planned at start-up (cudaMalloc can synchronise the device and can fail once
 * memory is fragmented). Same arguments and outputs as moe_permute, without
 * the workspace: the grouping scratch is a 4 MiB array built into libmoe.so
 * (every GPU that loads the library holds it until the process exits). The
 * call allocates nothing.
 *   - Limit: the shape's grouping scratch, moe_workspace_bytes(T, 0, E, K, 0)
 *     (about 24*T*K + 4*E*ceil(T/32) bytes), must fit in 4 MiB, i.e. T*K up to
 *     about 150000 slots; larger shapes return MOE_ERR_UNSUPPORTED_SHAPE before
 *     anything is enqueued.
 *   - The first call on each device (in each CUDA context) looks up the
 *     array's device address with that device current and keeps it for later
 *     calls in the same context. Under lazy module loading (the CUDA default)
 *     that first lookup also loads this part of the library onto the device,
 *     array included: it may need 4 MiB of free device memory and may
 *     synchronise the device. Make the first call once at start-up, before any
 *     stream capture, or run with CUDA_MODULE_LOADING=EAGER.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     the call clears what has to start at zero. Calls whose work overlaps on
 *     the GPU (other streams, other threads) race on the array: serialise them.
 *   - The device error word of these calls lives in the array and is never
 *     read back, so passing counts checks nothing here. A slot whose expert is
 *     out of range or repeated still shows up as row_of_slot == -1. */
moe_status_t moe_permute_noalloc(const int32_t *topk_idx, const int32_t *counts,
                                 int T, int E, int K,
                                 int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                                 int32_t *row_of_slot, int32_t *tiles, int32_t *num_tiles,
                                 void *stream);

/* Up-projection GEMM with the SwiGLU fused in its epilogue (SonicMoE page §1,
 * §2.2, §4.2): for every grouped row p of expert e,
 *   H[p,:] = bf16( SiLU(x W1[e]) * (x W3[e]) ),  x = X[perm_token[p],:].
 * Uses offsets [E+1] and perm_token from moe_permute; H [T*K,n] bf16. For
 * small experts the GEMM gathers the rows of X itself; for experts of >= 8
 * row tiles on average it gathers them into the workspace first and runs on
 * CTA pairs. A perm_token entry outside [0,T) is skipped and flagged.
 * ws: workspace of this shape. */
moe_status_t moe_gemm_gate_up(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                              const int32_t *perm_token, const int32_t *offsets,
                              int T, int d, int E, int K, int n, moe_bf16 *H,
                              void *ws, size_t ws_bytes, void *stream);

/* Down-projection GEMM with the routing weight applied in its epilogue:
 *   Z[p,:] = bf16( topk_w[perm_slot[p]] * (H[p,:] W2[e]) ).
 * H [T*K,n] bf16 grouped rows; Z [T*K,d] bf16. perm_slot may be NULL: the
 * weight of row p is then topk_w[p]. */
moe_status_t moe_gemm_down(const moe_bf16 *H, const moe_bf16 *W2, const float *topk_w,
                           const int32_t *perm_slot, const int32_t *offsets,
                           int T, int d, int E, int K, int n, moe_bf16 *Z,
                           void *ws, size_t ws_bytes, void *stream);

/* ---- Backward pass (SonicMoE page §2.2: the gradient of H with the routing
 * score's gradient dS computed inside it; §4.1: its TMA load pipeline). The
 * top-K choice is held fixed; the gradients follow, for every grouped row p of
 * expert e with token t = perm_token[p] and weight w = topk_w[perm_slot[p]]:
 *   g[p,j]   = sum_c dY[t,c] W2[e][j,c]                      (dH' = dY W2[e]^T)
 *   dS[p]    = sum_j g[p,j] SiLU(a1[p,j]) a3[p,j]            (dL/dw of that slot)
 *   dA1[p,j] = w g[p,j] a3[p,j] s (1 + a1[p,j] (1 - s)),  s = sigmoid(a1[p,j])
 *   dA3[p,j] = w g[p,j] SiLU(a1[p,j])
 * with a1 = x W1[e], a3 = x W3[e] the forward's pre-activations. */

/* The gate/up GEMM of a training forward: H exactly as moe_gemm_gate_up writes
 * it, and the pre-activations A1 = x W1[e], A3 = x W3[e] of every grouped row
 * (fp32 [T*K, n] each: the accumulators as they are, so that the backward's
 * sums over n do not inherit a bf16 rounding of every term) for
 * moe_backward_dh. Same arguments and workspace as moe_gemm_gate_up. */
moe_status_t moe_gemm_gate_up_train(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                                    const int32_t *perm_token, const int32_t *offsets, int T,
                                    int d, int E, int K, int n, moe_bf16 *H, float *A1,
                                    float *A3, void *ws, size_t ws_bytes, void *stream);

/* The backward's dH step: one grouped GEMM g = dY[perm_token] W2[e]^T (rows
 * of dY [T,d] bf16 gathered like X; W2 [E,n,d] read with d, the reduction, as
 * the contiguous dimension) whose epilogue forms, with A1, A3 [T*K,n] fp32
 * from moe_gemm_gate_up_train and the routing weights topk_w [T*K] fp32:
 * dA1, dA3 [T*K,n] bf16 (grouped rows) and dS [T*K] fp32 (grouped rows; each
 * row's sum over j in fp32: 32-column partials, added in a fixed order by a
 * second kernel). Needs n % 256 == 0, else MOE_ERR_UNSUPPORTED_SHAPE. ws:
 * workspace of this shape (its H region holds the partials; on CTA pairs its
 * gathered-rows region the dY rows). Two kernels, three on CTA pairs (experts of
 * >= 8 row tiles on average: a row gather first); a row index out of range is
 * skipped and flagged like the forward GEMMs'. */
moe_status_t moe_backward_dh(const moe_bf16 *dY, const moe_bf16 *W2, const float *A1,
                             const float *A3, const float *topk_w, const int32_t *perm_token,
                             const int32_t *perm_slot, const int32_t *offsets, int T, int d,
                             int E, int K, int n, moe_bf16 *dA1, moe_bf16 *dA3, float *dS,
                             void *ws, size_t ws_bytes, void *stream);

/* The backward's dX step for the expert MLPs: one grouped GEMM per row
 *   dXg[p,:] = dA1[p,:] W1[e]^T + dA3[p,:] W3[e]^T       (reduction 2n, fp32)
 * stored as bf16 [T*K, d] (grouped rows), then the combine of moe_combine:
 *   dX[t,:] = bf16( sum over k ascending of dXg[row_of_slot[t*K+k],:] )
 * dA1, dA3 [T*K, n] bf16 as moe_backward_dh writes them; W1, W3 [E,d,n] bf16
 * read with n, the reduction, as the contiguous dimension. dX is the experts'
 * share of the input gradient (the router adds dL Wr^T). ws: any workspace of
 * >= 64 bytes (its error word flags bad offsets). Two kernels. */
moe_status_t moe_backward_dx(const moe_bf16 *dA1, const moe_bf16 *dA3, const moe_bf16 *W1,
                             const moe_bf16 *W3, const int32_t *offsets,
                             const int32_t *row_of_slot, int T, int d, int E, int K, int n,
                             moe_bf16 *dXg, moe_bf16 *dX, void *ws, size_t ws_bytes,
                             void *stream);

/* The backward's weight gradients, with the top-K choice fixed (the sums over
 * each expert's grouped rows p, t = perm_token[p], w = topk_w[perm_slot[p]]):
 *   dW1[e] = sum_p X[t]^T dA1[p]      dW3[e] = sum_p X[t]^T dA3[p]    [E,d,n]
 *   dW2[e] = sum_p H[p]^T (w dY[t])                                   [E,n,d]
 * all fp32, one fp32 accumulation per output in the tensor cores. H [T*K,n]
 * bf16 (the forward's), dA1, dA3 [T*K,n] bf16 (moe_backward_dh), X, dY [T,d]
 * bf16. An expert with no rows gets zero gradients. w dY is rounded to bf16
 * once per element (an operand of the grouped GEMM). Two grouped GEMMs after
 * a gather of the rows into a layout where every expert's rows start on a
 * 64-row boundary. scratch: moe_backward_dw_scratch_bytes(T, d, E, K) bytes,
 * 256-byte aligned, whose first 4 bytes are a device error word as in a
 * workspace (zero them once before first use; moe_sync_check reads them). */
size_t moe_backward_dw_scratch_bytes(int T, int d, int E, int K);
moe_status_t moe_backward_dw(const moe_bf16 *X, const moe_bf16 *dY, const moe_bf16 *H,
                             const moe_bf16 *dA1, const moe_bf16 *dA3, const float *topk_w,
                             const int32_t *perm_token, const int32_t *perm_slot,
                             const int32_t *offsets, int T, int d, int E, int K, int n,
                             float *dW1, float *dW3, float *dW2, void *scratch,
                             size_t scratch_bytes, void *stream);

/* The router's backward (SonicMoE page §2.2: from dS, the gradient of the
 * routing scores' softmax; §3.2: the kept scores renormalised), with the
 * top-K choice fixed. Per token, with p = softmax(logits[t,:]) over all E
 * experts, kept = sum of p over the K chosen, w_k = p_k / kept (renorm) or p_k
 * and dS_k = dS[row_of_slot[t*K+k]] (moe_backward_dh):
 *   g_e     = (dS_k - sum_k' w_k' dS_k') / kept for e = topk_idx[t,k] with
 *             renorm, dS_k without; 0 for the other experts
 *   dL[t,e] = p_e (g_e - sum_e' p_e' g_e')                  fp32 [T, E]
 * and over the batch
 *   dbias   = sum over t of dL[t,:]                         fp32 [E]
 *   dWr     = X^T dL                                        fp32 [d, E]
 *   dX      = bf16( sum over k ascending of dXg[row_of_slot[t*K+k],:]
 *                   + (dL Wr^T)[t,:] )                      bf16 [T, d]
 * i.e. the full input gradient: the experts' rows (dXg from moe_backward_dx)
 * and the router's share, added in fp32 and rounded once. logits [T,E] as
 * moe_route wrote them. dWr is summed per chunk of tokens (fp32 fma chains,
 * t ascending; for E % 128 == 0, T % 1024 == 0 and d % 256 == 0 a tensor-core
 * GEMM over 1024-token chunks with dL split into bf16 high and low parts, fp32
 * accumulation) and the chunks' partials in ascending order; dL Wr^T is one
 * fp32 fma chain over e ascending per element; dbias column sums over chunks
 * of about 128 tokens (t ascending), then the chunks in ascending order: all
 * deterministic. ws: at least moe_workspace_bytes(T, d, E, K, 0) bytes (a
 * workspace of the layer's shape serves); T * d floats from its gathered-rows
 * region on hold the dbias and dWr partials (and the split dL), and one of its
 * control words the column sums' ticket. Five kernels (four when T is too
 * short to split into chunks); dL Wr^T is computed inside the last, the
 * combine. On the tensor-core path (E % 128 == 0, T % 1024 == 0, d % 256 == 0)
 * also five, or, with K >= 2, seven: dL Wr^T too is a tensor-core GEMM (Wr
 * split like dL; fp32 out, in the first T * d floats of the gathered-rows
 * region, the split operands after it), added by the combine. */
moe_status_t moe_backward_router(const moe_bf16 *X, const float *Wr, const float *logits,
                                 const int32_t *topk_idx, const float *dS,
                                 const int32_t *row_of_slot, int T, int d, int E, int K,
                                 int renorm, const moe_bf16 *dXg, moe_bf16 *dX, float *dL,
                                 float *dWr, float *dbias, void *ws, size_t ws_bytes,
                                 void *stream);

/* Both expert GEMMs: H as moe_gemm_gate_up writes it, then Z as moe_gemm_down
 * writes it, bit for bit. Two launches (three on CTA pairs); with
 * MOE_GEMM_FUSED=1 and n <= 2048, ONE persistent launch (the SonicMoE page's
 * fine-grained experts keep H small): its CTAs run rounds of gate/up units
 * (128 rows x 128 H columns) and of down units (128 rows x 256 Z columns), and a
 * down unit starts once the gate/up units of its row tile have stored H,
 * signalled through per-tile counter words in the workspace (bounded waits; a
 * wait that runs out sets MOE_DEVERR_TIMEOUT). On the SonicMoE-shaped layer the
 * fused launch measured slower than the two (0.183-0.191 against 0.170 ms).
 * ws: workspace of this shape, zeroed once before first use and not shared by
 * calls that overlap on the GPU. Takes no tile list: the GEMMs decode their
 * work units from offsets in their own order (expert-major, groups of tiles,
 * few-tile experts interleaved), which moe_permute's flat list cannot express. */
moe_status_t moe_expert_mlp(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                            const moe_bf16 *W2, const float *topk_w,
                            const int32_t *perm_token, const int32_t *perm_slot,
                            const int32_t *offsets, int T, int d, int E, int K, int n,
                            moe_bf16 *H, moe_bf16 *Z, void *ws, size_t ws_bytes,
                            void *stream);

/* Scatter back and combine (SpMM page §6, SonicMoE page §1 Scatter):
 *   Y[t,:] = bf16( sum over k = 0..K-1 ascending of Z[row_of_slot[t*K+k],:] ),
 * fp32 accumulation, one rounding; rows with row_of_slot < 0 are skipped.
 * Deterministic: no atomics. Z [T*K,d] bf16, Y [T,d] bf16. */
moe_status_t moe_combine(const moe_bf16 *Z, const int32_t *row_of_slot, int T, int K, int d,
                         moe_bf16 *Y, void *stream);

/* Kernels moe_forward (rounded = 0) or moe_forward_rounded (rounded = 1)
 * enqueues for this shape on the current device (its SM count bounds a fused
 * launch's rounds) under the current environment variables; -1 for an invalid
 * shape or flag. Host only: nothing is enqueued. */
int moe_forward_launches(int T, int d, int E, int K, int n, int rounded);

/* The part of moe_forward_launches that the expert GEMMs take: 1 fused, 2, or
 * 3 on CTA pairs; -1 for an invalid shape or flag. */
int moe_expert_mlp_launches(int T, int d, int E, int K, int n, int rounded);

/* The whole layer: route -> permute -> gate/up+SwiGLU -> down+weight -> combine.
 * topk_idx_out / topk_w_out [T,K] may be NULL (kept in the workspace then).
 * Enqueues moe_forward_launches(T, d, E, K, n, 0) kernels: the router (1 with
 * E <= 32 as moe_route says, else 2), the grouping (1 for T <= 65536, see
 * moe_permute; else 3), the expert GEMMs (2, 3
 * on CTA pairs, which gather their rows first, or 1 when both run in one launch,
 * see moe_expert_mlp) and the combine (1); and, unless E <= 16 and T <= 2048
 * with the two-kernel router, one memset of the counts; no host
 * synchronisation. The grouping here writes no tile list: the expert GEMMs
 * decode their work units from the offsets. */
moe_status_t moe_forward(const moe_bf16 *X, const float *Wr, const float *bias,
                         const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2,
                         int T, int d, int E, int K, int n, int renorm,
                         moe_bf16 *Y, int32_t *topk_idx_out, float *topk_w_out,
                         void *ws, size_t ws_bytes, void *stream);

/* moe_forward that also records CUDA events (cudaEvent_t as void*) on `stream`
 * between its stages, for per-kernel timing: events[0] before the router,
 * then after route, permute, gate/up GEMM, down GEMM, combine (6 events).
 * When both GEMMs run in one launch, the gate/up interval holds it and the
 * down interval is empty. n_events < 6 records the first n_events of them. */
moe_status_t moe_forward_traced(const moe_bf16 *X, const float *Wr, const float *bias,
                                const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2,
                                int T, int d, int E, int K, int n, int renorm,
                                moe_bf16 *Y, int32_t *topk_idx_out, float *topk_w_out,
                                void *ws, size_t ws_bytes, void *stream,
                                void *const *events, int n_events);

/* End to end from host memory: copies X_host [T,d] (host, ideally pinned) into
 * X_dev, runs moe_forward, copies Y back into Y_host [T,d] (host) and waits
 * for the stream. X_dev/Y_dev are caller-owned device buffers [T,d] bf16. */
moe_status_t moe_forward_host(const moe_bf16 *X_host, moe_bf16 *Y_host,
                              moe_bf16 *X_dev, moe_bf16 *Y_dev, const float *Wr,
                              const float *bias, const moe_bf16 *W1, const moe_bf16 *W3,
                              const moe_bf16 *W2, int T, int d, int E, int K, int n,
                              int renorm, void *ws, size_t ws_bytes, void *stream);

/* ---- Token Rounding (SonicMoE page §3): a routing mode whose per-expert row
 * counts are multiples of the tile size M, so grouped GEMM tiles carry no
 * padding rows. Starting from the top-K choice (moe_route):
 *   1. f_e = top-K count of expert e (§3.1);
 *   2. c_e = f_e rounded to the nearest multiple of M, halves up (§3.2), or the
 *      rounded-down multiple when that exceeds T;
 *   3. the second sort (§3.1): expert e keeps the first c_e tokens in the order
 *      (chose e in its top-K first, logit L[t,e] descending, t ascending), so a
 *      rounded-down expert drops its lowest-scoring chosen tokens and a
 *      rounded-up one gains the highest-scoring unchosen tokens;
 *   4. rows grouped by expert, ascending t; row_map[t,e] = row of (t,e) or -1;
 *   5. weights (§3.2): p = softmax(L[t,:]); row_w[row] = p_e / (sum of p over
 *      the experts that kept t) with renorm, else p_e.
 * A token may end with more or fewer than K experts, or none (its output is 0). */

/* Most rows Token Rounding can produce: min(T*E, T*K + E*floor(M/2));
 * -1 for invalid arguments. Size perm_token and row_w with it, and the tile
 * list with capacity/128 + E entries. */
int64_t moe_round_capacity(int T, int E, int K, int M);

/* Workspace bytes of moe_round_routing: the error word (256 bytes) plus the
 * per-expert candidate keys, 4*E*ceil(T/32)*32 bytes. */
size_t moe_round_workspace_bytes(int T, int E);

/* Token Rounding of a top-K routing. logits [T,E] fp32, topk_idx [T,K] and
 * counts [E] exactly as moe_route / moe_route_logits wrote them; 1 <= M <= 65536.
 * Outputs: counts_out [E] (c_e), offsets [E+1], perm_token [capacity]
 * (offsets[E] entries written), row_map [T,E], row_w [capacity], tiles
 * [capacity/128+E][4] int32 = {expert, first row, rows <= 128, 0} (16-byte
 * aligned) and num_tiles [1]. ws: moe_round_workspace_bytes, zeroed once before
 * first use (its first word is the device error word; counts that disagree
 * with topk_idx set MOE_DEVERR_COUNT_MISMATCH and no row is written out of
 * range). Three kernels; no host synchronisation. */
moe_status_t moe_round_routing(const float *logits, const int32_t *topk_idx,
                               const int32_t *counts, int T, int E, int K, int M, int renorm,
                               int32_t *counts_out, int32_t *offsets, int32_t *perm_token,
                               int32_t *row_map, float *row_w, int32_t *tiles,
                               int32_t *num_tiles, void *ws, size_t ws_bytes, void *stream);

/* Combine under a row map: Y[t,:] = bf16( sum over e = 0..E-1 ascending with
 * 0 <= row_map[t,e] < rows of Z[row_map[t,e],:] ), fp32 accumulation, one
 * rounding; a token with no row gets zeros. Z [rows,d] bf16, Y [T,d] bf16. */
moe_status_t moe_combine_rows(const moe_bf16 *Z, const int32_t *row_map, int T, int E, int d,
                              int64_t rows, moe_bf16 *Y, void *stream);

/* Workspace bytes of moe_forward_rounded for this shape (0 if invalid). */
size_t moe_workspace_bytes_rounded(int T, int d, int E, int K, int n);

/* The whole layer under Token Rounding with M = 128 (the GEMM row tile):
 * route -> round -> gate/up+SwiGLU -> down+row weight -> combine_rows.
 * row_map_out [T,E] may be NULL (kept in the workspace then). The rounded
 * counts, offsets, perm_token and row weights stay in the workspace.
 * Enqueues moe_forward_launches(T, d, E, K, n, 1) kernels (7, 8 or 9 as for
 * moe_forward) and at most one memset; no host synchronisation. */
moe_status_t moe_forward_rounded(const moe_bf16 *X, const float *Wr, const float *bias,
                                 const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2,
                                 int T, int d, int E, int K, int n, int renorm, moe_bf16 *Y,
                                 int32_t *row_map_out, void *ws, size_t ws_bytes, void *stream);

/* moe_forward_rounded recording 6 CUDA events like moe_forward_traced: before
 * the router, then after route, rounding, gate/up GEMM, down GEMM, combine. */
moe_status_t moe_forward_rounded_traced(const moe_bf16 *X, const float *Wr, const float *bias,
                                        const moe_bf16 *W1, const moe_bf16 *W3,
                                        const moe_bf16 *W2, int T, int d, int E, int K, int n,
                                        int renorm, moe_bf16 *Y, int32_t *row_map_out,
                                        void *ws, size_t ws_bytes, void *stream,
                                        void *const *events, int n_events);

/* A sequence of n_batches layer forwards straight from host memory, with the
 * copies overlapped with the layer: X_host / Y_host are [n_batches, T, d] bf16
 * (host, pinned for the copies to overlap); X_dev2 / Y_dev2 are caller-owned
 * device buffers [2, T, d] (double buffered). Batch i is uploaded on
 * h2d_stream while the layer runs batch i-1 on `stream`, and its output is
 * downloaded on d2h_stream while the layer runs batch i+1; events order the
 * reuse of each device buffer. The three streams must be distinct. Returns
 * after every output has reached Y_host (it waits for all three streams). */
moe_status_t moe_forward_host_stream(const moe_bf16 *X_host, moe_bf16 *Y_host, int n_batches,
                                     moe_bf16 *X_dev2, moe_bf16 *Y_dev2, const float *Wr,
                                     const float *bias, const moe_bf16 *W1, const moe_bf16 *W3,
                                     const moe_bf16 *W2, int T, int d, int E, int K, int n,
                                     int renorm, void *ws, size_t ws_bytes, void *stream,
                                     void *h2d_stream, void *d2h_stream);

/* Failure-detection self-test: enqueues one CTA that waits, through the same
 * bounded wait as the GEMM pipelines, on a barrier nothing arrives at. After
 * the wait limit (about 1 s) it sets MOE_DEVERR_TIMEOUT in the workspace's
 * error word and exits; moe_sync_check then returns MOE_ERR_DEVICE_TIMEOUT and
 * the context stays usable. ws: any workspace of >= 64 bytes. */
moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, void *stream);

/* Wait for `stream`, read and clear the workspace's device error word.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_CHECK (or
 * MOE_ERR_CUDA); *word_out (may be NULL) receives the raw bits. */
moe_status_t moe_sync_check(void *ws, void *stream, uint32_t *word_out);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
