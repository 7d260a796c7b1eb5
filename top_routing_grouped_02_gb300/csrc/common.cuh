// Internal declarations shared by the CUDA translation units of libmoe.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Rows per expert tile of the grouped GEMMs (the UMMA M dimension).
constexpr int kTileM = 128;
// Largest supported expert count and top-K.
constexpr int kMaxE = 256;
constexpr int kMaxK = 8;
// Rows per token kept in the compact per-token row list of the Token Rounding
// forward (a token with more falls back to its row_map entries).
constexpr int kTokCap = 16;
// Largest Token Rounding tile size accepted.
constexpr int kMaxRoundM = 1 << 16;
// Tokens per grouping chunk (one warp, one bit per token).
constexpr int kChunk = 32;
// One-kernel grouping: at most this many blocks (all resident at once), each of
// at most kGroupMaxCpb chunks; larger T takes the three-kernel grouping.
constexpr int kGroupMaxBlocks = 64;
constexpr int kGroupMaxCpb = 32;

// Byte offsets of the workspace regions for one layer shape (all 256-aligned).
struct WsLayout {
    size_t err;         // uint32 error word + control words (64 B)
    size_t group_flags; // uint32 [kGroupMaxBlocks] one-kernel grouping: block flags (fixed offset)
    size_t group_agg;   // int32 [kGroupMaxBlocks * E] one-kernel grouping: block counts
    size_t counts;      // int32 [E]
    size_t offsets;     // int32 [E+1]
    size_t tile_base;   // int32 [E+1]
    size_t totals;      // int32 [E]   per-expert recount (grouping)
    size_t chunk_base;  // int32 [E * nchunks]
    size_t rank;        // int32 [R]
    size_t perm_token;  // int32 [R]
    size_t perm_slot;   // int32 [R]
    size_t row_of_slot; // int32 [R]
    size_t topk_idx;    // int32 [R]
    size_t topk_w;      // fp32  [R]
    size_t tiles;       // int32 [max_tiles][4]
    size_t num_tiles;   // int32 [1]
    size_t grouping_end;// end of the grouping regions (what moe_permute needs)
    size_t dep;         // uint32 [max_tiles] row-tile counters of the fused expert MLP
    size_t xg;          // bf16  [R, d]  gathered rows (CTA-pair gate/up GEMM)
    size_t h;           // bf16  [R, n]
    size_t z;           // bf16  [R, d]
    size_t logits;      // fp32  [T, E] router logits (moe_forward only)
    size_t counts_round;// int32 [E]    Token Rounding counts (rounded layout only)
    size_t row_map;     // int32 [T, E] Token Rounding rows (rounded layout only)
    size_t row_w;       // fp32  [R]    Token Rounding row weights (rounded layout only)
    size_t round_scratch; // Token Rounding candidate keys (rounded layout only)
    size_t tok_rows;    // int32 [T, kTokCap] compact per-token rows (rounded layout only)
    size_t tok_n;       // int32 [T] (rounded layout only)
    size_t total;
    size_t rows;        // row capacity R of the grouped buffers
    int nchunks;
    int max_tiles;
};

// Control words at the start of the workspace (uint32 each): the error word,
// the grouping scan's ticket, the fused expert MLP's launch epoch and
// ticket (its row-tile counters carry the epoch, so they need no clearing),
// and the router backward's column-sum ticket (zeroed by the kernel before it).
enum : int { kWordErr = 0, kWordDone = 1, kWordEpoch = 2, kWordTicket = 3, kWordGroupEpoch = 4,
             kWordGroupTicket = 5, kWordColTicket = 6 };

WsLayout ws_layout(int T, int d, int E, int K, int n);
// Layout for the Token Rounding forward: grouped buffers sized for the largest
// rounded row count, plus row_map, row_w and the rounding scratch.
WsLayout ws_layout_rounded(int T, int d, int E, int K, int n);
// Most rows Token Rounding with tile size M can produce.
int64_t round_capacity(int T, int E, int K, int M);
// Workspace bytes the rounding kernel needs besides its outputs.
size_t round_scratch_bytes(int T, int E);

// ---- launchers (each returns the CUDA error of its launch) -----------------
cudaError_t launch_route(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T,
                         int d, int E, int K, int renorm, float *logits, int32_t *idx, float *w,
                         int32_t *counts, cudaStream_t s);
// Whether launch_route runs one kernel (logits and selection together) for
// this shape and router-weight alignment; otherwise two.
bool route_is_one_kernel(int d, int E, bool wr16);
cudaError_t launch_router_logits(const __nv_bfloat16 *X, const float *Wr, const float *bias,
                                 int T, int d, int E, float *L, cudaStream_t s);
cudaError_t launch_route_logits(const float *logits, int T, int E, int K, int renorm,
                                int32_t *idx, float *w, int32_t *counts, cudaStream_t s);
// Kernels launch_permute enqueues: 1 for T <= 65536 (the one-kernel grouping),
// else 3.
int permute_launch_count(int T);
cudaError_t launch_permute(const int32_t *idx, const int32_t *counts_in, int T, int E, int K,
                           int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                           int32_t *row_of_slot, int32_t *tiles, int32_t *num_tiles,
                           const WsLayout &L, char *ws, cudaStream_t s, bool one_kernel = true);
// Rows p < min(R, *rows_used) (rows_used: device, nullable); a token index out of
// range gives a zero row and sets MOE_DEVERR_BAD_EXPERT in *err.
cudaError_t launch_gather_rows(const __nv_bfloat16 *X, const int32_t *perm_token, int T, int R,
                               const int32_t *rows_used, int d, __nv_bfloat16 *Xg, uint32_t *err,
                               cudaStream_t s);
// xg: scratch [R, d] for the gathered rows (used when the CTA-pair kernel runs)
cudaError_t launch_gemm_gate_up(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                                const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                                const int32_t *offsets, int R, int d, int E, int n,
                                __nv_bfloat16 *H, __nv_bfloat16 *xg, uint32_t *err,
                                cudaStream_t s);
// The gate/up GEMM that also stores the pre-activations A1 = x W1[e] and
// A3 = x W3[e] (fp32 [R, n] each) beside H.
cudaError_t launch_gemm_gate_up_train(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                                      const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                                      const int32_t *offsets, int R, int d, int E, int n,
                                      __nv_bfloat16 *H, float *A1, float *A3,
                                      __nv_bfloat16 *xg, uint32_t *err, cudaStream_t s);
// Backward dH: dA1, dA3 [R, n] bf16 and dS [R] fp32 from dY [T, d], W2 and the
// pre-activations; xg: scratch [R, d] bf16 for the gathered dY rows (CTA-pair
// path), dspart: scratch [R, n/32] fp32 (n % 256 == 0).
cudaError_t launch_backward_dh(const __nv_bfloat16 *dY, const int32_t *perm_token, int T,
                               const __nv_bfloat16 *W2, const float *A1,
                               const float *A3, const float *topk_w,
                               const int32_t *perm_slot, const int32_t *offsets, int R, int d,
                               int E, int n, __nv_bfloat16 *dA1, __nv_bfloat16 *dA3,
                               __nv_bfloat16 *xg, float *dspart, float *dS, uint32_t *err,
                               cudaStream_t s);
// Backward dX: dXg [R, d] = dA1 W1[e]^T + dA3 W3[e]^T (bf16), then
// dX [T, d] = sum over k of dXg[row_of_slot[t*K + k]] (the combine).
cudaError_t launch_backward_dx(const __nv_bfloat16 *dA1, const __nv_bfloat16 *dA3,
                               const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                               const int32_t *offsets, const int32_t *row_of_slot, int T, int K,
                               int R, int d, int E, int n, __nv_bfloat16 *dXg,
                               __nv_bfloat16 *dX, uint32_t *err, cudaStream_t s);
// Router backward (backward.cu): dL [T, E], dbias [E], dWr [d, E] (fp32) and
// dX [T, d] = bf16(sum_k dXg[row_of_slot[t*K+k]] + dL Wr^T), with `scratch`
// (T * d floats) for the partial sums of dWr and, on the tensor-core path with
// a second scratch region (nullable), the fp32 router share dL Wr^T.
cudaError_t launch_backward_router(const __nv_bfloat16 *X, const float *Wr, const float *L,
                                   const int32_t *idx, const float *dS,
                                   const int32_t *row_of_slot, int T, int d, int E, int K,
                                   int renorm, const __nv_bfloat16 *dXg, float *dL, float *dWr,
                                   float *dbias, float *scratch, char *scratch2,
                                   size_t scratch2_bytes, __nv_bfloat16 *dX, uint32_t *err,
                                   cudaStream_t s);
// dWr partials on the tensor cores: P[c][j][col] = sum over the tokens t of chunk c
// of X[t][j] dLc[t][col] (fp32 [nchunks*d, 2E]), chunk c = tokens offsets[c] ..
// offsets[c+1] - 1 (multiples of 64); dLc [T, 2E] bf16. E % 128 == 0, d % 128 == 0.
// The router's share dXr [T, d] fp32 = (dLh + dLl)(Wrh + Wrl)^T on the tensor
// cores: dLc = [dLh | dLl] [T, 2E], WrA = [Wrh | Wrh], WrB = [Wrl | Wrl] [d, 2E]
// bf16; offsets = {0, T}. 2E % 64 == 0, d % 256 == 0.
cudaError_t launch_router_dx_tc(const __nv_bfloat16 *dLc, const __nv_bfloat16 *WrA,
                                const __nv_bfloat16 *WrB, const int32_t *offsets, int T, int d,
                                int E, float *dXr, uint32_t *err, cudaStream_t s);
cudaError_t launch_router_dwr_tc(const __nv_bfloat16 *X, const __nv_bfloat16 *dLc,
                                 const int32_t *offsets, int T, int d, int E, int nchunks,
                                 float *P, uint32_t *err, cudaStream_t s);
// Rows of src gathered into the padded grouped layout of the weight gradients
// (each expert's rows from a 64-row boundary, zeros after them), optionally
// scaled by w[perm_slot[p]]; poff [E+1] receives (or, offsets_done, holds) the
// padded offsets. dst: [cap, d] with cap >= R + 64*E.
cudaError_t launch_gather_padded(const __nv_bfloat16 *src, const int32_t *perm_token, int T,
                                 const int32_t *offsets, int E, int d, const float *w,
                                 const int32_t *perm_slot, int64_t R, int64_t cap,
                                 int32_t *poff, __nv_bfloat16 *dst, bool offsets_done,
                                 cudaStream_t s);
// Weight gradients: dW1, dW3 [E, d, n] and dW2 [E, n, d] (fp32). pad: scratch
// [R + 64*E, d] bf16, poff: scratch [E+1].
cudaError_t launch_backward_dw(const __nv_bfloat16 *X, const __nv_bfloat16 *dY,
                               const __nv_bfloat16 *H, const __nv_bfloat16 *dA1,
                               const __nv_bfloat16 *dA3, const float *topk_w,
                               const int32_t *perm_token, const int32_t *perm_slot,
                               const int32_t *offsets, int T, int R, int d, int E, int n,
                               float *dW1, float *dW3, float *dW2, __nv_bfloat16 *pad,
                               int32_t *poff, uint32_t *err, cudaStream_t s);
cudaError_t launch_gemm_down(const __nv_bfloat16 *H, const __nv_bfloat16 *W2,
                             const float *topk_w, const int32_t *perm_slot,
                             const int32_t *offsets, int R, int d, int E, int n,
                             __nv_bfloat16 *Z, uint32_t *err, cudaStream_t s);
// Both expert GEMMs, H then Z. With small n (and the single-CTA variant) one
// persistent kernel runs the units of both (see gemm.cu), which needs the
// workspace's control words (err points at them) and dep [max_tiles];
// otherwise launch_gemm_gate_up then launch_gemm_down.
cudaError_t launch_expert_mlp(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                              const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                              const __nv_bfloat16 *W2, const float *topk_w,
                              const int32_t *perm_slot, const int32_t *offsets, int R, int d,
                              int E, int n, __nv_bfloat16 *H, __nv_bfloat16 *Z,
                              __nv_bfloat16 *xg, uint32_t *dep, uint32_t *err, cudaStream_t s);
// Whether launch_expert_mlp runs the fused kernel for this shape, and whether
// the gate/up GEMM runs on CTA pairs (after a separate row gather).
bool use_fused_mlp(int R, int d, int E, int n);
bool gemm_uses_pair(int R, int E);
cudaError_t launch_combine(const __nv_bfloat16 *Z, const int32_t *row_of_slot, int T, int K,
                           int d, __nv_bfloat16 *Y, cudaStream_t s);

// Token Rounding of a top-K routing (rounding.cu): rounded counts, grouped
// offsets, perm_token, row_map [T,E], row weights and the 128-row tile list.
cudaError_t launch_round(const float *L, const int32_t *idx, const int32_t *counts, int T, int E,
                         int K, int M, int renorm, int32_t *counts_out, int32_t *offsets,
                         int32_t *perm_token, int32_t *row_map, float *row_w, int32_t *tiles,
                         int32_t *num_tiles, int32_t *tok_rows, int32_t *tok_n, void *scratch,
                         uint32_t *err, cudaStream_t s);
// Y[t] = sum of Z[row_map[t,e]] over e ascending (rows >= rows_cap are skipped);
// tok_rows [T][kTokCap] / tok_n [T] (nullable) list each token's rows compactly.
cudaError_t launch_combine_rows(const __nv_bfloat16 *Z, const int32_t *row_map,
                                const int32_t *tok_rows, const int32_t *tok_n, int T, int E,
                                int d, int64_t rows_cap, __nv_bfloat16 *Y, cudaStream_t s);

// One CTA whose pipeline wait on a barrier nothing arrives at runs out after the
// wait limit (about 1 s) and sets MOE_DEVERR_TIMEOUT in *err.
cudaError_t launch_wait_timeout_selftest(uint32_t *err, cudaStream_t s);

// ---- programmatic dependent launch ------------------------------------------
// Kernels of the path are launched so that each may start (and run the setup
// that touches no global memory) while its predecessor on the stream finishes.
// Every such kernel calls pdl_wait() before its first global-memory access, which
// returns once the predecessor grid has completed and its writes are visible
// (at once for a launch without the attribute), then pdl_trigger(), which lets
// its own dependent be scheduled. A dependent launches only after every CTA of
// its predecessor is resident, so waiting CTAs never block their predecessor.
// MOE_PDL=0 in the environment launches them in plain stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count();
// Unique id of the CUDA context current on this thread (never reused, unlike a
// context handle); false when there is none yet or the driver cannot say.
bool current_context_id(unsigned long long *id);
// Raises the kernel's dynamic shared-memory limit to `bytes` in the current
// context. Remembered per (kernel, context), so each context gets it once;
// safe to call from several host threads.
cudaError_t ensure_dynamic_smem(const void *kernel, int bytes);
// MOE_OK when the current device is sm_103 (cached per device), MOE_ERR_ARCH
// otherwise, MOE_ERR_CUDA when the device cannot be queried. Clears a CUDA error
// left pending by an earlier, unrelated call first.
moe_status_t check_arch();

}  // namespace moe
