// Router backward: the gradient reaching the router logits, the router weights
// and bias, and the router's share of the input gradient.
//
// Pages: "混合专家模型(MoE)架构优化与SonicMoE实践" §2.2 (the routing scores'
// gradient dS computed with dH; from it the gradient of the scores' softmax) and
// §3.2 (the kept scores renormalised); "Triton优化MoE模型：topk_gating算子融合实战"
// §2.1 (softmax over a token's expert scores).
//
// With the top-K choice of each token fixed, p = softmax(L[t,:]) over all E
// experts, kept = sum of p over the K chosen experts and w_k = p_k / kept
// (renorm) or p_k; dS_k is the gradient of w_k (moe_backward_dh, one value per
// grouped row). Then, per token:
//   g_e  = (dS_k - sum_k' w_k' dS_k') / kept  for e = idx[t,k] (renorm), dS_k
//          without renormalisation, 0 for unchosen experts
//   dL_e = p_e (g_e - sum_e' p_e' g_e')          (the softmax's backward)
// and over the batch: dbias = sum_t dL[t,:], dWr = X^T dL, and the router's
// share of dX is dL Wr^T, added to the experts' share in the final combine.
//
// All deterministic (fixed summation orders, no atomics):
//  1. dl:       one warp per token (lane l holds experts l, l+32, ...); on the
//               tensor-core path it also writes dL's bf16 split.
//  2. dbias:    column sums per chunk of tokens (t ascending, coalesced rows),
//               then the chunks in ascending order by the last block.
//  3. dWr:      per chunk of tokens, fp32 fma chains over the chunk's tokens in
//               ascending order; then the chunks' partials added in ascending
//               order (no second kernel when a single chunk covers T).
//  4. combine:  dX[t,:] = bf16( sum over k ascending of dXg[row_of_slot[t,k],:]
//               (fp32) + (dL Wr^T)[t,:] ), one rounding, with dL Wr^T one fma
//               chain over e ascending per element, computed in the kernel.
// For E % 128 == 0, T % 1024 == 0 and d % 256 == 0, steps 3 and 4 run on the
// tensor cores instead: dL (and Wr) split into bf16 high and low parts, dWr as
// the weight-gradient GEMM over 1024-token chunks plus a fixed-order reduce,
// and (given a second scratch region) dL Wr^T as the dX GEMM with fp32
// outputs, which combine_add_kernel adds to the experts' rows.
#include <algorithm>

#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kDlThreads = 256;

// Also zeroes the column sums' ticket and, given dLc, writes dL's bf16 high and
// low parts beside it (dLc[t][e] = bf16(dL), dLc[t][E + e] = bf16(dL - high))
// and the token chunks' offsets c * chunk (c <= nchunks) for the tensor-core dWr.
template <int NPL>
__global__ void __launch_bounds__(kDlThreads)
router_dl_kernel(const float *__restrict__ L, const int32_t *__restrict__ idx,
                 const float *__restrict__ dS, const int32_t *__restrict__ row_of_slot, int T,
                 int E, int K, int renorm, int64_t R, float *__restrict__ dL,
                 uint32_t *__restrict__ ticket, __nv_bfloat16 *__restrict__ dLc,
                 int32_t *__restrict__ coff, int nchunks, int chunk) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) *ticket = 0u;
        if (dLc != nullptr && (int)threadIdx.x <= nchunks) coff[threadIdx.x] = threadIdx.x * chunk;
    }
    const int64_t t = (int64_t)blockIdx.x * (kDlThreads / 32) + warp;
    if (t >= T) return;
    const float *lt = L + t * E;
    float v[NPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(lt + e) : -INFINITY;
        m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float p[NPL], z = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        p[i] = lane + 32 * i < E ? expf(v[i] - m) : 0.f;
        z += p[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
    for (int i = 0; i < NPL; ++i) p[i] = p[i] / z;
    // the K chosen experts: their probabilities and weight gradients (every lane)
    int ek[kMaxK];
    float pk[kMaxK], sk[kMaxK];
    float kept = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        ek[k] = -1;
        pk[k] = 0.f;
        sk[k] = 0.f;
        if (k < K) {
            const int e = __ldg(idx + t * K + k);
            const int64_t row = __ldg(row_of_slot + t * K + k);
            if (e >= 0 && e < E) {
                ek[k] = e;
                pk[k] = expf(__ldg(lt + e) - m) / z;
                sk[k] = (row >= 0 && row < R) ? __ldg(dS + row) : 0.f;
            }
            kept += pk[k];
        }
    }
    float sw = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
        if (k < K) sw += (renorm ? pk[k] / kept : pk[k]) * sk[k];
    float g[NPL], mean = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        g[i] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k)
            if (k < K && ek[k] == e) g[i] = renorm ? (sk[k] - sw) / kept : sk[k];
        mean += p[i] * g[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mean += __shfl_xor_sync(0xffffffffu, mean, o);
    float *out = dL + t * E;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float v = p[i] * (g[i] - mean);
            out[e] = v;
            if (dLc != nullptr) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                dLc[t * 2 * E + e] = hi;
                dLc[t * 2 * E + E + e] = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));
            }
        }
    }
}

// dbias[e] = sum over t of dL[t, e] in a fixed order. Block (g, c) takes
// columns 32g..32g+31 of token chunk c: warp w adds the chunk's tokens w, w + 8,
// ... in ascending order (a warp reads 32 neighbouring columns of a row at once),
// then the 8 warps are added in order into part[c][e]. With one chunk that is
// dbias itself; otherwise the last block to finish (a ticket, zeroed by the
// kernel before this one) adds the chunks in ascending c. Either way the
// result does not depend on which block finishes when.
constexpr int kColThreads = 256;
__global__ void __launch_bounds__(kColThreads)
col_sum_kernel(const float *__restrict__ dL, int T, int E, int tc, float *__restrict__ part,
               uint32_t *__restrict__ ticket, float *__restrict__ dbias) {
    pdl_wait();
    pdl_trigger();
    __shared__ float ws[kColThreads / 32][32];
    __shared__ bool last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 32 + lane;
    const int64_t t0 = (int64_t)blockIdx.y * tc, t1 = std::min<int64_t>(T, t0 + tc);
    float s = 0.f;
    if (e < E) {
        // (unrolled so that several rows' loads are in flight; the adds keep their order)
#pragma unroll 8
        for (int64_t t = t0 + warp; t < t1; t += kColThreads / 32) s += __ldg(dL + t * E + e);
    }
    ws[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && e < E) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kColThreads / 32; ++w) v += ws[w][lane];
        if (gridDim.y == 1) dbias[e] = v;
        else part[(int64_t)blockIdx.y * E + e] = v;
    }
    if (gridDim.y == 1) return;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int ee = threadIdx.x; ee < E; ee += kColThreads) {
        float v = 0.f;
        for (int c = 0; c < (int)gridDim.y; ++c) v += __ldcg(part + (int64_t)c * E + ee);
        dbias[ee] = v;
    }
    if (threadIdx.x == 0) *ticket = 0u;
}

// dWr[j, e] = sum over t of x[t, j] dL[t, e], in two fixed orders: chunk c of
// TC tokens gives the partial P[c][j][e], one fma chain over its tokens in
// ascending order; dwr_reduce_kernel adds the partials in ascending c. (With
// one chunk the partial is dWr itself.) A thread holds JPT = 64 / EB
// consecutive j and EB experts; block: 128 threads, i.e. JB = 128 * JPT
// columns j; grid (j blocks, chunks, expert blocks of EB). The chunk's tokens
// go through shared memory in stages of ST tokens (ST x JB bf16 of X = 16 KB,
// and ST x EB of dL), copied by cp.async into two buffers, the next stage's
// copies in flight while the current one is used: per token a thread reads its
// JPT x values (one conflict-free load), EB/4 broadcast loads of dL, 64 fmas.
constexpr int kPThreads = 128;
template <int EB>
struct DwrCfg {
    static constexpr int JPT = 64 / EB;
    static constexpr int JB = kPThreads * JPT;
    static constexpr int ST = 8192 / JB;               // tokens per stage
    static constexpr int XBYTES = ST * JB * 2;         // 16 KB
    static constexpr int LBYTES = ST * EB * 4;
    static constexpr int SMEM = 2 * (XBYTES + LBYTES);
};
template <int EB>
__global__ void __launch_bounds__(kPThreads)
router_dwr_part_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ dL, int T,
                       int d, int E, int TC, float *__restrict__ P) {
    using C = DwrCfg<EB>;
    constexpr int JPT = C::JPT, ST = C::ST;
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t dsm[];
    const int tid = threadIdx.x;
    const int jb0 = blockIdx.x * C::JB;
    const int j0 = jb0 + tid * JPT;
    const int e0 = blockIdx.z * EB;
    const int64_t tb = (int64_t)blockIdx.y * TC;
    const int64_t te = min((int64_t)T, tb + TC);
    const int nst = (int)((te - tb + ST - 1) / ST);
    const uint32_t sbase = ptx::smem_addr(dsm);
    auto xbuf = [&](int b) { return sbase + b * (C::XBYTES + C::LBYTES); };
    // stage k's copies: rows tb + k*ST + r (zeros past te), columns jb0.. of X in
    // 16-byte chunks (zeros past d), and dL's EB experts from e0 (zeros past E)
    auto issue = [&](int k) {
        const int64_t t0 = tb + (int64_t)k * ST;
        const uint32_t xs = xbuf(k & 1), ls = xs + C::XBYTES;
        constexpr int XCH = ST * C::JB / 8;
        for (int q = tid; q < XCH; q += kPThreads) {
            const int r = q / (C::JB / 8), c = q % (C::JB / 8);
            const int64_t t = t0 + r;
            const int j = jb0 + c * 8;
            const bool ok = t < te && j < d;
            ptx::cp_async_16_zfill(xs + q * 16, ok ? X + t * d + j : X, ok);
        }
        for (int q = tid; q < ST * EB; q += kPThreads) {
            const int r = q / EB, ee = q % EB;
            const int64_t t = t0 + r;
            const bool ok = t < te && e0 + ee < E;
            ptx::cp_async_4_zfill(ls + q * 4, ok ? dL + t * E + e0 + ee : dL, ok);
        }
        ptx::cp_async_commit_group();
    };
    float acc[JPT][EB];
#pragma unroll
    for (int a = 0; a < JPT; ++a)
#pragma unroll
        for (int b = 0; b < EB; ++b) acc[a][b] = 0.f;
    if (nst > 0) issue(0);
    for (int k = 0; k < nst; ++k) {
        if (k + 1 < nst) {
            issue(k + 1);
            ptx::cp_async_wait_group<1>();
        } else {
            ptx::cp_async_wait_group<0>();
        }
        __syncthreads();
        const uint8_t *xs = dsm + (k & 1) * (C::XBYTES + C::LBYTES);
        const float *ls = reinterpret_cast<const float *>(xs + C::XBYTES);
        const int tn = (int)min((int64_t)ST, te - (tb + (int64_t)k * ST));
        if (j0 < d) {
#pragma unroll 2
            for (int tt = 0; tt < tn; ++tt) {
                float xv[JPT];
                const uint8_t *xp = xs + (tt * C::JB + tid * JPT) * 2;
                if constexpr (JPT == 8) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(xp);
                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 f = __bfloat1622float2(h[u]);
                        xv[2 * u] = f.x;
                        xv[2 * u + 1] = f.y;
                    }
                } else if constexpr (JPT == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(xp);
                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const float2 f = __bfloat1622float2(h[u]);
                        xv[2 * u] = f.x;
                        xv[2 * u + 1] = f.y;
                    }
                } else {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(xp));
                    xv[0] = f.x;
                    xv[1] = f.y;
                }
#pragma unroll
                for (int b4 = 0; b4 < EB; b4 += 4) {
                    const float4 l = *reinterpret_cast<const float4 *>(ls + tt * EB + b4);
                    const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                    for (int a = 0; a < JPT; ++a)
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            acc[a][b4 + b] = __fmaf_rn(xv[a], lv[b], acc[a][b4 + b]);
                }
            }
        }
        __syncthreads();  // the buffer is refilled by the issue two stages on
    }
    if (j0 >= d) return;  // d % 8 == 0: j0 < d means all JPT columns exist
    float *out = P + (int64_t)blockIdx.y * d * E;
#pragma unroll
    for (int a = 0; a < JPT; ++a)
#pragma unroll
        for (int b = 0; b < EB; ++b)
            if (e0 + b < E) out[(int64_t)(j0 + a) * E + e0 + b] = acc[a][b];
}

// dWr[i] = sum over chunks c ascending of P[c][i], i < d * E.
__global__ void __launch_bounds__(256)
dwr_reduce_kernel(const float *__restrict__ P, int64_t n, int chunks, float *__restrict__ dWr) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= n) return;
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) s = __fadd_rn(s, __ldg(P + c * n + i));
    dWr[i] = s;
}

// Wr split the same way for the router's share on the tensor cores:
// WrA[j] = [high | high], WrB[j] = [low | low] ([d, 2E] bf16), so that the
// 4E-long reduction over [dLh | dLl] gives (dLh + dLl)(high + low). Block 0
// also writes the one-group offsets {0, T}.
__global__ void __launch_bounds__(256)
wr_split_kernel(const float *__restrict__ Wr, int d, int E, int T, __nv_bfloat16 *__restrict__ WrA,
                __nv_bfloat16 *__restrict__ WrB, int32_t *__restrict__ off2) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (blockIdx.x == 0 && threadIdx.x < 2) off2[threadIdx.x] = threadIdx.x == 0 ? 0 : T;
    if (i >= (int64_t)d * E) return;
    const int64_t j = i / E;
    const int e = (int)(i - j * E);
    const float v = __ldg(Wr + i);
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(v, __bfloat162float(hi)));
    WrA[j * 2 * E + e] = hi;
    WrA[j * 2 * E + E + e] = hi;
    WrB[j * 2 * E + e] = lo;
    WrB[j * 2 * E + E + e] = lo;
}

// dX[t, :] = bf16( sum over k ascending of dXg[row_of_slot[t*K+k], :] (fp32) +
// dXr[t, :] ), one rounding: a warp per token, 8 columns per lane and step.
constexpr int kCThreads = 256;
__global__ void __launch_bounds__(kCThreads)
combine_add_kernel(const __nv_bfloat16 *__restrict__ dXg, const int32_t *__restrict__ row_of_slot,
                   const float *__restrict__ dXr, int T, int K, int d, int64_t R,
                   __nv_bfloat16 *__restrict__ dX) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * (kCThreads / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    int rows[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        rows[k] = -1;
        if (k < K) {
            const int r = __ldg(row_of_slot + t * K + k);
            rows[k] = (r >= 0 && r < R) ? r : -1;
        }
    }
    for (int c = lane; c < d / 8; c += 32) {
        uint4 raw[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k)
            raw[k] = rows[k] >= 0
                         ? __ldg(reinterpret_cast<const uint4 *>(dXg + (int64_t)rows[k] * d) + c)
                         : make_uint4(0, 0, 0, 0);
        const float4 a = __ldg(reinterpret_cast<const float4 *>(dXr + t * d) + 2 * c);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(dXr + t * d) + 2 * c + 1);
        float acc[8] = {};
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (rows[k] < 0) continue;
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw[k]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                acc[2 * u] = __fadd_rn(acc[2 * u], f.x);
                acc[2 * u + 1] = __fadd_rn(acc[2 * u + 1], f.y);
            }
        }
        const float add[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint4 out;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            o2[u] = __floats2bfloat162_rn(__fadd_rn(acc[2 * u], add[2 * u]),
                                          __fadd_rn(acc[2 * u + 1], add[2 * u + 1]));
        reinterpret_cast<uint4 *>(dX + t * d)[c] = out;
    }
}

// dWr[j][e] = sum over chunks c ascending of (P[c][j][e] + P[c][j][E + e]): the
// token chunks' partial products with the high and low parts, fixed order.
__global__ void __launch_bounds__(256)
dwr_reduce_halves_kernel(const float *__restrict__ P, int d, int E, int chunks,
                         float *__restrict__ dWr) {
    pdl_wait();
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= (int64_t)d * E) return;
    const int64_t j = i / E;
    const int e = (int)(i - j * E);
    float s = 0.f;
    for (int c = 0; c < chunks; ++c) {
        const float *row = P + ((int64_t)c * d + j) * 2 * E;
        s = __fadd_rn(s, __fadd_rn(__ldg(row + e), __ldg(row + E + e)));
    }
    dWr[i] = s;
}

// The router's share of dX computed in the final combine, for any E. Block: 8
// warps of 8 tokens (64 tokens) x 256 columns (8 per lane). Experts go in
// chunks of 32: Wr's 256 x 32 slice staged transposed in shared memory and
// dL's 64 x 32 slice as [e][token], by cp.async into two buffers (the next
// chunk's copies in flight while the current one is used). For each output,
// r = one fma chain over e ascending of dL[t,e] Wr[j,e]; then
// dX = bf16((sum over k ascending of the token's dXg rows, fp32) + r), one
// rounding. Per expert a warp reads 8 Wr values per lane and 8 dL values (two
// broadcast loads) for 64 fmas. Grid: (token blocks, column blocks).
constexpr int kFTok = 64, kFCols = 256, kFE = 32, kFWrLd = kFCols + 4, kFLLd = kFTok + 4;
constexpr int kFTpw = kFTok / 8;  // tokens per warp
constexpr int kFBufFloats = kFE * kFWrLd + kFE * kFLLd;  // one chunk's Wr and dL slices
constexpr int kFSmem = 2 * kFBufFloats * 4;
__global__ void __launch_bounds__(256, 2)
combine_router_kernel(const __nv_bfloat16 *__restrict__ dXg,
                      const int32_t *__restrict__ row_of_slot, const float *__restrict__ dL,
                      const float *__restrict__ Wr, int T, int K, int d, int E, int64_t R,
                      __nv_bfloat16 *__restrict__ dX) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) float fsm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = blockIdx.y * kFCols;
    const int64_t t0 = (int64_t)blockIdx.x * kFTok;
    const int j = c0 + lane * 8;
    // chunk k's copies into buffer k & 1: Wr[c0 + jj, e0 + ee] at ws[ee][jj] and
    // dL[t0 + tt, e0 + ee] at ls[ee][tt] (zeros outside), 4-byte cp.async with
    // consecutive threads on consecutive experts (coalesced reads)
    auto issue = [&](int k) {
        const int e0 = k * kFE;
        float *ws = fsm + (k & 1) * kFBufFloats, *ls = ws + kFE * kFWrLd;
        for (int q = tid; q < kFCols * kFE; q += 256) {
            const int jj = q / kFE, ee = q % kFE;
            const bool ok = c0 + jj < d && e0 + ee < E;
            ptx::cp_async_4_zfill(ptx::smem_addr(ws + ee * kFWrLd + jj),
                                  ok ? Wr + (int64_t)(c0 + jj) * E + e0 + ee : Wr, ok);
        }
        for (int q = tid; q < kFTok * kFE; q += 256) {
            const int tt = q / kFE, ee = q % kFE;
            const bool ok = t0 + tt < T && e0 + ee < E;
            ptx::cp_async_4_zfill(ptx::smem_addr(ls + ee * kFLLd + tt),
                                  ok ? dL + (t0 + tt) * E + e0 + ee : dL, ok);
        }
        ptx::cp_async_commit_group();
    };
    float r[kFTpw][8];
#pragma unroll
    for (int a = 0; a < kFTpw; ++a)
#pragma unroll
        for (int u = 0; u < 8; ++u) r[a][u] = 0.f;
    const int nch = (E + kFE - 1) / kFE;
    issue(0);
    for (int k = 0; k < nch; ++k) {
        if (k + 1 < nch) {
            issue(k + 1);
            ptx::cp_async_wait_group<1>();
        } else {
            ptx::cp_async_wait_group<0>();
        }
        __syncthreads();
        const float *ws = fsm + (k & 1) * kFBufFloats, *ls = ws + kFE * kFWrLd;
        const int en = min(kFE, E - k * kFE);
        if (j < d) {
            for (int ee = 0; ee < en; ++ee) {
                const float4 w0 = *reinterpret_cast<const float4 *>(ws + ee * kFWrLd + lane * 8);
                const float4 w1 = *reinterpret_cast<const float4 *>(ws + ee * kFWrLd + lane * 8 + 4);
                const float4 l0 = *reinterpret_cast<const float4 *>(ls + ee * kFLLd + warp * kFTpw);
                const float4 l1 = *reinterpret_cast<const float4 *>(ls + ee * kFLLd + warp * kFTpw + 4);
                const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                const float lv[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
#pragma unroll
                for (int a = 0; a < kFTpw; ++a)
#pragma unroll
                    for (int u = 0; u < 8; ++u) r[a][u] = __fmaf_rn(lv[a], wv[u], r[a][u]);
            }
        }
        __syncthreads();  // the buffer is refilled by the issue two chunks on
    }
    if (j >= d) return;
    // the experts' rows, four tokens at a time: their k-th rows in flight at once
#pragma unroll
    for (int h = 0; h < kFTpw; h += 4) {
        float acc[4][8];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[a][u] = 0.f;
        for (int k = 0; k < K; ++k) {
            uint4 raw[4];
            bool ok[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int64_t t = t0 + warp * kFTpw + h + a;
                const int row = t < T ? __ldg(row_of_slot + t * K + k) : -1;
                ok[a] = row >= 0 && row < R;
                raw[a] = ok[a] ? __ldg(reinterpret_cast<const uint4 *>(dXg + (int64_t)row * d + j))
                               : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (!ok[a]) continue;
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw[a]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = __bfloat1622float2(h2[u]);
                    acc[a][2 * u] = __fadd_rn(acc[a][2 * u], f.x);
                    acc[a][2 * u + 1] = __fadd_rn(acc[a][2 * u + 1], f.y);
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int64_t t = t0 + warp * kFTpw + h + a;
            if (t >= T) break;
            uint4 out;
            __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                o2[u] = __floats2bfloat162_rn(__fadd_rn(acc[a][2 * u], r[h + a][2 * u]),
                                              __fadd_rn(acc[a][2 * u + 1], r[h + a][2 * u + 1]));
            *reinterpret_cast<uint4 *>(dX + t * d + j) = out;
        }
    }
}

// Padded row offsets of the weight gradients: each expert's rows rounded up to
// a multiple of 64; poff[E] is the padded total. One block (E <= 256).
__global__ void __launch_bounds__(256)
pad_offsets_kernel(const int32_t *__restrict__ offsets, int E, int32_t *__restrict__ poff) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t c[kMaxE];
    const int e = threadIdx.x;
    if (e < E) {
        const int32_t n = offsets[e + 1] - offsets[e];
        c[e] = n > 0 ? (n + 63) / 64 * 64 : 0;
    }
    __syncthreads();
    if (e == 0) {
        int32_t acc = 0;
        for (int i = 0; i < E; ++i) {
            poff[i] = acc;
            acc += c[i];
        }
        poff[E] = acc;
    }
}

// dst[q] for padded rows q < poff[E]: the source row of grouped row
// p = offsets[e] + (q - poff[e]) (src[perm_token[p]], times w[perm_slot[p]]
// when w is given, rounded to bf16 once), or zeros past the expert's rows. One
// warp per row; indices out of range give a zero row. The block first copies
// poff into shared memory, so each warp's search over the experts costs no
// global round trips.
__global__ void __launch_bounds__(256)
gather_pad_kernel(const __nv_bfloat16 *__restrict__ src, const int32_t *__restrict__ perm_token,
                  int T, const int32_t *__restrict__ offsets, const int32_t *__restrict__ poff,
                  int E, int d, const float *__restrict__ w, const int32_t *__restrict__ perm_slot,
                  int64_t R, int64_t cap, __nv_bfloat16 *__restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t spoff[kMaxE + 1];
    for (int i = threadIdx.x; i <= E; i += blockDim.x) spoff[i] = __ldg(poff + i);
    __syncthreads();
    const int64_t q = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= cap || q >= spoff[E]) return;
    int lo = 0, hi = E - 1;  // the last expert whose padded rows start at or before q
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (spoff[mid] <= q) lo = mid; else hi = mid - 1;
    }
    const int64_t local = q - spoff[lo];
    const int64_t p = (int64_t)__ldg(offsets + lo) + local;
    bool ok = local < (int64_t)__ldg(offsets + lo + 1) - __ldg(offsets + lo) && p >= 0 && p < R;
    int64_t t = ok ? __ldg(perm_token + p) : -1;
    ok = ok && t >= 0 && t < T;
    float scale = 1.f;
    if (ok && w != nullptr) {
        const int32_t slot = __ldg(perm_slot + p);
        ok = slot >= 0 && slot < R;
        scale = ok ? __ldg(w + slot) : 0.f;
    }
    uint4 *out = reinterpret_cast<uint4 *>(dst + q * d);
    for (int c = lane; c < d / 8; c += 32) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (ok) {
            v = __ldg(reinterpret_cast<const uint4 *>(src + t * d) + c);
            if (w != nullptr) {
                __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = __bfloat1622float2(h2[u]);
                    h2[u] = __floats2bfloat162_rn(scale * f.x, scale * f.y);
                }
            }
        }
        out[c] = v;
    }
}

}  // namespace

namespace {
template <int EB>
cudaError_t launch_dwr_part(const __nv_bfloat16 *X, const float *dL, int T, int d, int E, int TC,
                            int chunks, float *part, cudaStream_t s) {
    using C = DwrCfg<EB>;
    {
        const cudaError_t e =
            ensure_dynamic_smem(reinterpret_cast<const void *>(router_dwr_part_kernel<EB>), C::SMEM);
        if (e != cudaSuccess) return e;
    }
    return launch_k(router_dwr_part_kernel<EB>,
                    dim3((d + C::JB - 1) / C::JB, chunks, (E + EB - 1) / EB), dim3(kPThreads),
                    C::SMEM, s, X, dL, T, d, E, TC, part);
}
cudaError_t launch_combine_router(const __nv_bfloat16 *dXg, const int32_t *row_of_slot,
                                  const float *dL, const float *Wr, int T, int K, int d, int E,
                                  int64_t R, __nv_bfloat16 *dX, cudaStream_t s) {
    {
        const cudaError_t e =
            ensure_dynamic_smem(reinterpret_cast<const void *>(combine_router_kernel), kFSmem);
        if (e != cudaSuccess) return e;
    }
    return launch_k(combine_router_kernel,
                    dim3((unsigned)((T + kFTok - 1) / kFTok), (d + kFCols - 1) / kFCols),
                    dim3(256), kFSmem, s, dXg, row_of_slot, dL, Wr, T, K, d, E, R, dX);
}
}  // namespace

cudaError_t launch_gather_padded(const __nv_bfloat16 *src, const int32_t *perm_token, int T,
                                 const int32_t *offsets, int E, int d, const float *w,
                                 const int32_t *perm_slot, int64_t R, int64_t cap,
                                 int32_t *poff, __nv_bfloat16 *dst, bool offsets_done,
                                 cudaStream_t s) {
    if (!offsets_done) {
        cudaError_t e = launch_k(pad_offsets_kernel, dim3(1), dim3(256), 0, s, offsets, E, poff);
        if (e != cudaSuccess) return e;
    }
    return launch_k(gather_pad_kernel, dim3((unsigned)((cap + 7) / 8)), dim3(256), 0, s, src,
                    perm_token, T, offsets, static_cast<const int32_t *>(poff), E, d, w, perm_slot,
                    R, cap, dst);
}

cudaError_t launch_backward_router(const __nv_bfloat16 *X, const float *Wr, const float *L,
                                   const int32_t *idx, const float *dS,
                                   const int32_t *row_of_slot, int T, int d, int E, int K,
                                   int renorm, const __nv_bfloat16 *dXg, float *dL, float *dWr,
                                   float *dbias, float *scratch, char *scratch2,
                                   size_t scratch2_bytes, __nv_bfloat16 *dX, uint32_t *err,
                                   cudaStream_t s) {
    const int64_t R = (int64_t)T * K;
    // On the tensor cores where the shape allows: dWr with chunks of 1024 tokens as
    // the weight-gradient GEMM's groups (partials [chunk][d][2E] fp32, then dL's
    // split [T][2E] bf16, written with dL, and the chunk offsets); and, given the
    // second scratch region, the router's share dXr = dL Wr^T (fp32 [T, d] in the
    // first scratch, Wr's split and the offsets {0, T} in the second) for a
    // combine that adds it.
    const int tc_chunk = 1024;
    const int tc_chunks = T / tc_chunk;
    const size_t tc_part = (size_t)tc_chunks * d * 2 * E * 4;
    const size_t tc_split = (size_t)T * 2 * E * 2;
    const size_t tc_off = 16 * (size_t)((tc_chunks + 1 + 3) / 4);
    const size_t tc_wr = (size_t)d * 2 * E * 2;
    const bool tc_shape = E % 128 == 0 && T % tc_chunk == 0 && d % 256 == 0 && tc_chunks >= 1 &&
                          tc_chunks <= 255;
    const bool tc_dx = tc_shape && scratch2 != nullptr &&
                       tc_part + tc_split + tc_off + 2 * tc_wr + 16 <= scratch2_bytes;
    const bool tc = tc_shape && (tc_dx || tc_part + tc_split + tc_off <= (size_t)T * d * 4);
    char *base = tc_dx ? scratch2 : reinterpret_cast<char *>(scratch);
    float *P = reinterpret_cast<float *>(base);
    __nv_bfloat16 *dLc = tc ? reinterpret_cast<__nv_bfloat16 *>(base + tc_part) : nullptr;
    int32_t *coff = reinterpret_cast<int32_t *>(base + tc_part + tc_split);
    uint32_t *ticket = err + kWordColTicket;

    const unsigned tb = (unsigned)((T + kDlThreads / 32 - 1) / (kDlThreads / 32));
    auto dl = E <= 32    ? router_dl_kernel<1>
              : E <= 64  ? router_dl_kernel<2>
              : E <= 128 ? router_dl_kernel<4>
                         : router_dl_kernel<8>;
    cudaError_t e = launch_k(dl, dim3(tb), dim3(kDlThreads), 0, s, L, idx, dS, row_of_slot, T, E, K,
                             renorm, R, dL, ticket, dLc, coff, tc_chunks, tc_chunk);
    if (e != cudaSuccess) return e;
    // dbias: chunks of about 128 tokens (at most 256, their partials in the
    // scratch region while the column sums run)
    const int64_t cmax = std::max<int64_t>(1, std::min<int64_t>(256, (int64_t)T * d / E));
    const int cch = (int)std::min<int64_t>(cmax, (T + 127) / 128);
    const int ctc = (T + cch - 1) / cch;
    e = launch_k(col_sum_kernel, dim3((unsigned)((E + 31) / 32), (unsigned)cch), dim3(kColThreads),
                 0, s, static_cast<const float *>(dL), T, E, ctc, scratch, ticket, dbias);
    if (e != cudaSuccess) return e;
    if (tc) {
        e = launch_router_dwr_tc(X, dLc, coff, T, d, E, tc_chunks, P, err, s);
        if (e != cudaSuccess) return e;
        const int64_t m = (int64_t)d * E;
        e = launch_k(dwr_reduce_halves_kernel, dim3((unsigned)((m + 255) / 256)), dim3(256), 0, s,
                     static_cast<const float *>(P), d, E, tc_chunks, dWr);
        if (e != cudaSuccess) return e;
        if (!tc_dx) return launch_combine_router(dXg, row_of_slot, dL, Wr, T, K, d, E, R, dX, s);
        __nv_bfloat16 *WrA = reinterpret_cast<__nv_bfloat16 *>(base + tc_part + tc_split + tc_off);
        __nv_bfloat16 *WrB = WrA + (size_t)d * 2 * E;
        int32_t *off2 = reinterpret_cast<int32_t *>(WrB + (size_t)d * 2 * E);
        e = launch_k(wr_split_kernel, dim3((unsigned)((m + 255) / 256)), dim3(256), 0, s, Wr, d, E,
                     T, WrA, WrB, off2);
        if (e != cudaSuccess) return e;
        e = launch_router_dx_tc(dLc, WrA, WrB, off2, T, d, E, scratch, err, s);
        if (e != cudaSuccess) return e;
        return launch_k(combine_add_kernel,
                        dim3((unsigned)((T + kCThreads / 32 - 1) / (kCThreads / 32))),
                        dim3(kCThreads), 0, s, dXg, row_of_slot, static_cast<const float *>(scratch),
                        T, K, d, R, dX);
    }
    // dWr on the FP32 pipe: chunks of TC tokens, their partials in the scratch
    // region (T * d floats; TC grows until the chunks' d x E partials fit), then
    // the reduce
    int64_t TC = 32;
    while (TC < T && (((T + TC - 1) / TC) * E > T || (T + TC - 1) / TC > 65535)) TC *= 2;
    TC = std::min<int64_t>(TC, T);
    const int chunks = (int)((T + TC - 1) / TC);
    float *part = chunks > 1 ? scratch : dWr;
    if (E <= 8)
        e = launch_dwr_part<8>(X, dL, T, d, E, (int)TC, chunks, part, s);
    else if (E <= 16)
        e = launch_dwr_part<16>(X, dL, T, d, E, (int)TC, chunks, part, s);
    else
        e = launch_dwr_part<32>(X, dL, T, d, E, (int)TC, chunks, part, s);
    if (e != cudaSuccess) return e;
    if (chunks > 1) {
        const int64_t n = (int64_t)d * E;
        e = launch_k(dwr_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                     static_cast<const float *>(part), n, chunks, dWr);
        if (e != cudaSuccess) return e;
    }
    // the router's share dL Wr^T and the final combine, in one kernel
    return launch_combine_router(dXg, row_of_slot, dL, Wr, T, K, d, E, R, dX, s);
}

}  // namespace moe
