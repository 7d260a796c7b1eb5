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
// Five kernels, all deterministic (fixed summation orders, no atomics):
//  1. dl:       one warp per token (lane l holds experts l, l+32, ...).
//  2. dbias:    one block per expert, a fixed-shape tree over the tokens.
//  3. dWr:      64 (j) x 32 (e) output tiles; each output is one fp32 fma
//               chain over t ascending, operands staged through shared memory.
//  4. dL Wr^T:  32 (t) x 64 (j) output tiles; one fma chain over e ascending.
//  5. combine:  dX[t,:] = bf16( sum over k ascending of dXg[row_of_slot[t,k],:]
//               (fp32) + (dL Wr^T)[t,:] ), one rounding.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kDlThreads = 256;

template <int NPL>
__global__ void __launch_bounds__(kDlThreads)
router_dl_kernel(const float *__restrict__ L, const int32_t *__restrict__ idx,
                 const float *__restrict__ dS, const int32_t *__restrict__ row_of_slot, int T,
                 int E, int K, int renorm, int64_t R, float *__restrict__ dL) {
    pdl_wait();
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
        if (e < E) out[e] = p[i] * (g[i] - mean);
    }
}

// dbias[e] = sum over t of dL[t, e]: thread i adds tokens i, i + 256, ...
// (ascending), then a fixed tree over the block's threads.
constexpr int kColThreads = 256;
__global__ void __launch_bounds__(kColThreads)
col_sum_kernel(const float *__restrict__ dL, int T, int E, float *__restrict__ dbias) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[kColThreads];
    const int e = blockIdx.x;
    float s = 0.f;
    for (int64_t t = threadIdx.x; t < T; t += kColThreads) s += __ldg(dL + t * E + e);
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = kColThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) dbias[e] = part[0];
}

// dWr[j, e] = sum over t ascending of x[t, j] dL[t, e] (one fma chain each).
// Block: 64 j x 32 e, 128 threads of 4 x 4 outputs; 32 tokens per stage.
constexpr int kWJ = 64, kWE = 32, kWT = 32;
__global__ void __launch_bounds__(128)
router_dwr_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ dL, int T, int d,
                  int E, float *__restrict__ dWr) {
    pdl_wait();
    pdl_trigger();
    __shared__ float xs[kWT][kWJ];
    __shared__ float ls[kWT][kWE];
    const int tid = threadIdx.x;
    const int jg = tid % 16, eg = tid / 16;  // outputs j0 + 4jg .. +3, e0 + 4eg .. +3
    const int j0 = blockIdx.x * kWJ, e0 = blockIdx.y * kWE;
    float acc[4][4] = {};
    for (int t0 = 0; t0 < T; t0 += kWT) {
        for (int q = tid; q < kWT * kWJ; q += 128) {
            const int tt = q / kWJ, jj = q % kWJ;
            const int64_t t = t0 + tt;
            xs[tt][jj] = (t < T && j0 + jj < d) ? __bfloat162float(X[t * d + j0 + jj]) : 0.f;
        }
        for (int q = tid; q < kWT * kWE; q += 128) {
            const int tt = q / kWE, ee = q % kWE;
            const int64_t t = t0 + tt;
            ls[tt][ee] = (t < T && e0 + ee < E) ? __ldg(dL + t * E + e0 + ee) : 0.f;
        }
        __syncthreads();
        const int tn = min(kWT, T - t0);
        for (int tt = 0; tt < tn; ++tt) {
            float xv[4], lv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) xv[a] = xs[tt][4 * jg + a];
#pragma unroll
            for (int b = 0; b < 4; ++b) lv[b] = ls[tt][4 * eg + b];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = __fmaf_rn(xv[a], lv[b], acc[a][b]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int j = j0 + 4 * jg + a, e = e0 + 4 * eg + b;
            if (j < d && e < E) dWr[(int64_t)j * E + e] = acc[a][b];
        }
}

// dXr[t, j] = sum over e ascending of dL[t, e] Wr[j, e] (one fma chain each).
// Block: 32 t x 64 j, 128 threads of 4 x 4 outputs; 32 experts per stage.
constexpr int kXT = 32, kXJ = 64, kXE = 32;
__global__ void __launch_bounds__(128)
router_dx_kernel(const float *__restrict__ dL, const float *__restrict__ Wr, int T, int d, int E,
                 float *__restrict__ dXr) {
    pdl_wait();
    pdl_trigger();
    __shared__ float ls[kXT][kXE + 1];
    __shared__ float ws[kXJ][kXE + 1];
    const int tid = threadIdx.x;
    const int jg = tid % 16, tg = tid / 16;  // outputs t0 + 4tg .. +3, j0 + 4jg .. +3
    const int64_t t0 = (int64_t)blockIdx.y * kXT;
    const int j0 = blockIdx.x * kXJ;
    float acc[4][4] = {};
    for (int e0 = 0; e0 < E; e0 += kXE) {
        for (int q = tid; q < kXT * kXE; q += 128) {
            const int tt = q / kXE, ee = q % kXE;
            const int64_t t = t0 + tt;
            ls[tt][ee] = (t < T && e0 + ee < E) ? __ldg(dL + t * E + e0 + ee) : 0.f;
        }
        for (int q = tid; q < kXJ * kXE; q += 128) {
            const int jj = q / kXE, ee = q % kXE;
            ws[jj][ee] = (j0 + jj < d && e0 + ee < E) ? __ldg(Wr + (int64_t)(j0 + jj) * E + e0 + ee) : 0.f;
        }
        __syncthreads();
        const int en = min(kXE, E - e0);
        for (int ee = 0; ee < en; ++ee) {
            float lv[4], wv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) lv[a] = ls[4 * tg + a][ee];
#pragma unroll
            for (int b = 0; b < 4; ++b) wv[b] = ws[4 * jg + b][ee];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = __fmaf_rn(lv[a], wv[b], acc[a][b]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int64_t t = t0 + 4 * tg + a;
            const int j = j0 + 4 * jg + b;
            if (t < T && j < d) dXr[t * d + j] = acc[a][b];
        }
}

// dX[t, :] = bf16( sum over k ascending of dXg[row_of_slot[t*K+k], :] + dXr[t, :] ):
// one warp per token, 8 columns per lane and step.
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
        float acc[8] = {};
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (rows[k] < 0) continue;
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(dXg + (int64_t)rows[k] * d) + c);
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                acc[2 * u] = __fadd_rn(acc[2 * u], f.x);
                acc[2 * u + 1] = __fadd_rn(acc[2 * u + 1], f.y);
            }
        }
        const float4 a = __ldg(reinterpret_cast<const float4 *>(dXr + t * d) + 2 * c);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(dXr + t * d) + 2 * c + 1);
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
// warp per row; indices out of range give a zero row.
__global__ void __launch_bounds__(256)
gather_pad_kernel(const __nv_bfloat16 *__restrict__ src, const int32_t *__restrict__ perm_token,
                  int T, const int32_t *__restrict__ offsets, const int32_t *__restrict__ poff,
                  int E, int d, const float *__restrict__ w, const int32_t *__restrict__ perm_slot,
                  int64_t R, int64_t cap, __nv_bfloat16 *__restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const int64_t q = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (q >= cap || q >= __ldg(poff + E)) return;
    int lo = 0, hi = E - 1;  // the last expert whose padded rows start at or before q
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(poff + mid) <= q) lo = mid; else hi = mid - 1;
    }
    const int64_t local = q - __ldg(poff + lo);
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
                                   float *dbias, float *dXr, __nv_bfloat16 *dX, cudaStream_t s) {
    const int64_t R = (int64_t)T * K;
    const unsigned tb = (unsigned)((T + kDlThreads / 32 - 1) / (kDlThreads / 32));
    auto dl = E <= 32    ? router_dl_kernel<1>
              : E <= 64  ? router_dl_kernel<2>
              : E <= 128 ? router_dl_kernel<4>
                         : router_dl_kernel<8>;
    cudaError_t e = launch_k(dl, dim3(tb), dim3(kDlThreads), 0, s, L, idx, dS, row_of_slot, T, E, K,
                             renorm, R, dL);
    if (e != cudaSuccess) return e;
    e = launch_k(col_sum_kernel, dim3(E), dim3(kColThreads), 0, s, static_cast<const float *>(dL), T,
                 E, dbias);
    if (e != cudaSuccess) return e;
    e = launch_k(router_dwr_kernel, dim3((d + kWJ - 1) / kWJ, (E + kWE - 1) / kWE), dim3(128), 0, s,
                 X, static_cast<const float *>(dL), T, d, E, dWr);
    if (e != cudaSuccess) return e;
    e = launch_k(router_dx_kernel, dim3((d + kXJ - 1) / kXJ, (unsigned)((T + kXT - 1) / kXT)),
                 dim3(128), 0, s, static_cast<const float *>(dL), Wr, T, d, E, dXr);
    if (e != cudaSuccess) return e;
    return launch_k(combine_add_kernel, dim3((unsigned)((T + kCThreads / 32 - 1) / (kCThreads / 32))),
                    dim3(kCThreads), 0, s, dXg, row_of_slot, static_cast<const float *>(dXr), T, K,
                    d, R, dX);
}

}  // namespace moe
