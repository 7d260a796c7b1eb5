// Router: logits -> softmax -> top-K -> renormalised weights -> per-expert counts.
//
// Pages: "Triton优化MoE模型：topk_gating算子融合实战" §2.1 (one fused pass: logits,
// online softmax, local top-k, cross-warp merge, output), §2.2 (max-subtracted
// softmax and top-2 in one kernel), §4.1 (subtract the maximum first), §4.2
// (per-expert counts with atomics, bucketed); "混合专家模型(MoE)架构优化与SonicMoE实践"
// §1 (E scores per token, keep the best K), §3.2 (renormalise the kept scores);
// "Triton GPU 内核编程实战：用 Python 写高性能 AI 推理算子" §5.2 (the online softmax
// recurrence m_new = max(m_old, .), l_new = e^(m_old-m_new) l_old + sum e^(s-m_new)).
//
// Logits are computed as a register-tiled SIMT product: every (token, expert)
// accumulator is one fp32 fused multiply-add chain over j = 0..d-1 in ascending
// order from +0.0f, followed by one fp32 add of the bias. That order is the
// definition the results are pinned to, so the logits (and hence the top-K
// indices) are bit-identical to a sequential evaluation. The chain cannot be
// split across threads or tensor-core instructions without changing the
// rounding, so the kernel keeps whole chains per thread and gets its
// parallelism from tokens x experts.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBK = 32;  // reduction steps staged in shared memory per pass

// Block / thread tiling of the logit product for a padded expert count EP.
template <int EP>
struct RouterTile {
    static constexpr bool kNarrow = EP <= 32;
    static constexpr int TE = kNarrow ? EP / 8 : 8;          // experts per thread
    static constexpr int TX = EP / TE;                        // threads along experts
    static constexpr int TY = kThreads / TX;                  // threads along tokens
    static constexpr int TT = kNarrow ? 1 : (EP >= 128 ? 4 : 2);  // tokens per thread
    static constexpr int BT = TY * TT;                        // tokens per block
    static constexpr int WTX = kNarrow ? 8 : 4;               // warp shape (experts)
    static constexpr int WTY = 32 / WTX;                      // warp shape (tokens)
    static constexpr int NWX = TX / WTX;                      // warps along experts
    static constexpr int LS = EP + 4;                         // logit row stride (smem)
    static constexpr size_t kStageFloats = (size_t)kBK * BT + (size_t)kBK * EP;
    static constexpr size_t kLogitFloats = (size_t)BT * LS;
    static constexpr size_t kSmemFloats = kStageFloats > kLogitFloats ? kStageFloats : kLogitFloats;
    static_assert(TX * TY == kThreads, "tiling");
    static_assert(TX % WTX == 0 && TY % WTY == 0, "warp tiling");
};

__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
    // higher score wins; equal scores: lower expert index wins
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Softmax + top-K + weights + histogram for one token whose E logits are held
// by the warp: lane l owns experts l, l+32, ... (NPL per lane; -inf padding).
template <int NPL>
__device__ __forceinline__ void select_topk_warp(float (&v)[NPL], int E, int K, int renorm,
                                                 int64_t t, int32_t *idx_out, float *w_out,
                                                 int *hist) {
    const int lane = threadIdx.x & 31;
    // online softmax statistics (max, sum of exp) per lane, merged across the warp
    float m = -INFINITY, s = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        if (e < E) {
            float mn = fmaxf(m, v[i]);
            s = s * __expf(m - mn) + __expf(v[i] - mn);
            m = mn;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float mo = __shfl_xor_sync(0xffffffffu, m, off);
        float so = __shfl_xor_sync(0xffffffffu, s, off);
        float mn = fmaxf(m, mo);
        float a = (m == -INFINITY) ? 0.f : s * expf(m - mn);
        float b = (mo == -INFINITY) ? 0.f : so * expf(mo - mn);
        s = a + b;
        m = mn;
    }
    bool taken[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) taken[i] = (lane + 32 * i) >= E;
    int sel_idx[kMaxK];
    float sel_val[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                int e = lane + 32 * i;
                if (!taken[i] && better(v[i], e, bv, bi)) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (lane + 32 * i == bi) taken[i] = true;
            sel_idx[k] = bi;
            sel_val[k] = bv;
        }
    }
    // weights: exp(L_k - max) over the kept sum (renormalised) or the full sum
    const float mtop = sel_val[0];
    float kept = 0.f;
    float ex[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
            ex[k] = expf(sel_val[k] - mtop);
            kept += ex[k];
        }
    }
    const float full = s * expf(m - mtop);  // m == mtop; kept for clarity
    const float denom = renorm ? kept : full;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K && lane == k) {
            idx_out[t * K + k] = sel_idx[k];
            w_out[t * K + k] = ex[k] / denom;
            atomicAdd(&hist[sel_idx[k]], 1);
        }
    }
}

template <int EP>
__global__ void __launch_bounds__(kThreads)
router_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ Wr,
              const float *__restrict__ bias, int T, int d, int E, int K, int renorm,
              int32_t *__restrict__ idx_out, float *__restrict__ w_out,
              int32_t *__restrict__ counts) {
    using C = RouterTile<EP>;
    extern __shared__ __align__(16) float smem[];
    __shared__ int hist[EP];
    float *xs = smem;                    // [kBK][BT]  x values, j-major
    float *ws = smem + kBK * C::BT;      // [kBK][EP]  router weights
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wx = warp % C::NWX, wy = warp / C::NWX;
    const int tx = wx * C::WTX + lane % C::WTX;
    const int ty = wy * C::WTY + lane / C::WTX;
    const int64_t t0 = (int64_t)blockIdx.x * C::BT;

    for (int e = tid; e < EP; e += kThreads) hist[e] = 0;

    float acc[C::TT][C::TE];
#pragma unroll
    for (int a = 0; a < C::TT; ++a)
#pragma unroll
        for (int b = 0; b < C::TE; ++b) acc[a][b] = 0.f;

    for (int j0 = 0; j0 < d; j0 += kBK) {
        const int jn = min(kBK, d - j0);
        // stage x: BT tokens x jn columns (8 bf16 per 16-byte load), transposed
        for (int q = tid; q < C::BT * (kBK / 8); q += kThreads) {
            const int tt = q / (kBK / 8), c8 = (q % (kBK / 8)) * 8;
            const int64_t t = t0 + tt;
            float f[8];
            if (t < T && c8 < jn) {
                uint4 raw = *reinterpret_cast<const uint4 *>(X + t * d + j0 + c8);
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float2 p = __bfloat1622float2(h2[u]);
                    f[2 * u] = p.x;
                    f[2 * u + 1] = p.y;
                }
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) f[u] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) xs[(c8 + u) * C::BT + tt] = f[u];
        }
        // stage Wr rows j0..j0+jn-1 (zero padding for experts >= E)
        for (int q = tid; q < kBK * EP; q += kThreads) {
            const int jj = q / EP, e = q % EP;
            ws[q] = (jj < jn && e < E) ? __ldg(Wr + (int64_t)(j0 + jj) * E + e) : 0.f;
        }
        __syncthreads();
        if (jn == kBK) {
#pragma unroll 8
            for (int jj = 0; jj < kBK; ++jj) {
                float xv[C::TT], wv[C::TE];
#pragma unroll
                for (int a = 0; a < C::TT; ++a) xv[a] = xs[jj * C::BT + ty * C::TT + a];
#pragma unroll
                for (int b = 0; b < C::TE; ++b) wv[b] = ws[jj * EP + tx * C::TE + b];
#pragma unroll
                for (int a = 0; a < C::TT; ++a)
#pragma unroll
                    for (int b = 0; b < C::TE; ++b) acc[a][b] = __fmaf_rn(xv[a], wv[b], acc[a][b]);
            }
        } else {
            for (int jj = 0; jj < jn; ++jj) {
                float xv[C::TT], wv[C::TE];
#pragma unroll
                for (int a = 0; a < C::TT; ++a) xv[a] = xs[jj * C::BT + ty * C::TT + a];
#pragma unroll
                for (int b = 0; b < C::TE; ++b) wv[b] = ws[jj * EP + tx * C::TE + b];
#pragma unroll
                for (int a = 0; a < C::TT; ++a)
#pragma unroll
                    for (int b = 0; b < C::TE; ++b) acc[a][b] = __fmaf_rn(xv[a], wv[b], acc[a][b]);
            }
        }
        __syncthreads();
    }

    // logits tile -> shared memory, bias added as one fp32 add
    float *ls = smem;  // [BT][LS]
#pragma unroll
    for (int a = 0; a < C::TT; ++a)
#pragma unroll
        for (int b = 0; b < C::TE; ++b) {
            const int e = tx * C::TE + b;
            float v = acc[a][b];
            if (bias != nullptr && e < E) v = __fadd_rn(v, __ldg(bias + e));
            ls[(ty * C::TT + a) * C::LS + e] = v;
        }
    __syncthreads();

    constexpr int NPL = EP >= 32 ? EP / 32 : 1;
    for (int tt = warp; tt < C::BT; tt += kThreads / 32) {
        const int64_t t = t0 + tt;
        if (t >= T) break;
        float v[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? ls[tt * C::LS + e] : -INFINITY;
        }
        select_topk_warp<NPL>(v, E, K, renorm, t, idx_out, w_out, hist);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads)
        if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
}

// Router from given logits: one warp per token row.
template <int NPL>
__global__ void __launch_bounds__(kThreads)
router_logits_kernel(const float *__restrict__ logits, int T, int E, int K, int renorm,
                     int32_t *__restrict__ idx_out, float *__restrict__ w_out,
                     int32_t *__restrict__ counts) {
    __shared__ int hist[kMaxE];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < kMaxE; e += kThreads) hist[e] = 0;
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * (kThreads / 32) + warp;
    if (t < T) {
        float v[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? __ldg(logits + t * E + e) : -INFINITY;
        }
        select_topk_warp<NPL>(v, E, K, renorm, t, idx_out, w_out, hist);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads)
        if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
}

template <int EP>
cudaError_t launch_router_ep(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T,
                             int d, int E, int K, int renorm, int32_t *idx, float *w,
                             int32_t *counts, cudaStream_t s) {
    using C = RouterTile<EP>;
    const size_t smem = C::kSmemFloats * sizeof(float);
    cudaError_t err = cudaFuncSetAttribute(router_kernel<EP>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int blocks = (T + C::BT - 1) / C::BT;
    router_kernel<EP><<<blocks, kThreads, smem, s>>>(X, Wr, bias, T, d, E, K, renorm, idx, w,
                                                     counts);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T,
                         int d, int E, int K, int renorm, int32_t *idx, float *w,
                         int32_t *counts, uint32_t *err, cudaStream_t s) {
    (void)err;
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
    if (E <= 8) return launch_router_ep<8>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
    if (E <= 16) return launch_router_ep<16>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
    if (E <= 32) return launch_router_ep<32>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
    if (E <= 64) return launch_router_ep<64>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
    if (E <= 128) return launch_router_ep<128>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
    return launch_router_ep<256>(X, Wr, bias, T, d, E, K, renorm, idx, w, counts, s);
}

cudaError_t launch_route_logits(const float *logits, int T, int E, int K, int renorm,
                                int32_t *idx, float *w, int32_t *counts, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
    const int blocks = (T + kThreads / 32 - 1) / (kThreads / 32);
    if (E <= 32)
        router_logits_kernel<1><<<blocks, kThreads, 0, s>>>(logits, T, E, K, renorm, idx, w, counts);
    else if (E <= 64)
        router_logits_kernel<2><<<blocks, kThreads, 0, s>>>(logits, T, E, K, renorm, idx, w, counts);
    else if (E <= 128)
        router_logits_kernel<4><<<blocks, kThreads, 0, s>>>(logits, T, E, K, renorm, idx, w, counts);
    else
        router_logits_kernel<8><<<blocks, kThreads, 0, s>>>(logits, T, E, K, renorm, idx, w, counts);
    return cudaGetLastError();
}

}  // namespace moe
