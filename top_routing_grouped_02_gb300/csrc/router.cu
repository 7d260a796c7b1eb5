// Router: logits -> softmax -> top-K -> renormalised weights -> per-expert counts.
//
// Pages: "Triton优化MoE模型：topk_gating算子融合实战" §2.1 (logits, online softmax,
// local top-k, cross-warp merge, output), §2.2 (max-subtracted softmax and top-2),
// §4.1 (subtract the maximum first), §4.2 (per-expert counts with atomics,
// bucketed per block); "混合专家模型(MoE)架构优化与SonicMoE实践" §1 (E scores per
// token, keep the best K), §3.2 (renormalise the kept scores); "Triton GPU 内核编程
// 实战：用 Python 写高性能 AI 推理算子" §5.2 (softmax statistics: the maximum
// and the sum of exp(s - max); here the maximum is the top-1 score, so one pass
// over the scores suffices).
//
// Logits: L[t,e] in fp32, then one fp32 add of bias[e]. With E > 32 the sum is
// one fused multiply-add chain over j = 0..d-1 in ascending order from +0.0f;
// with E <= 32 it runs in blocks of 1024 steps, one such chain per block, the
// block sums added in ascending block order (a few-expert router has too few
// (token, expert) chains to hide a d-long dependency). That order is the
// definition the results are pinned to, so L (and hence the top-K indices) is
// bit-identical to a sequential evaluation of it. A chain cannot be split over
// threads or tensor-core instructions without changing the rounding, so every
// chain stays in one thread.
//  - E <= 32 (E % 4 == 0): ONE kernel computes the logits and selects: each
//    lane runs 4 tokens x 2 experts of one 1024-step block (packed FMAs over
//    token pairs, operands from cp.async shared-memory rings), the CTA adds
//    the block sums in order and a thread per token ranks its experts.
//  - E > 32: a logits kernel, then the select kernel below:
//      - two-warp blocks on 32-token x 64-expert tiles, 4 x 8 register
//        micro-tiles fed by conflict-free float4 shared-memory reads;
//      - E >= 128 with many tokens: one 8-warp block per SM, two warps per
//        scheduler, each lane 2*PA or 2*PB tokens x 8 experts with x widened to
//        fp32 pairs once per stage, so the FP32 FMA pipe is the limit.
//  - Select (given logits, or after the E > 32 logits): one warp per token reads its E logits, picks K by repeated warp
//     argmax over order-preserving keys (ties -> lower index), writes indices
//     and weights, and counts per expert in a block histogram flushed with one
//     atomic per (block, expert). The softmax needs no separate maximum pass: the
//     maximum is the first kept score, so the renormalised weights come from the
//     K kept scores alone and the full denominator from one sum of exp(L - max).
//     For small E and T a single block with one thread per token does the same
//     and writes the counts directly, so no memset is needed.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <stdlib.h>

#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
// 8-byte copy, or 8 zero bytes when !ok (the source is then not read)
__device__ __forceinline__ void cp_async8_zfill(void *smem_dst, const void *gmem_src, bool ok) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(d), "l"(gmem_src),
                 "r"(ok ? 8 : 0)
                 : "memory");
}
// 16-byte copy, or 16 zero bytes when !ok (the source is then not read)
__device__ __forceinline__ void cp_async16_zfill(void *smem_dst, const void *gmem_src, bool ok) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(gmem_src),
                 "r"(ok ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// With E <= 32 the logits' reduction runs in blocks of kLogitBlock steps: one
// fma chain per block, the block sums added in ascending block order (with
// d <= kLogitBlock the single chain over j). The E <= 32 kernel's stage length
// divides kLogitBlock.
constexpr int kLogitBlock = 1024;

// ---- E <= 32: logits and selection in one kernel ------------------------------
// Lane (q, p) of a warp owns the chains of 4 tokens (rows q, q + QPW, q + 2QPW,
// q + 3QPW of its token group) x 2 experts (expert pair p) over one 1024-step
// block of the reduction: EP/2 lanes per token quad, so a warp covers TPW =
// 256/EP tokens (32, 16 or 8). A work item is (token group of TPW tokens,
// block); a CTA holds `tg` token groups and all their blocks, its warps taking
// the items in turn, so the blocks of one logit run side by side. Each warp
// streams its item through its own ring of 64-step stages (cp.async): the TPW
// rows of X (bf16, rows padded to 144 bytes) and, per expert pair, the pair's
// 64 weights as (w[j][2p], w[j][2p+1]) rows (padded to 528 bytes). The
// paddings put the rows a warp reads at once in distinct banks, so every load
// address is the lane's base plus a constant. Per 8 steps a lane loads 16
// bytes of x per token and four 128-bit weight words, one 8-step group ahead
// of its use, and issues 4 packed FMAs per step over token pairs (each
// component rounds like __fmaf_rn, so every block sum is one sequential fma
// chain): 16 bytes of operands per 8 FMAs. Steps past d are zero-filled, which
// leaves a chain unchanged (fmaf(0, w, acc) = acc for the +0-started chains).
// At the end the block sums go to shared memory, one thread per token adds
// them in ascending block order, adds the bias, stores the logits and runs the
// selection below on its token, and the CTA's per-expert counts are added into
// counts (zeroed before the launch).
// What bounds it (Mixtral shape, 4096 tokens, d = 4096, E = 8): the definition
// gives 131072 independent chains of 1024 steps, one warp per scheduler at 8
// chains per lane, so each step's operand latency and the packed-FMA dispatch
// (about 10 cycles per step for 4 packed FMAs) are exposed; X streams at about
// half of HBM bandwidth behind them.
// Requires E % 4 == 0, a 16-byte-aligned Wr and at most kRouteMaxBlocks blocks.
constexpr int kRouteJS = 64;         // steps per stage
constexpr int kRouteStages = 4;
constexpr int kRouteMaxBlocks = 32;  // d <= 32768
constexpr int kRouteWarps = 4;       // most warps per CTA

template <int EP>
struct RouteCfg {
    static constexpr int PAIRS = EP / 2;               // lanes per token quad
    static constexpr int QPW = 32 / PAIRS;             // token quads per warp
    static constexpr int TPW = 4 * QPW;                // tokens per warp
    static constexpr int XROW = kRouteJS * 2 + 16;     // x row pitch: 64 bf16 + 16 bytes
    static constexpr int XB = TPW * XROW;              // x rows of a stage
    static constexpr int WROW = kRouteJS * 8 + 16;     // one expert pair's 64 steps + 16 bytes
    static constexpr int WB = PAIRS * WROW;            // weights of a stage
    static constexpr int SB = XB + WB;
    static constexpr int WARP_SMEM = kRouteStages * SB;
    static constexpr int PART = TPW * EP * 4;          // block sums of one item
};

// Selection for one token with its EP scores in registers (entries >= E are
// ignored): the maximum, then K passes (higher score wins, equal scores: lower
// index), weights exp(L_k - max) over their sum (renorm) or over a compensated
// (Kahan) sum of exp(L_e - max) over every expert. Writes idx/w of token t and
// counts the choices in the shared histogram.
template <int EP>
__device__ __forceinline__ void select_token(const float (&v)[EP], int E, int K, int renorm,
                                                 int64_t t, int32_t *__restrict__ idx_out,
                                                 float *__restrict__ w_out, int *hist) {
    float m = v[0];
#pragma unroll
    for (int e = 1; e < EP; ++e)
        if (e < E) m = fmaxf(m, v[e]);
    uint32_t taken = 0;
    int sel[kMaxK];
    float kept = 0.f, ex[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
            int bi = -1;
            float bv = -INFINITY;
#pragma unroll
            for (int e = 0; e < EP; ++e)
                if (e < E && !(taken >> e & 1u) && (bi < 0 || v[e] > bv)) {
                    bv = v[e];
                    bi = e;
                }
            taken |= 1u << bi;
            sel[k] = bi;
            ex[k] = expf(bv - m);
            kept += ex[k];
        }
    }
    float denom = kept;
    if (!renorm) {
        float sum = 0.f, comp = 0.f;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (e < E) {
                const float y = expf(v[e] - m) - comp;
                const float tt = sum + y;
                comp = (tt - sum) - y;
                sum = tt;
            }
        }
        denom = sum;
    }
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
            idx_out[t * K + k] = sel[k];
            w_out[t * K + k] = ex[k] / denom;
            atomicAdd(&hist[sel[k]], 1);
        }
    }
}

template <int EP>
__global__ void __launch_bounds__(32 * kRouteWarps)
route_chain_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ Wr,
                   const float *__restrict__ bias, int T, int d, int E, int K, int renorm,
                   int tg, float *__restrict__ L, int32_t *__restrict__ idx_out,
                   float *__restrict__ w_out, int32_t *__restrict__ counts) {
    using C = RouteCfg<EP>;
    constexpr int TPW = C::TPW;
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char sm[];
    __shared__ int hist[EP];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int nb = (d + kLogitBlock - 1) / kLogitBlock;
    const int items = tg * nb;
    const int64_t tcta = (int64_t)blockIdx.x * tg * TPW;
    unsigned char *ring = sm + warp * C::WARP_SMEM;
    float *part = reinterpret_cast<float *>(sm + nw * C::WARP_SMEM);  // [items][TPW][EP]
    const int q = lane / C::PAIRS, p = lane % C::PAIRS;
    for (int e = threadIdx.x; e < EP; e += blockDim.x) hist[e] = 0;

    for (int it = warp; it < items; it += nw) {
        const int g = it / nb, b = it % nb;
        const int64_t t0 = tcta + (int64_t)g * TPW;
        const int jb = b * kLogitBlock;
        const int len = min(kLogitBlock, d - jb);
        const int nst = (len + kRouteJS - 1) / kRouteJS;
        // stage st of this item into ring slot st % kRouteStages (zero-filled
        // beyond T, d and E)
        auto issue = [&](int st) {
            unsigned char *xs = ring + (st % kRouteStages) * C::SB;
            unsigned char *ws = xs + C::XB;
            const int j0 = jb + st * kRouteJS;
#pragma unroll
            for (int i = 0; i < TPW * 8 / 32; ++i) {
                const int cidx = lane + 32 * i;
                const int r = cidx >> 3, c = cidx & 7;
                const int64_t t = t0 + r;
                const int j = j0 + 8 * c;
                const bool ok = t < T && j < d;
                cp_async16_zfill(xs + r * C::XROW + c * 16, ok ? X + t * d + j : X, ok);
            }
#pragma unroll
            for (int i = 0; i < kRouteJS * C::PAIRS / 32; ++i) {
                const int cidx = lane + 32 * i;
                const int jj = cidx / C::PAIRS, pp = cidx % C::PAIRS;
                const int j = j0 + jj;
                const bool ok = j < d && 2 * pp < E;
                cp_async8_zfill(ws + pp * C::WROW + jj * 8, ok ? Wr + (int64_t)j * E + 2 * pp : Wr, ok);
            }
        };
#pragma unroll
        for (int st = 0; st < kRouteStages - 1; ++st) {
            if (st < nst) issue(st);
            cp_async_commit();
        }
        // chains: a[i][h] = (token pair i of the quad, expert 2p + h)
        float2 a[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) a[i][0] = a[i][1] = make_float2(0.f, 0.f);
        for (int st = 0; st < nst; ++st) {
            cp_async_wait<kRouteStages - 2>();
            __syncwarp();  // stage st landed for every lane; all lanes are past st - 1
            if (st + kRouteStages - 1 < nst) issue(st + kRouteStages - 1);
            cp_async_commit();
            const unsigned char *xs = ring + (st % kRouteStages) * C::SB;
            const unsigned char *xq = xs + q * C::XROW;                  // the lane's first token row
            const unsigned char *wrow = xs + C::XB + p * C::WROW;        // its expert pair's weights
            // 8-step groups: x words of the 4 tokens and 4 weight words, loaded one
            // group ahead of their use
            uint4 xr[2][4];
            float4 wq[2][4];
            auto load = [&](int v, int bs) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    xr[bs][i] = *reinterpret_cast<const uint4 *>(xq + i * C::QPW * C::XROW + v * 16);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    wq[bs][m] = *reinterpret_cast<const float4 *>(wrow + (8 * v + 2 * m) * 8);
            };
            load(0, 0);
#pragma unroll
            for (int v = 0; v < kRouteJS / 8; ++v) {
                const int cb = v & 1;
                if (v + 1 < kRouteJS / 8) load(v + 1, cb ^ 1);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    // word u of a row holds steps 8v + 2u (low half) and 8v + 2u + 1 (high)
                    const uint32_t w0 = (&xr[cb][0].x)[u], w1 = (&xr[cb][1].x)[u];
                    const uint32_t w2v = (&xr[cb][2].x)[u], w3 = (&xr[cb][3].x)[u];
                    const float4 wv4 = wq[cb][u];  // (e0, e1) of step 8v + 2u, then of the next step
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const float e0 = hh ? wv4.z : wv4.x, e1 = hh ? wv4.w : wv4.y;
                        const float2 we0 = make_float2(e0, e0), we1 = make_float2(e1, e1);
                        const float2 x01 =
                            make_float2(__uint_as_float(hh ? (w0 & 0xffff0000u) : (w0 << 16)),
                                        __uint_as_float(hh ? (w1 & 0xffff0000u) : (w1 << 16)));
                        const float2 x23 =
                            make_float2(__uint_as_float(hh ? (w2v & 0xffff0000u) : (w2v << 16)),
                                        __uint_as_float(hh ? (w3 & 0xffff0000u) : (w3 << 16)));
                        a[0][0] = __ffma2_rn(x01, we0, a[0][0]);
                        a[0][1] = __ffma2_rn(x01, we1, a[0][1]);
                        a[1][0] = __ffma2_rn(x23, we0, a[1][0]);
                        a[1][1] = __ffma2_rn(x23, we1, a[1][1]);
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncwarp();  // the ring is free for the warp's next item
        float *pp = part + (size_t)it * TPW * EP;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            // token pair i of the lane: rows q + 2i*QPW and q + (2i+1)*QPW
            const int ta = q + 2 * i * C::QPW, tb = ta + C::QPW;
            pp[ta * EP + 2 * p] = a[i][0].x;
            pp[ta * EP + 2 * p + 1] = a[i][1].x;
            pp[tb * EP + 2 * p] = a[i][0].y;
            pp[tb * EP + 2 * p + 1] = a[i][1].y;
        }
    }
    __syncthreads();
    // one thread per token: block sums in ascending block order, bias, logits,
    // selection
    for (int tau = threadIdx.x; tau < tg * TPW; tau += blockDim.x) {
        const int64_t t = tcta + tau;
        if (t >= T) continue;
        const int g = tau / TPW, tl = tau % TPW;
        float v[EP];
        const float *p0 = part + (size_t)(g * nb) * TPW * EP + tl * EP;
#pragma unroll
        for (int e = 0; e < EP; ++e) v[e] = p0[e];
        for (int b = 1; b < nb; ++b) {
            const float *pb = p0 + (size_t)b * TPW * EP;
#pragma unroll
            for (int e = 0; e < EP; ++e) v[e] = __fadd_rn(v[e], pb[e]);
        }
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            if (e < E) {
                if (bias != nullptr) v[e] = __fadd_rn(v[e], __ldg(bias + e));
                L[t * E + e] = v[e];
            }
        }
        select_token<EP>(v, E, K, renorm, t, idx_out, w_out, hist);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
}

// Fallback for E <= 32 with E % 4 != 0 (or an unaligned Wr): operands straight
// from global memory, one thread per (token, expert).
constexpr int kSmallThreads = 64;

template <int EP>
__global__ void __launch_bounds__(kSmallThreads)
logits_small_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ Wr,
                    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ L) {
    pdl_wait();
    pdl_trigger();
    constexpr int kTok = kSmallThreads / EP;
    const int e = threadIdx.x % EP;
    const int64_t t = (int64_t)blockIdx.x * kTok + threadIdx.x / EP;
    if (t >= T) return;
    const int ec = e < E ? e : E - 1;  // padding lanes compute a copy and store nothing
    const uint4 *xr = reinterpret_cast<const uint4 *>(X + t * d);
    const float *wc = Wr + ec;
    float tot = 0.f, acc = 0.f;  // block sums folded so far; the current block's chain
    const int nv = d / 8;
#pragma unroll 4
    for (int v = 0; v < nv; ++v) {
        const uint4 raw = __ldg(xr + v);
        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
        float w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) w[u] = __ldg(wc + (int64_t)(8 * v + u) * E);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(h2[u]);
            acc = __fmaf_rn(f.x, w[2 * u], acc);
            acc = __fmaf_rn(f.y, w[2 * u + 1], acc);
        }
        if ((8 * (v + 1)) % kLogitBlock == 0 || v + 1 == nv) {  // a block ends here
            tot = 8 * v < kLogitBlock ? acc : __fadd_rn(tot, acc);
            acc = 0.f;
        }
    }
    if (e < E) {
        if (bias != nullptr) tot = __fadd_rn(tot, __ldg(bias + e));
        L[t * E + e] = tot;
    }
}

// ---- E > 32: register-tiled product ------------------------------------------
// Block tile 32 tokens x 64 experts, two warps of 16 tokens each, so a launch
// has ceil(T/32) * ceil(E/64) blocks and about 13 warps per SM at the workload
// sizes (the FP32 pipe needs several warps per scheduler to hide latency). In
// warp w, lane (ty, tx) = (lane / 8, lane % 8) owns tokens 16w + 4ty .. +3 and
// experts {4tx..4tx+3, 32+4tx..32+4tx+3}: per reduction step it reads one
// float4 of x and two float4 of weights, all conflict-free, and issues 16
// packed FMAs over expert pairs (each component rounds exactly like
// __fmaf_rn, so every output is still one sequential fma chain over j).
// 32-step stages are double-buffered: weights by cp.async, x through registers
// (converted to fp32 and transposed on the way into shared memory).
constexpr int kWT = 32;  // tokens per block tile
constexpr int kWE = 64;  // experts per block tile
constexpr int kWK = 32;  // reduction steps per stage
constexpr int kWThreads = 64;

template <bool VEC>
__global__ void __launch_bounds__(kWThreads)
logits_tiled_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ Wr,
                    const float *__restrict__ bias, int T, int d, int E, float *__restrict__ L) {
    pdl_wait();
    pdl_trigger();
    __shared__ __align__(16) float xs[2][kWK][kWT];
    __shared__ __align__(16) float ws[2][kWK][kWE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = lane >> 3, tx = lane & 7;
    const int64_t t0 = (int64_t)blockIdx.x * kWT;
    const int e0 = blockIdx.y * kWE;
    const int nchunk = (d + kWK - 1) / kWK;

    // x: thread tid loads token t0 + (tid & 31), 16 consecutive j from 16*(tid >> 5)
    uint4 xr[2];
    const int xt = tid & 31, xj = 16 * (tid >> 5);
    auto load_x = [&](int c) {
        const int j0 = c * kWK + xj;
        const int64_t t = t0 + xt;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (t < T && j0 + 8 * i < d)
                xr[i] = __ldg(reinterpret_cast<const uint4 *>(X + t * d + j0 + 8 * i));
            else
                xr[i] = make_uint4(0, 0, 0, 0);
        }
    };
    auto store_x = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&xr[i]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                xs[buf][xj + 8 * i + 2 * u][xt] = f.x;
                xs[buf][xj + 8 * i + 2 * u + 1][xt] = f.y;
            }
        }
    };
    // weights: 32 rows j x 64 experts = 512 x 16 B, 8 per thread
    auto issue_w = [&](int c, int buf) {
        const int j0 = c * kWK;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = tid + kWThreads * i;
            const int jj = q >> 4, e4 = (q & 15) * 4;
            const int j = j0 + jj, e = e0 + e4;
            if (j >= d) continue;
            const float *src = Wr + (int64_t)j * E + e;
            if (VEC) {
                if (e < E) cp_async16(&ws[buf][jj][e4], src);
            } else {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e + 0 < E) v.x = __ldg(src + 0);
                if (e + 1 < E) v.y = __ldg(src + 1);
                if (e + 2 < E) v.z = __ldg(src + 2);
                if (e + 3 < E) v.w = __ldg(src + 3);
                *reinterpret_cast<float4 *>(&ws[buf][jj][e4]) = v;
            }
        }
        cp_async_commit();
    };

    // accumulators paired along experts: acc[a][p] = (expert 2p, expert 2p+1) of
    // the lane's 8 experts, for its token a
    float2 acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[a][p] = make_float2(0.f, 0.f);

    const int xo = 16 * warp + 4 * ty;  // the lane's first token within the tile
    issue_w(0, 0);
    load_x(0);
    store_x(0);
    cp_async_wait<0>();
    __syncthreads();
    for (int c = 0; c < nchunk; ++c) {
        const int buf = c & 1;
        if (c + 1 < nchunk) {
            issue_w(c + 1, buf ^ 1);
            load_x(c + 1);
        }
        const int jn = min(kWK, d - c * kWK);
        auto step = [&](int jj) {
            const float4 x0 = *reinterpret_cast<const float4 *>(&xs[buf][jj][xo]);
            const float4 w0 = *reinterpret_cast<const float4 *>(&ws[buf][jj][4 * tx]);
            const float4 w1 = *reinterpret_cast<const float4 *>(&ws[buf][jj][32 + 4 * tx]);
            const float xa[4] = {x0.x, x0.y, x0.z, x0.w};
            const float2 wp[4] = {make_float2(w0.x, w0.y), make_float2(w0.z, w0.w),
                                  make_float2(w1.x, w1.y), make_float2(w1.z, w1.w)};
            // packed fp32 FMA: each component rounds exactly like __fmaf_rn
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const float2 xx = make_float2(xa[a], xa[a]);
#pragma unroll
                for (int p = 0; p < 4; ++p) acc[a][p] = __ffma2_rn(xx, wp[p], acc[a][p]);
            }
        };
        if (jn == kWK) {
#pragma unroll 8
            for (int jj = 0; jj < kWK; ++jj) step(jj);
        } else {
            for (int jj = 0; jj < jn; ++jj) step(jj);
        }
        if (c + 1 < nchunk) {
            store_x(buf ^ 1);
            cp_async_wait<0>();
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t t = t0 + xo + a;
        if (t >= T) continue;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int e = e0 + (b < 4 ? 4 * tx + b : 32 + 4 * tx + b - 4);
            if (e < E) {
                float v = (b & 1) ? acc[a][b >> 1].y : acc[a][b >> 1].x;
                if (bias != nullptr) v = __fadd_rn(v, __ldg(bias + e));
                L[t * E + e] = v;
            }
        }
    }
}

// ---- E >= 128 with many tokens: one block per SM, two warps per scheduler -----
// Block: 8 warps on 16(PA+PB) tokens x 128 experts. Lane (ty, tx) = (lane / 16,
// lane % 16) of warp w owns the tokens of group g = 2w + ty (2PA of them for
// w < 4, 2PB for w >= 4) and experts {4tx..4tx+3, 64+4tx..64+4tx+3}; its
// accumulators are float2 pairs over neighbouring tokens. Warps w and w + 4 share
// a scheduler, so each scheduler carries PA + PB token pairs in two warps: one
// warp's issue slots fill the other's gaps after packed FMAs. Per reduction step
// a lane reads its tokens' x as fp32 pairs (one or two 128-bit loads) and its 8
// weights (two 128-bit loads, conflict-free), and issues 8PA or 8PB packed FMAs;
// each component rounds like __fmaf_rn, so every output is still one sequential
// fma chain over j. 64-step stages, 3 deep, arrive by cp.async (zero-filled
// beyond T, d and E): the weights as [j][e] rows, X as its own [t][j] rows with
// the 16-byte chunks of a row pair XOR-swizzled, which one pass per stage turns
// into the transposed, token-paired fp32 layout the steps read (widening each
// bf16 there once, instead of in every step that reads it).
// PA + PB (4..8) is chosen on the host so that the block count fills the SMs.
constexpr int kBK = 64;        // reduction steps per stage
constexpr int kBE = 128;       // experts per block
constexpr int kBWords = 64;    // pairs in a transposed x row: 16 groups x 4 token pairs
constexpr int kBStages = 3;
constexpr int kBThreads = 256;
constexpr int kBWBytes = kBK * kBE * 4;        // weight stage: 32 KB
constexpr int kBXBytes = 2 * kBWords * kBK * 2;  // raw X stage (up to 128 rows): 16 KB
constexpr int kBStage = kBWBytes + kBXBytes;
constexpr int kBXsBytes = kBK * kBWords * 8;   // transposed x, fp32 pairs: 32 KB
constexpr int kBSmem = kBStages * kBStage + 2 * kBXsBytes;


// jn reduction steps of one stage for a lane with N token pairs (acc[0..N-1])
template <int N, int PMAX, bool FULL>
__device__ __forceinline__ void big_steps(float2 (&acc)[PMAX][8], const float2 *xs,
                                          const float *w, int jn) {
    auto step = [&](int jj) {
        const float4 xa = *reinterpret_cast<const float4 *>(xs + jj * kBWords);
        float4 xb = xa;
        if (N > 2) xb = *reinterpret_cast<const float4 *>(xs + jj * kBWords + 2);
        const float4 w0 = *reinterpret_cast<const float4 *>(w + jj * kBE);
        const float4 w1 = *reinterpret_cast<const float4 *>(w + jj * kBE + 64);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const float2 xq[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w),
                              make_float2(xb.x, xb.y), make_float2(xb.z, xb.w)};
        float2 xp[N];
#pragma unroll
        for (int i = 0; i < N; ++i) xp[i] = xq[i];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const float2 ww = make_float2(wv[b], wv[b]);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i][b] = __ffma2_rn(xp[i], ww, acc[i][b]);
        }
    };
    if (FULL) {
#pragma unroll 4
        for (int jj = 0; jj < kBK; ++jj) step(jj);
    } else {
        for (int jj = 0; jj < jn; ++jj) step(jj);
    }
}

template <int PA, int PB>
__global__ void __launch_bounds__(kBThreads, 1)
logits_big_kernel(const __nv_bfloat16 *__restrict__ X, const float *__restrict__ Wr,
                  const float *__restrict__ bias, int T, int d, int E, float *__restrict__ L) {
    static_assert(PA >= PB && PA <= 4 && PB >= 1, "token pairs per lane");
    pdl_wait();
    pdl_trigger();
    constexpr int kTok = 16 * (PA + PB);  // tokens per block
    extern __shared__ __align__(16) uint8_t big_smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = lane >> 4, tx = lane & 15;
    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int e0 = blockIdx.y * kBE;
    const int nchunk = (d + kBK - 1) / kBK;

    auto stage_w = [&](int c) {
        return reinterpret_cast<float *>(big_smem + (c % kBStages) * kBStage);
    };
    auto stage_x = [&](int c) { return big_smem + (c % kBStages) * kBStage + kBWBytes; };
    auto xs_of = [&](int c) {
        return reinterpret_cast<float2 *>(big_smem + kBStages * kBStage + (c & 1) * kBXsBytes);
    };

    auto issue = [&](int c) {
        if (c < nchunk) {
            const int j0 = c * kBK;
            float *w = stage_w(c);
#pragma unroll
            for (int i = 0; i < kBK * 32 / kBThreads; ++i) {
                const int q = tid + kBThreads * i;
                const int jj = q >> 5, ch = q & 31;
                const int j = j0 + jj, e = e0 + 4 * ch;
                const bool ok = j < d && e < E;
                cp_async16_zfill(w + jj * kBE + 4 * ch, ok ? Wr + (int64_t)j * E + e : Wr, ok);
            }
            uint8_t *x = stage_x(c);
            for (int q = tid; q < kTok * 8; q += kBThreads) {
                const int r = q >> 3, ch = q & 7;
                const int64_t t = t0 + r;
                const int j = j0 + 8 * ch;
                const bool ok = t < T && j < d;
                cp_async16_zfill(x + r * 128 + ((ch ^ ((r >> 1) & 7)) << 4),
                                 ok ? X + t * d + j : X, ok);
            }
        }
        cp_async_commit();
    };
    // raw rows 2p, 2p+1 -> transposed pairs xs[j][4g + i] = (x[2p][j], x[2p+1][j])
    // widened to fp32, where pair p is pair i of token group g
    auto transpose = [&](int c) {
        const uint8_t *x = stage_x(c);
        float2 *xs = xs_of(c);
        for (int q = tid; q < 8 * (PA + PB) * 8; q += kBThreads) {
            const int p = q % (8 * (PA + PB)), ch = q / (8 * (PA + PB));
            const int pos = (ch ^ (p & 7)) << 4;
            const uint4 a = *reinterpret_cast<const uint4 *>(x + (2 * p) * 128 + pos);
            const uint4 b = *reinterpret_cast<const uint4 *>(x + (2 * p + 1) * 128 + pos);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
            const int word = p < 8 * PA ? 4 * (p / PA) + p % PA
                                        : 4 * (8 + (p - 8 * PA) / PB) + (p - 8 * PA) % PB;
            float2 *dst = xs + (8 * ch) * kBWords + word;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                // word m holds steps 8ch + 2m (low half) and 8ch + 2m + 1 (high half)
                dst[(2 * m) * kBWords] = make_float2(__uint_as_float(aw[m] << 16),
                                                     __uint_as_float(bw[m] << 16));
                dst[(2 * m + 1) * kBWords] = make_float2(__uint_as_float(aw[m] & 0xffff0000u),
                                                         __uint_as_float(bw[m] & 0xffff0000u));
            }
        }
    };

    float2 acc[PA][8];
#pragma unroll
    for (int i = 0; i < PA; ++i)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[i][b] = make_float2(0.f, 0.f);

    const int g = 2 * warp + ty;  // the lane's token group
    const bool wa = warp < 4;     // PA token pairs (else PB)

    issue(0);
    issue(1);
    cp_async_wait<1>();
    __syncthreads();
    transpose(0);
    for (int c = 0; c < nchunk; ++c) {
        cp_async_wait<0>();  // stage c + 1 (issued one stage earlier) has landed
        __syncthreads();     // and every thread is past stage c - 1 and transpose(c)
        issue(c + 2);        // into the slot stage c - 1 used
        if (c + 1 < nchunk) transpose(c + 1);
        const float2 *xs = xs_of(c) + 4 * g;
        const float *w = stage_w(c) + 4 * tx;
        const int jn = min(kBK, d - c * kBK);
        if (jn == kBK) {
            if (wa) big_steps<PA, PA, true>(acc, xs, w, jn);
            else big_steps<PB, PA, true>(acc, xs, w, jn);
        } else {
            if (wa) big_steps<PA, PA, false>(acc, xs, w, jn);
            else big_steps<PB, PA, false>(acc, xs, w, jn);
        }
    }
    cp_async_wait<0>();

    // lane's token 2i (.x) and 2i+1 (.y) of its group; experts 4tx+b (b < 4),
    // 64+4tx+b-4
    const int np = wa ? PA : PB;
    const int64_t tg = t0 + (g < 8 ? 2 * PA * g : 16 * PA + 2 * PB * (g - 8));
#pragma unroll
    for (int i = 0; i < PA; ++i) {
        if (i >= np) break;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t t = tg + 2 * i + h;
            if (t >= T) continue;
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int e = e0 + 64 * gg + 4 * tx;
                if (e >= E) continue;
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 a = acc[i][4 * gg + u];
                    v[u] = h ? a.y : a.x;
                    if (bias != nullptr) v[u] = __fadd_rn(v[u], __ldg(bias + e + u));
                }
                *reinterpret_cast<float4 *>(L + t * E + e) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
    }
}

// ---------------------------------------------------------------- select --

constexpr int kSelThreads = 256;

// Scores as unsigned keys in the same order as the floats: larger score, larger
// key. -0.0 is first made +0.0 (adding +0.0 does that and changes nothing else),
// so the two zeros stay equal scores. Finite scores map above 0, which marks an
// expert that is taken or does not exist.
__device__ __forceinline__ uint32_t score_key(float v) {
    const uint32_t b = __float_as_uint(__fadd_rn(v, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp per token: lane l holds experts l, l+32, ... (NPL per lane). Each of
// the K rounds takes the warp maximum of the lanes' best untaken keys and then
// the lowest expert index among the lanes that hold it (two warp reductions),
// so ties go to the lower index. The weights need only the kept scores and
// the maximum, which is the first kept score: exp(L_k - L_max) over their sum
// (renormalised) or over the sum of exp(L_e - L_max) over every expert.
template <int NPL>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ logits, int T, int E, int K, int renorm,
              int32_t *__restrict__ idx_out, float *__restrict__ w_out,
              int32_t *__restrict__ counts) {
    pdl_wait();
    pdl_trigger();
    __shared__ int hist[kMaxE];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int e = tid; e < kMaxE; e += kSelThreads) hist[e] = 0;
    __syncthreads();
    const int64_t t = (int64_t)blockIdx.x * (kSelThreads / 32) + warp;
    if (t < T) {
        float v[NPL];
        uint32_t key[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            v[i] = (e < E) ? __ldg(logits + t * E + e) : 0.f;
            key[i] = (e < E) ? score_key(v[i]) : 0u;
        }
        int sel_idx[kMaxK];
        float sel_val[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (k < K) {
                // lane's best untaken key; within a lane the indices ascend, so
                // the strict comparison keeps the lower index on equal keys
                uint32_t bk = 0u;
                int bi = -1;
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (key[i] > bk) {
                        bk = key[i];
                        bi = lane + 32 * i;
                    }
                const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
                const uint32_t win = __reduce_min_sync(
                    0xffffffffu, (bk == kmax && bi >= 0) ? (uint32_t)bi : 0xffffffffu);
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if ((uint32_t)(lane + 32 * i) == win) key[i] = 0u;
                sel_idx[k] = (int)win;
                sel_val[k] = key_score(kmax);
            }
        }
        const float mtop = sel_val[0];
        float kept = 0.f, ex[kMaxK];
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (k < K) {
                ex[k] = expf(sel_val[k] - mtop);
                kept += ex[k];
            }
        }
        float denom = kept;
        if (!renorm) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (lane + 32 * i < E) s += expf(v[i] - mtop);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            denom = s;
        }
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (k < K && lane == k) {
                idx_out[t * K + k] = sel_idx[k];
                w_out[t * K + k] = ex[k] / denom;
                atomicAdd(&hist[sel_idx[k]], 1);
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kSelThreads)
        if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
}

// E <= 16: one thread per token. With T <= 2048 a single block zeroes and
// writes the counts itself (no memset, one launch); above that, blocks of 256
// threads add their histograms into counts zeroed before the logits kernel.
// Softmax statistics in the thread: the maximum, then a compensated (Kahan) sum
// of exp(L - max) for the full denominator; top-K by K passes (higher score
// wins, equal scores: lower index). VEC (E == EP, logits 16-byte aligned): a
// token's logits arrive as EP/4 128-bit loads.
constexpr int kSelSingleThreads = 1024;
constexpr int kSelSingleMaxT = 2048;
constexpr int kSelThreadBlock = 256;

template <int EP, bool SINGLE, bool VEC>
__global__ void __launch_bounds__(SINGLE ? kSelSingleThreads : kSelThreadBlock)
select_thread_kernel(const float *__restrict__ logits, int T, int E, int K, int renorm,
                     int32_t *__restrict__ idx_out, float *__restrict__ w_out,
                     int32_t *__restrict__ counts) {
    pdl_wait();
    pdl_trigger();
    __shared__ int hist[EP];
    for (int e = threadIdx.x; e < EP; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    // multi-block: a grid-stride loop over a grid of a few blocks per SM, so that
    // the blocks' histograms reach the E global counters in few atomics
    const int64_t t0 = SINGLE ? threadIdx.x : (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t tstep = SINGLE ? blockDim.x : (int64_t)gridDim.x * blockDim.x;
    auto load = [&](int64_t t, float (&v)[EP]) {
        if constexpr (VEC) {
            const float4 *src = reinterpret_cast<const float4 *>(logits + t * EP);
#pragma unroll
            for (int q = 0; q < EP / 4; ++q) {
                const float4 f = __ldg(src + q);
                v[4 * q] = f.x;
                v[4 * q + 1] = f.y;
                v[4 * q + 2] = f.z;
                v[4 * q + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < EP; ++e) v[e] = (e < E) ? __ldg(logits + t * E + e) : -INFINITY;
        }
    };
    for (int64_t t = t0; t < T; t += tstep) {
        float v[EP];
        load(t, v);
        select_token<EP>(v, E, K, renorm, t, idx_out, w_out, hist);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (SINGLE) counts[e] = hist[e];
        else if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
    }
}

// The single-block select writes the counts itself; the multi-block one adds
// into counts that must be zero first.
bool select_needs_zero_counts(int T, int E) { return !(E <= 16 && T <= kSelSingleMaxT); }

// counts_zeroed: the caller has already set counts to zero on this stream (so
// that no memset sits between the logits and select kernels).
cudaError_t launch_select(const float *logits, int T, int E, int K, int renorm, int32_t *idx,
                          float *w, int32_t *counts, bool counts_zeroed, cudaStream_t s) {
    const bool vec = (E == 8 || E == 16) && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
    if (!select_needs_zero_counts(T, E)) {
        auto kern = E <= 8 ? (vec ? select_thread_kernel<8, true, true>
                                  : select_thread_kernel<8, true, false>)
                           : (vec ? select_thread_kernel<16, true, true>
                                  : select_thread_kernel<16, true, false>);
        return launch_k(kern, dim3(1), dim3(kSelSingleThreads), 0, s, logits, T, E, K, renorm, idx,
                        w, counts);
    }
    if (!counts_zeroed) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        if (e != cudaSuccess) return e;
    }
    if (E <= 16) {
        auto kern = E <= 8 ? (vec ? select_thread_kernel<8, false, true>
                                  : select_thread_kernel<8, false, false>)
                           : (vec ? select_thread_kernel<16, false, true>
                                  : select_thread_kernel<16, false, false>);
        // as many blocks as are resident at once
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kSelThreadBlock, 0) !=
                cudaSuccess || per_sm < 1)
            per_sm = 1;
        const int64_t need = (T + kSelThreadBlock - 1) / kSelThreadBlock;
        const unsigned blocks =
            (unsigned)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)per_sm * sm_count()));
        return launch_k(kern, dim3(blocks), dim3(kSelThreadBlock), 0, s, logits, T, E, K, renorm,
                        idx, w, counts);
    }
    const unsigned blocks = (unsigned)((T + kSelThreads / 32 - 1) / (kSelThreads / 32));
    auto kern = E <= 32    ? select_kernel<1>
                : E <= 64  ? select_kernel<2>
                : E <= 128 ? select_kernel<4>
                           : select_kernel<8>;
    return launch_k(kern, dim3(blocks), dim3(kSelThreads), 0, s, logits, T, E, K, renorm, idx, w,
                    counts);
}

// Token groups per CTA of the fused E <= 32 route kernel: the CTA holds all
// blocks of its groups, up to kRouteWarps items; with few blocks it takes more
// groups, unless that leaves SMs idle.
int route_token_groups(int T, int d, int tpw) {
    const int nb = (d + kLogitBlock - 1) / kLogitBlock;
    int tg = nb >= kRouteWarps ? 1 : kRouteWarps / nb;
    const int64_t groups = (T + tpw - 1) / tpw;
    while (tg > 1 && (groups + tg - 1) / tg < sm_count()) --tg;
    return tg;
}

template <int EP>
cudaError_t launch_route_chain(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T,
                              int d, int E, int K, int renorm, float *L, int32_t *idx, float *w,
                              int32_t *counts, cudaStream_t s) {
    using C = RouteCfg<EP>;
    const int nb = (d + kLogitBlock - 1) / kLogitBlock;
    const int tg = route_token_groups(T, d, C::TPW);
    const int warps = std::min(kRouteWarps, tg * nb);
    const size_t smem = (size_t)warps * C::WARP_SMEM + (size_t)tg * nb * C::PART;
    {
        // the most any call of this kernel asks for, so the limit is set once
        const size_t most = (size_t)kRouteWarps * C::WARP_SMEM + (size_t)kRouteMaxBlocks * C::PART;
        const cudaError_t e =
            ensure_dynamic_smem(reinterpret_cast<const void *>(route_chain_kernel<EP>), (int)most);
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = (unsigned)(((int64_t)T + (int64_t)tg * C::TPW - 1) / ((int64_t)tg * C::TPW));
    return launch_k(route_chain_kernel<EP>, dim3(grid), dim3(32 * warps), smem, s, X, Wr, bias, T,
                    d, E, K, renorm, tg, L, idx, w, counts);
}

template <int PA, int PB>
cudaError_t launch_big(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T, int d,
                       int E, float *L, cudaStream_t s) {
    {
        const cudaError_t e =
            ensure_dynamic_smem(reinterpret_cast<const void *>(logits_big_kernel<PA, PB>), kBSmem);
        if (e != cudaSuccess) return e;
    }
    constexpr int kTok = 16 * (PA + PB);
    const dim3 grid((unsigned)((T + kTok - 1) / kTok), (unsigned)((E + kBE - 1) / kBE));
    return launch_k(logits_big_kernel<PA, PB>, grid, dim3(kBThreads), (size_t)kBSmem, s, X, Wr,
                    bias, T, d, E, L);
}

// Token pairs per scheduler (P = PA + PB) of the one-block-per-SM kernel (0: use
// the 4 x 8 tile). Every block runs the same d steps of 8P packed FMAs per
// scheduler lane, so the time is about (waves of blocks) x P; the smallest such cost wins, the larger P on a
// tie. MOE_ROUTER_PAIRS=4..8 forces P and MOE_ROUTER_PAIRS=0 the 4 x 8 tile
// (tests and measurements use it to run each variant).
int big_tile_pairs(int T, int E) {
    if (const char *env = getenv("MOE_ROUTER_PAIRS"); env != nullptr && *env != 0) {
        const int p = atoi(env);
        if (p == 0 || (p >= 4 && p <= 8)) return p;
    }
    if (E < kBE || (int64_t)T * E < (int64_t)1 << 20) return 0;
    const int64_t sms = sm_count(), eb = (E + kBE - 1) / kBE;
    int best = 0;
    int64_t best_cost = 0;
    for (int P = 8; P >= 4; --P) {
        const int64_t blocks = (T + 16 * P - 1) / (16 * P) * eb;
        const int64_t cost = (blocks + sms - 1) / sms * P;
        if (best == 0 || cost < best_cost) best = P, best_cost = cost;
    }
    return best;
}

}  // namespace

cudaError_t launch_router_logits(const __nv_bfloat16 *X, const float *Wr, const float *bias,
                                 int T, int d, int E, float *L, cudaStream_t s) {
    const bool wr16 = (reinterpret_cast<uintptr_t>(Wr) & 15u) == 0;
    if (E > 32 && E % 4 == 0 && wr16) {
        switch (big_tile_pairs(T, E)) {
            case 4: return launch_big<2, 2>(X, Wr, bias, T, d, E, L, s);
            case 5: return launch_big<3, 2>(X, Wr, bias, T, d, E, L, s);
            case 6: return launch_big<3, 3>(X, Wr, bias, T, d, E, L, s);
            case 7: return launch_big<4, 3>(X, Wr, bias, T, d, E, L, s);
            case 8: return launch_big<4, 4>(X, Wr, bias, T, d, E, L, s);
            default: break;
        }
    }
    if (E <= 32) {
        const int ep = E <= 8 ? 8 : (E <= 16 ? 16 : 32);
        auto kern = E <= 8 ? logits_small_kernel<8>
                           : (E <= 16 ? logits_small_kernel<16> : logits_small_kernel<32>);
        const unsigned grid = (unsigned)(((int64_t)T * ep + kSmallThreads - 1) / kSmallThreads);
        return launch_k(kern, dim3(grid), dim3(kSmallThreads), 0, s, X, Wr, bias, T, d, E, L);
    }
    const dim3 grid((unsigned)((T + kWT - 1) / kWT), (unsigned)((E + kWE - 1) / kWE));
    auto kern = (E % 4 == 0 && wr16) ? logits_tiled_kernel<true> : logits_tiled_kernel<false>;
    return launch_k(kern, grid, dim3(kWThreads), 0, s, X, Wr, bias, T, d, E, L);
}

bool route_is_one_kernel(int d, int E, bool wr16) {
    return E <= 32 && E % 4 == 0 && wr16 && d <= kRouteMaxBlocks * kLogitBlock;
}

cudaError_t launch_route(const __nv_bfloat16 *X, const float *Wr, const float *bias, int T,
                         int d, int E, int K, int renorm, float *logits, int32_t *idx, float *w,
                         int32_t *counts, cudaStream_t s) {
    const bool wr16 = (reinterpret_cast<uintptr_t>(Wr) & 15u) == 0;
    if (route_is_one_kernel(d, E, wr16)) {
        // logits and selection in one kernel; its CTAs add into zeroed counts
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        if (e != cudaSuccess) return e;
        if (E <= 8)
            return launch_route_chain<8>(X, Wr, bias, T, d, E, K, renorm, logits, idx, w, counts, s);
        if (E <= 16)
            return launch_route_chain<16>(X, Wr, bias, T, d, E, K, renorm, logits, idx, w, counts, s);
        return launch_route_chain<32>(X, Wr, bias, T, d, E, K, renorm, logits, idx, w, counts, s);
    }
    const bool zero = select_needs_zero_counts(T, E);
    if (zero) {
        cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_router_logits(X, Wr, bias, T, d, E, logits, s);
    if (e != cudaSuccess) return e;
    return launch_select(logits, T, E, K, renorm, idx, w, counts, zero, s);
}

cudaError_t launch_route_logits(const float *logits, int T, int E, int K, int renorm,
                                int32_t *idx, float *w, int32_t *counts, cudaStream_t s) {
    return launch_select(logits, T, E, K, renorm, idx, w, counts, false, s);
}

}  // namespace moe
