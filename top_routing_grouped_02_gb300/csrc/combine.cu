// Row movement: the Gather of activation rows into expert-grouped order (used
// ahead of the CTA-pair gate/up GEMM, which loads A by TMA; the single-CTA GEMM
// gathers rows itself) and the Scatter/combine of weighted expert outputs back
// into token order.
//
// Pages: "混合专家模型(MoE)架构优化与SonicMoE实践" §1 (Gather rows by routing
// result; Scatter results back to the tokens' original positions);
// "稀疏矩阵乘法（SpMM）在MoE中的应用：利用Triton内核加速稀疏专家的计算" §6 (the
// selected experts' outputs are combined with their routing weights; the weights
// are applied in the down-projection epilogue, so the combine is a plain sum).
//
// Both kernels are HBM-bound copies/reductions: one warp per row, 16-byte
// vector loads and stores, fixed summation order (ascending k, fp32, one final
// bf16 rounding) so the result is deterministic and needs no atomics.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const __nv_bfloat16 *__restrict__ X, const int32_t *__restrict__ perm_token,
                   int T, int R, const int32_t *__restrict__ rows_used, int d,
                   __nv_bfloat16 *__restrict__ Xg, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int64_t p = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (p >= R || (rows_used != nullptr && p >= __ldg(rows_used))) return;
    const int lane = threadIdx.x & 31;
    const int64_t t = perm_token[p];
    uint4 *dst = reinterpret_cast<uint4 *>(Xg + p * d);
    const int nv = d / 8;
    if (t < 0 || t >= T) {  // a token index out of range: zeros, flagged
        for (int c = lane; c < nv; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
        if (lane == 0 && err != nullptr) atomicOr(err, MOE_DEVERR_BAD_EXPERT);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(X + t * d);
    for (int c = lane; c < nv; c += 32) dst[c] = __ldg(src + c);
}

template <int KU>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const __nv_bfloat16 *__restrict__ Z, const int32_t *__restrict__ row_of_slot,
               int T, int K, int d, __nv_bfloat16 *__restrict__ Y) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    int myrow = lane < K ? row_of_slot[t * K + lane] : -1;
    if (myrow >= T * K) myrow = -1;  // out of range: treated as a missing slot
    int rows[KU];
#pragma unroll
    for (int k = 0; k < KU; ++k) rows[k] = __shfl_sync(0xffffffffu, myrow, k);
    const int nv = d / 8;
    uint4 *dst = reinterpret_cast<uint4 *>(Y + t * d);
    for (int c = lane; c < nv; c += 32) {
        uint4 v[KU];
#pragma unroll
        for (int k = 0; k < KU; ++k)
            if (k < K && rows[k] >= 0)
                v[k] = __ldg(reinterpret_cast<const uint4 *>(Z + (int64_t)rows[k] * d) + c);
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#pragma unroll
        for (int k = 0; k < KU; ++k) {
            if (k < K && rows[k] >= 0) {
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v[k]);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float2 f = __bfloat1622float2(h2[u]);
                    acc[2 * u] = __fadd_rn(acc[2 * u], f.x);
                    acc[2 * u + 1] = __fadd_rn(acc[2 * u + 1], f.y);
                }
            }
        }
        uint4 out;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
        for (int u = 0; u < 4; ++u) o2[u] = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
        dst[c] = out;
    }
}

}  // namespace

cudaError_t launch_gather_rows(const __nv_bfloat16 *X, const int32_t *perm_token, int T, int R,
                               const int32_t *rows_used, int d, __nv_bfloat16 *Xg, uint32_t *err,
                               cudaStream_t s) {
    return launch_k(gather_rows_kernel, dim3((R + kWarps - 1) / kWarps), dim3(kThreads), 0, s, X,
                    perm_token, T, R, rows_used, d, Xg, err);
}

cudaError_t launch_combine(const __nv_bfloat16 *Z, const int32_t *row_of_slot, int T, int K,
                           int d, __nv_bfloat16 *Y, cudaStream_t s) {
    const unsigned blocks = (unsigned)((T + kWarps - 1) / kWarps);
    if (K <= 2) return launch_k(combine_kernel<2>, dim3(blocks), dim3(kThreads), 0, s, Z, row_of_slot, T, K, d, Y);
    if (K <= 4) return launch_k(combine_kernel<4>, dim3(blocks), dim3(kThreads), 0, s, Z, row_of_slot, T, K, d, Y);
    return launch_k(combine_kernel<8>, dim3(blocks), dim3(kThreads), 0, s, Z, row_of_slot, T, K, d, Y);
}

}  // namespace moe
