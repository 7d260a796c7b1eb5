// Token Rounding: a routing mode whose per-expert row counts are multiples of
// the GEMM row tile, so no expert tile carries padding rows.
//
// Page "混合专家模型(MoE)架构优化与SonicMoE实践" §3: count each expert's top-K
// choices (§3.1, expert frequency), round every count to a multiple of the tile
// size (§3.2: to the nearest multiple, halves up), and settle by a second sort
// which tokens an expert drops (rounded down: its chosen tokens with the lowest
// scores) or gains (rounded up: the unchosen tokens with the highest scores);
// the kept scores are then renormalised by a softmax (§3.2).
//
// Kernels:
//   round_select_kernel   one CTA per expert. Every CTA recomputes all rounded
//                         counts and their prefix sums from counts[] (E <= 256,
//                         one warp), so the grouped offsets need no second
//                         launch. The second sort is a selection, not a full
//                         sort: an MSB-first radix select on order-preserving
//                         32-bit keys of the expert's logit column finds the
//                         threshold score, ties at the threshold go to the
//                         lowest token indices, and one ordered pass over the
//                         tokens writes perm_token and the expert's column of
//                         row_map. The column (keys + chosen flags) is staged
//                         in shared memory when it fits, else in workspace.
//   round_weights_kernel  one warp per token: softmax of the logit row, the
//                         weight of every kept (token, expert) pair, fp64 sums.
//   combine_rows_kernel   one warp per token: sum of the token's kept rows in
//                         ascending expert order (fp32, one bf16 rounding).
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRThreads = 1024;
constexpr int kRWarps = kRThreads / 32;
static_assert(kRWarps == 32, "the block scan assumes 32 warps");

// Largest token count whose logit column is staged in shared memory
// (4-byte key + 1-byte flag per token: 160 KB).
constexpr int kRoundSmemT = 32768;

// Monotone map of an fp32 value to uint32 (larger value, larger key); -0 ranks
// as +0 so that equal values have equal keys.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive prefix count of `flag` over the block in thread order. Every thread
// of the block must call it; *total receives the block's count.
__device__ __forceinline__ int block_excl_count(bool flag, int *ws, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) ws[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        const int v = ws[lane];
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        ws[lane] = incl - v;
        if (lane == 31) ws[32] = incl;
    }
    __syncthreads();
    const int r = ws[warp] + in_warp;
    *total = ws[32];
    __syncthreads();  // ws is reused by the next call
    return r;
}

// Histogram update with one shared-memory atomic per distinct digit of a warp.
// Every lane of the warp must call it.
__device__ __forceinline__ void hist_add(int *hist, bool active, uint32_t digit) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (active) {
        const unsigned peers = __match_any_sync(act, digit);
        if ((int)(__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[digit], __popc(peers));
    }
}

struct RoundArgs {
    const float *L;         // [T,E] logits
    const int32_t *idx;     // [T,K] top-K choice
    const int32_t *counts;  // [E]   top-K counts
    int T, E, K, M;
    int64_t cap;            // length of perm_token (rows beyond it are never written)
    int max_tiles;          // length of the tile list
    int32_t *counts_out;    // [E]
    int32_t *offsets;       // [E+1]
    int32_t *perm_token;    // [capacity]
    int32_t *row_map;       // [T,E]
    int32_t *tiles;         // [tiles][4]
    int32_t *num_tiles;     // [1]
    uint32_t *keys_g;       // [E*T] column scratch when T > kRoundSmemT
    uint8_t *flags_g;       // [E*T]
    uint32_t *err;
};

enum : int { kKeep = 0, kDown = 1, kUp = 2 };

__global__ void __launch_bounds__(kRThreads, 1) round_select_kernel(RoundArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ int s_off[kMaxE + 1];  // exclusive prefix of the rounded counts
    __shared__ int s_tb[kMaxE + 1];   // exclusive prefix of the 128-row tile counts
    __shared__ int s_hist[256];
    __shared__ int s_ws[33];
    __shared__ int s_members;
    __shared__ uint32_t s_sel[3];     // threshold prefix, still to take, equal-key count
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, E = a.E, K = a.K, M = a.M;

    // rounded counts of all experts and their prefix sums: 8 experts per lane
    if (warp == 0) {
        int c8[8], t8[8], cs = 0, ts = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ex = lane * 8 + i;
            int c = 0;
            if (ex < E) {
                const int f = max(0, min(a.counts[ex], T));
                c = M * ((f + M / 2) / M);
                if (c > T) c = M * (f / M);
            }
            c8[i] = c;
            t8[i] = (c + kTileM - 1) / kTileM;
            cs += c;
            ts += t8[i];
        }
        int ci = cs, ti = ts;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n1 = __shfl_up_sync(0xffffffffu, ci, o);
            const int n2 = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) {
                ci += n1;
                ti += n2;
            }
        }
        int cb = ci - cs, tb = ti - ts;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ex = lane * 8 + i;
            if (ex <= E) {
                s_off[ex] = cb;
                s_tb[ex] = tb;
            }
            cb += c8[i];
            tb += t8[i];
        }
        if (lane == 31 && E == 256) {
            s_off[E] = ci;
            s_tb[E] = ti;
        }
    }
    if (tid == 0) s_members = 0;
    if (tid < 256) s_hist[tid] = 0;
    __syncthreads();

    const int base = s_off[e], ce = s_off[e + 1] - base;
    const int f = max(0, min(a.counts[e], T));
    if (e == 0) {
        for (int i = tid; i <= E; i += kRThreads) a.offsets[i] = s_off[i];
        if (tid == 0) a.num_tiles[0] = s_tb[E];
    }
    if (tid == 0) a.counts_out[e] = ce;
    {
        const int tb = s_tb[e], nt = s_tb[e + 1] - tb;
        for (int i = tid; i < nt && tb + i < a.max_tiles; i += kRThreads)
            reinterpret_cast<int4 *>(a.tiles)[tb + i] =
                make_int4(e, base + i * kTileM, min(kTileM, ce - i * kTileM), 0);
    }
    const int mode = ce == f ? kKeep : (ce < f ? kDown : kUp);
    const int N = mode == kDown ? ce : (mode == kUp ? ce - f : 0);
    const bool need_sel = N > 0;

    const bool in_smem = T <= kRoundSmemT;
    uint32_t *keys = in_smem ? reinterpret_cast<uint32_t *>(dyn) : a.keys_g + (size_t)e * T;
    uint8_t *flg = in_smem ? dyn + (size_t)4 * T : a.flags_g + (size_t)e * T;

    // pass 0: membership from the top-K choice, keys of the logit column, and the
    // histogram of the top key byte over the candidates
    int members = 0;
    for (int t0 = 0; t0 < T; t0 += kRThreads) {
        const int t = t0 + tid;
        const bool in = t < T;
        bool m = false;
        uint32_t key = 0;
        if (in) {
            const int32_t *ir = a.idx + (size_t)t * K;
            for (int k = 0; k < K; ++k) m |= (__ldg(ir + k) == e);
            key = order_key(__ldg(a.L + (size_t)t * E + e));
            keys[t] = key;
            flg[t] = m ? 1 : 0;
        }
        members += m ? 1 : 0;
        const bool cand = in && need_sel && (mode == kDown ? m : !m);
        hist_add(s_hist, cand, key >> 24);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) members += __shfl_xor_sync(0xffffffffu, members, o);
    if (lane == 0) atomicAdd(&s_members, members);
    __syncthreads();
    if (tid == 0 && s_members != f) atomicOr(a.err, MOE_DEVERR_COUNT_MISMATCH);

    // radix select of the N-th largest candidate key, one byte per pass
    uint32_t prefix = 0;
    int remaining = N, eq_count = 0;
    if (need_sel) {
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (pass > 0) {
                if (tid < 256) s_hist[tid] = 0;
                __syncthreads();
                const uint32_t hm = 0xFFFFFFFFu << (shift + 8);
                for (int t0 = 0; t0 < T; t0 += kRThreads) {
                    const int t = t0 + tid;
                    bool cand = false;
                    uint32_t key = 0;
                    if (t < T) {
                        key = keys[t];
                        const bool m = flg[t] != 0;
                        cand = (mode == kDown ? m : !m) && ((key & hm) == (prefix & hm));
                    }
                    hist_add(s_hist, cand, (key >> shift) & 255u);
                }
                __syncthreads();
            }
            if (warp == 0) {
                // lane l holds digits 255-8l .. 248-8l (descending)
                int h[8], sum = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    h[i] = s_hist[255 - 8 * lane - i];
                    sum += h[i];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
                if (hit == 0) {
                    // fewer candidates than the count asks for (counts[] does not
                    // match idx): take none; the row count check flags it
                    if (lane == 0) {
                        s_sel[0] = 0xFFFFFFFFu;
                        s_sel[1] = 0;
                        s_sel[2] = 1;
                    }
                } else if (lane == __ffs(hit) - 1) {
                    int acc = incl - sum, dg = 0, cnt = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (cnt == 0 && acc + h[i] >= remaining) {
                            dg = 255 - 8 * lane - i;
                            cnt = h[i];
                        } else if (cnt == 0) {
                            acc += h[i];
                        }
                    }
                    s_sel[0] = prefix | ((uint32_t)dg << shift);
                    s_sel[1] = (uint32_t)(remaining - acc);
                    s_sel[2] = (uint32_t)cnt;
                }
            }
            __syncthreads();
            prefix = s_sel[0];
            remaining = (int)s_sel[1];
            eq_count = (int)s_sel[2];
            if (remaining == 0) break;  // (only after a mismatch) nothing more to take
        }
    }
    const uint32_t v = prefix;
    const bool all_eq = remaining >= eq_count;

    // ordered pass: which tokens the expert keeps, their rows, its row_map column
    int carry_eq = 0, carry_keep = 0;
    for (int t0 = 0; t0 < T; t0 += kRThreads) {
        const int t = t0 + tid;
        const bool in = t < T;
        uint32_t key = 0;
        bool m = false;
        if (in) {
            key = keys[t];
            m = flg[t] != 0;
        }
        bool chosen = false;
        if (need_sel) {
            const bool cand = in && (mode == kDown ? m : !m);
            const bool gt = cand && key > v, eq = cand && key == v && remaining > 0;
            if (all_eq) {
                chosen = gt || eq;
            } else {
                int tot;
                const int r = block_excl_count(eq, s_ws, &tot);
                chosen = gt || (eq && carry_eq + r < remaining);
                carry_eq += tot;
            }
        }
        const bool keep = in && (mode == kKeep ? m : (mode == kDown ? chosen : (m || chosen)));
        int tot;
        const int r = block_excl_count(keep, s_ws, &tot);
        if (in) {
            int row = -1;
            if (keep && carry_keep + r < ce && (int64_t)base + carry_keep + r < a.cap) {
                row = base + carry_keep + r;
                a.perm_token[row] = t;
            }
            a.row_map[(size_t)t * E + e] = row;
        }
        carry_keep += tot;
    }
    if (tid == 0 && (carry_keep != ce || (int64_t)base + ce > a.cap))
        atomicOr(a.err, MOE_DEVERR_COUNT_MISMATCH);
}

constexpr int kWThreads = 256;
constexpr int kWWarps = kWThreads / 32;
constexpr int kPerLane = kMaxE / 32;

__global__ void __launch_bounds__(kWThreads)
round_weights_kernel(const float *__restrict__ L, const int32_t *__restrict__ row_map, int T,
                     int E, int renorm, float *__restrict__ row_w) {
    const int64_t t = (int64_t)blockIdx.x * kWWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    float l[kPerLane];
    int r[kPerLane];
    float m_all = -INFINITY, m_kept = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        l[i] = -INFINITY;
        r[i] = -1;
        if (e < E) {
            l[i] = __ldg(L + t * E + e);
            r[i] = __ldg(row_map + t * E + e);
            m_all = fmaxf(m_all, l[i]);
            if (r[i] >= 0) m_kept = fmaxf(m_kept, l[i]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m_all = fmaxf(m_all, __shfl_xor_sync(0xffffffffu, m_all, o));
        m_kept = fmaxf(m_kept, __shfl_xor_sync(0xffffffffu, m_kept, o));
    }
    if (m_kept == -INFINITY) return;  // no expert kept this token
    // renormalised: exp(l - max over kept) / sum over kept; else the softmax over all
    const float mref = renorm ? m_kept : m_all;
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int e = lane + 32 * i;
        if (e < E && (!renorm || r[i] >= 0)) s += (double)expf(l[i] - mref);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
        if (r[i] >= 0) row_w[r[i]] = (float)((double)expf(l[i] - mref) / s);
}

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;

__device__ __forceinline__ void add_bf16x8(float *acc, const uint4 &v) {
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h2[u]);
        acc[2 * u] = __fadd_rn(acc[2 * u], f.x);
        acc[2 * u + 1] = __fadd_rn(acc[2 * u + 1], f.y);
    }
}

__global__ void __launch_bounds__(kCThreads)
combine_rows_kernel(const __nv_bfloat16 *__restrict__ Z, const int32_t *__restrict__ row_map,
                    int T, int E, int d, int64_t rows_cap, __nv_bfloat16 *__restrict__ Y) {
    __shared__ int s_rows[kCWarps][kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCWarps + warp;
    if (t >= T) return;
    int *rows = s_rows[warp];
    int n = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        int r = e < E ? __ldg(row_map + t * E + e) : -1;
        if (r >= rows_cap) r = -1;  // out of range: treated as not kept
        const unsigned bal = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) rows[n + __popc(bal & ((1u << lane) - 1u))] = r;
        n += __popc(bal);
    }
    __syncwarp();
    const int nv = d / 8;
    uint4 *dst = reinterpret_cast<uint4 *>(Y + t * d);
    for (int c = lane; c < nv; c += 32) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
        int i = 0;
        for (; i + 4 <= n; i += 4) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = __ldg(reinterpret_cast<const uint4 *>(Z + (int64_t)rows[i + j] * d) + c);
#pragma unroll
            for (int j = 0; j < 4; ++j) add_bf16x8(acc, v[j]);
        }
        for (; i < n; ++i)
            add_bf16x8(acc, __ldg(reinterpret_cast<const uint4 *>(Z + (int64_t)rows[i] * d) + c));
        uint4 out;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
        for (int u = 0; u < 4; ++u) o2[u] = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
        dst[c] = out;
    }
}

}  // namespace

size_t round_scratch_bytes(int T, int E) {
    if (T <= kRoundSmemT) return 0;
    return (size_t)5 * E * T;
}

cudaError_t launch_round(const float *L, const int32_t *idx, const int32_t *counts, int T, int E,
                         int K, int M, int renorm, int32_t *counts_out, int32_t *offsets,
                         int32_t *perm_token, int32_t *row_map, float *row_w, int32_t *tiles,
                         int32_t *num_tiles, void *scratch, uint32_t *err, cudaStream_t s) {
    RoundArgs a{};
    a.L = L;
    a.idx = idx;
    a.counts = counts;
    a.T = T;
    a.E = E;
    a.K = K;
    a.M = M;
    a.cap = round_capacity(T, E, K, M);
    a.max_tiles = (int)(a.cap / kTileM) + E;
    a.counts_out = counts_out;
    a.offsets = offsets;
    a.perm_token = perm_token;
    a.row_map = row_map;
    a.tiles = tiles;
    a.num_tiles = num_tiles;
    a.keys_g = static_cast<uint32_t *>(scratch);
    a.flags_g = scratch ? static_cast<uint8_t *>(scratch) + (size_t)4 * E * T : nullptr;
    a.err = err;
    const size_t smem = T <= kRoundSmemT ? (size_t)5 * T : 0;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(round_select_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             5 * kRoundSmemT);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    round_select_kernel<<<E, kRThreads, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    round_weights_kernel<<<(unsigned)((T + kWWarps - 1) / kWWarps), kWThreads, 0, s>>>(
        L, row_map, T, E, renorm, row_w);
    return cudaGetLastError();
}

cudaError_t launch_combine_rows(const __nv_bfloat16 *Z, const int32_t *row_map, int T, int E,
                                int d, int64_t rows_cap, __nv_bfloat16 *Y, cudaStream_t s) {
    combine_rows_kernel<<<(unsigned)((T + kCWarps - 1) / kCWarps), kCThreads, 0, s>>>(
        Z, row_map, T, E, d, rows_cap, Y);
    return cudaGetLastError();
}

}  // namespace moe
