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
//   round_prep_kernel     32 tokens per block: transposes the logit tile through
//                         shared memory into per-expert candidate keys keyT[E][Tp]
//                         (coalesced rows; 0 marks a token that is not a
//                         candidate of that expert's selection) and fills the
//                         tile's row_map with -1.
//   round_select_kernel   one CTA per expert. Every CTA recomputes all rounded
//                         counts and their prefix sums from counts[] (E <= 256,
//                         one warp), so the grouped offsets need no extra
//                         launch. The second sort is a selection, not a full
//                         sort: an MSB-first radix select on the order-preserving
//                         32-bit keys finds the threshold score, ties at the
//                         threshold go to the lowest token indices. Each thread
//                         owns a contiguous run of tokens, so one block-wide
//                         prefix sum orders the kept tokens; they go to
//                         perm_token and to the expert's entries of row_map.
//   round_weights_kernel  one warp per token: softmax of the logit row and the
//                         weight of every kept (token, expert) pair, with
//                         compensated fp32 sums.
//   combine_rows_kernel   one warp per token: sum of the token's kept rows in
//                         ascending expert order (fp32, one bf16 rounding).
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

enum : int { kKeep = 0, kDown = 1, kUp = 2 };

// Monotone map of an fp32 value to uint32 (larger value, larger key); -0 ranks
// as +0 so that equal values have equal keys. Finite values never map to 0.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Rounded count of an expert chosen f times: nearest multiple of M (halves up),
// the rounded-down multiple when that exceeds T.
__device__ __forceinline__ int rounded_count(int f, int M, int T) {
    const int c = M * ((f + M / 2) / M);
    return c > T ? M * (f / M) : c;
}

// Token-axis stride of the key rows (a multiple of 32 tokens: 16-byte rows).
__host__ __device__ __forceinline__ int key_stride(int T) { return (T + 31) / 32 * 32; }

// ---------------------------------------------------------------- prep ----
constexpr int kPT = 32;        // tokens per prep block
constexpr int kPThreads = 256;

__global__ void __launch_bounds__(kPThreads)
round_prep_kernel(const float *__restrict__ L, const int32_t *__restrict__ idx,
                  const int32_t *__restrict__ counts, int T, int E, int K, int M, bool vec,
                  uint32_t *__restrict__ keyT, int32_t *__restrict__ row_map, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_L[kPT][kMaxE + 1];
    __shared__ uint32_t s_mem[kPT][kMaxE / 32];
    __shared__ int s_mode[kMaxE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * kPT;
    const int Tp = key_stride(T);
    for (int e = tid; e < E; e += kPThreads) {
        const int f = max(0, min(__ldg(counts + e), T));
        const int c = rounded_count(f, M, T);
        s_mode[e] = c == f ? kKeep : (c < f ? kDown : kUp);
    }
    for (int i = tid; i < kPT * (kMaxE / 32); i += kPThreads) (&s_mem[0][0])[i] = 0u;
    // the tile's logits: rows t0..t0+31 are contiguous in L
    const int rows = min(kPT, T - t0);
    if (vec) {
        const float4 *src = reinterpret_cast<const float4 *>(L + (size_t)t0 * E);
        for (int q = tid; q < rows * E / 4; q += kPThreads) {
            const float4 v = __ldg(src + q);
            const int j = 4 * q / E, e = 4 * q - j * E;
            s_L[j][e] = v.x;
            s_L[j][e + 1] = v.y;
            s_L[j][e + 2] = v.z;
            s_L[j][e + 3] = v.w;
        }
    } else {
        for (int q = tid; q < rows * E; q += kPThreads) {
            const int j = q / E, e = q - j * E;
            s_L[j][e] = __ldg(L + (size_t)t0 * E + q);
        }
    }
    __syncthreads();
    for (int q = tid; q < kPT * K; q += kPThreads) {
        const int j = q / K;
        if (t0 + j >= T) continue;
        const int ex = __ldg(idx + (size_t)t0 * K + q);
        if (ex >= 0 && ex < E) atomicOr(&s_mem[j][ex >> 5], 1u << (ex & 31));
        else atomicOr(err, MOE_DEVERR_BAD_EXPERT);
    }
    __syncthreads();
    // candidate keys, one expert row per warp step: lane = token
    {
        const int t = t0 + lane;
        for (int e = warp; e < E; e += kPThreads / 32) {
            uint32_t key = 0;
            if (t < T) {
                const bool m = (s_mem[lane][e >> 5] >> (e & 31)) & 1u;
                const int mode = s_mode[e];
                // kept without a choice (kKeep): members, marked 1; rounded down:
                // members compete; rounded up: non-members compete
                if (mode == kKeep) key = m ? 1u : 0u;
                else if (mode == kDown ? m : !m) key = order_key(s_L[lane][e]);
            }
            if (t < Tp) keyT[(size_t)e * Tp + t] = key;
        }
    }
    if (vec) {
        int4 *dst = reinterpret_cast<int4 *>(row_map + (size_t)t0 * E);
        for (int q = tid; q < rows * E / 4; q += kPThreads) dst[q] = make_int4(-1, -1, -1, -1);
    } else {
        for (int q = tid; q < rows * E; q += kPThreads) row_map[(size_t)t0 * E + q] = -1;
    }
}

// -------------------------------------------------------------- select ----
constexpr int kRThreads = 1024;
static_assert(kRThreads / 32 == 32, "the block scan assumes 32 warps");

// Exclusive prefix sum of v over the block in thread order; every thread of the
// block must call it; *total receives the block's sum.
__device__ __forceinline__ int block_excl_sum(int v, int *ws, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int x = ws[lane];
        int xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, xi, o);
            if (lane >= o) xi += n;
        }
        ws[lane] = xi - x;
        if (lane == 31) ws[32] = xi;
    }
    __syncthreads();
    const int r = ws[warp] + incl - v;
    *total = ws[32];
    __syncthreads();  // ws is reused by the next call
    return r;
}

// Radix histograms of 2^W bins (5 <= W <= 12) are split into 32 groups of
// P = 2^(W-5) consecutive bins, each followed by 4 padding words: a group starts
// 16-byte aligned and the 32 groups fall on different banks, so warp 0 reads a
// group per lane with 16-byte loads and no bank conflicts.
__device__ __forceinline__ int hpad(uint32_t bin, int W) { return (int)(bin + 4u * (bin >> (W - 5))); }
constexpr int kHistWords = 4096 + 4 * 32;

// The bin, scanning bins 2^W-1 down to 0, at which the running count reaches
// `remaining`: sel = {bin, count in higher bins, count in the bin}, or
// sel[0] = 0xFFFFFFFF when the histogram holds fewer than `remaining`. Lane l
// of warp 0 takes group 31-l (the bins 2^W-1-l*P down to 2^W-(l+1)*P); every
// thread of the block must call it.
__device__ __forceinline__ void digit_select(const int *hist, int W, int remaining, uint32_t *sel) {
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int P = 1 << (W - 5), grp = 31 - lane;
        const int4 *g4 = reinterpret_cast<const int4 *>(hist + grp * (P + 4));
        int sum = 0;
        for (int j = 0; j < P / 4; ++j) {
            const int4 h = g4[j];
            sum += h.x + h.y + h.z + h.w;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
        if (hit == 0) {
            if (lane == 0) sel[0] = 0xFFFFFFFFu;
        } else if (lane == __ffs(hit) - 1) {
            // this group's bins from the highest down
            int acc = incl - sum;
            for (int j = P / 4 - 1; j >= 0; --j) {
                const int4 h = g4[j];
                const int hv[4] = {h.w, h.z, h.y, h.x};
                int found = -1;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (found < 0 && acc + hv[u] >= remaining) found = u;
                    else if (found < 0) acc += hv[u];
                }
                if (found >= 0) {
                    sel[0] = (uint32_t)(grp * P + 4 * j + 3 - found);
                    sel[1] = (uint32_t)acc;
                    sel[2] = (uint32_t)hv[found];
                    break;
                }
            }
        }
    }
    __syncthreads();
}

// Candidate keys are copied on chip when there are at most this many (all of
// an expert's candidates, or those sharing the threshold's first 12 bits).
constexpr int kListCap = 6144;

// Appends the keys with `in` set to list[*count...] (warp-aggregated); keys
// past the list's capacity are counted but not stored. Every lane of the warp
// must call it.
__device__ __forceinline__ void list_append(uint32_t *list, int *count, bool in, uint32_t key) {
    const int lane = threadIdx.x & 31;
    const unsigned bal = __ballot_sync(0xffffffffu, in);
    if (bal != 0) {
        int at = 0;
        if (lane == __ffs(bal) - 1) at = atomicAdd(count, __popc(bal));
        at = __shfl_sync(0xffffffffu, at, __ffs(bal) - 1);
        const int pos = at + __popc(bal & ((1u << lane) - 1u));
        if (in && pos < kListCap) list[pos] = key;
    }
}

struct RoundArgs {
    const uint32_t *keyT;   // [E][Tp] candidate keys (round_prep_kernel)
    const int32_t *counts;  // [E]   top-K counts
    int T, E, M;
    int64_t cap;            // length of perm_token (rows beyond it are never written)
    int max_tiles;          // length of the tile list
    int32_t *counts_out;    // [E]
    int32_t *offsets;       // [E+1]
    int32_t *perm_token;    // [capacity]
    int32_t *row_map;       // [T,E]
    int32_t *tiles;         // [tiles][4]
    int32_t *num_tiles;     // [1]
    uint32_t *err;
};

// Loop over the groups of 4 keys of this thread's run (unrolled when they are
// held in registers).
#define FOR_RUN(g)                                     \
    _Pragma("unroll") for (int g = 0; g < kLoopG; ++g) \
        if (g >= G) break;                             \
        else

// GM > 0: a thread's run has at most GM groups of 4 keys (T <= 4096*GM), which
// stay in registers for all passes; GM == 0: every pass reads them again.
template <int GM>
__global__ void __launch_bounds__(kRThreads, 1) round_select_kernel(RoundArgs a) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_off[kMaxE + 1];  // exclusive prefix of the rounded counts
    __shared__ int s_tb[kMaxE + 1];   // exclusive prefix of the 128-row tile counts
    __shared__ __align__(16) int s_hist[kHistWords];
    __shared__ uint32_t s_list[kListCap];
    __shared__ int s_ws[33];
    __shared__ int s_members, s_nlist;
    __shared__ uint32_t s_sel[3];     // see digit_select
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, E = a.E, M = a.M;
    const int Tp = key_stride(T);

    // rounded counts of all experts and their prefix sums: 8 experts per lane
    if (warp == 0) {
        int c8[8], t8[8], cs = 0, ts = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ex = lane * 8 + i;
            const int c = ex < E ? rounded_count(max(0, min(a.counts[ex], T)), M, T) : 0;
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
        if (lane == 31 && E == kMaxE) {
            s_off[E] = ci;
            s_tb[E] = ti;
        }
    }
    if (tid == 0) {
        s_members = 0;
        s_nlist = 0;
    }
    for (int i = tid; i < kHistWords / 4; i += kRThreads)
                reinterpret_cast<int4 *>(s_hist)[i] = make_int4(0, 0, 0, 0);

    // this expert's own rounded count, without waiting for the scan
    const int f = max(0, min(a.counts[e], T));
    const int ce = rounded_count(f, M, T);
    const int mode = ce == f ? kKeep : (ce < f ? kDown : kUp);
    const int N = mode == kDown ? ce : (mode == kUp ? ce - f : 0);
    const int ncand = mode == kDown ? f : (mode == kUp ? T - f : 0);
    const bool need_sel = N > 0;

    // this thread's run: G consecutive groups of 4 tokens
    const uint4 *keys4 = reinterpret_cast<const uint4 *>(a.keyT + (size_t)e * Tp);
    const int nq = Tp / 4;
    const int G = (nq + kRThreads - 1) / kRThreads;
    const int q0 = tid * G;
    auto load4 = [&](int g) -> uint4 {
        const int q = q0 + g;
        return q < nq ? __ldg(keys4 + q) : make_uint4(0, 0, 0, 0);
    };
    constexpr int kLoopG = GM > 0 ? GM : 0x7fffffff;
    uint4 kr[GM > 0 ? GM : 1];
    if constexpr (GM > 0) {
#pragma unroll
        for (int g = 0; g < GM; ++g) kr[g] = g < G ? load4(g) : make_uint4(0, 0, 0, 0);
    }
    auto key4 = [&](int g) -> uint4 {
        if constexpr (GM > 0) return kr[g];
        else return load4(g);
    };

    // the expert's membership must agree with counts[] (checked at the end)
    int members = 0;
    FOR_RUN(g) {
        const uint4 v = key4(g);
        const uint32_t k4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 4 * (q0 + g) + i;
            members += (t < T && ((k4[i] != 0) == (mode != kUp))) ? 1 : 0;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) members += __shfl_xor_sync(0xffffffffu, members, o);
    __syncthreads();
    if (lane == 0) atomicAdd(&s_members, members);

    const int base = s_off[e];
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

    // radix select of the N-th largest candidate key, most significant digit
    // first. Few candidates: all of them are copied on chip and take digits of
    // 11, 11 and 10 bits there. Many: a 12-bit digit over every key first, then
    // the keys of the threshold bin are copied on chip for two 10-bit digits.
    // A digit whose bin is taken whole ends the search early.
    uint32_t prefix = 0;
    int pbits = 0;  // leading bits of the threshold fixed so far
    int remaining = N, eq_count = 0;
    bool bad = false, whole = false;
    if (need_sel) {
        bool on_chip = ncand <= kListCap;
        if (on_chip) {
            FOR_RUN(g) {
                const uint4 q = key4(g);
                const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) list_append(s_list, &s_nlist, k4[i] != 0, k4[i]);
            }
        } else {
            FOR_RUN(g) {
                const uint4 q = key4(g);
                const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (k4[i] != 0) atomicAdd(&s_hist[hpad(k4[i] >> 20, 12)], 1);
            }
            __syncthreads();
            digit_select(s_hist, 12, remaining, s_sel);
            if (s_sel[0] == 0xFFFFFFFFu) {
                bad = true;
            } else {
                prefix = s_sel[0] << 20;
                pbits = 12;
                remaining -= (int)s_sel[1];
                eq_count = (int)s_sel[2];
                whole = eq_count == remaining;
                on_chip = eq_count <= kListCap;
                if (on_chip && !whole) {
                    FOR_RUN(g) {
                        const uint4 q = key4(g);
                        const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            list_append(s_list, &s_nlist, k4[i] != 0 && (k4[i] >> 20) == (prefix >> 20),
                                        k4[i]);
                    }
                }
            }
        }
        __syncthreads();
        const int nl = min(s_nlist, kListCap);
        while (!bad && !whole && pbits < 32) {
            const int W = pbits == 0 ? 11 : (pbits == 11 ? 11 : (32 - pbits > 10 ? 10 : 32 - pbits));
            const int shift = 32 - pbits - W;
            const uint32_t hm = pbits == 0 ? 0u : (0xFFFFFFFFu << (32 - pbits));
            for (int i = tid; i < kHistWords / 4; i += kRThreads)
                reinterpret_cast<int4 *>(s_hist)[i] = make_int4(0, 0, 0, 0);
            __syncthreads();
            if (on_chip) {
                for (int j2 = tid; j2 < nl; j2 += kRThreads) {
                    const uint32_t k = s_list[j2];
                    if ((k & hm) == (prefix & hm))
                        atomicAdd(&s_hist[hpad((k >> shift) & ((1u << W) - 1u), W)], 1);
                }
            } else {
                FOR_RUN(g) {
                    const uint4 q = key4(g);
                    const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (k4[i] != 0 && (k4[i] & hm) == (prefix & hm))
                            atomicAdd(&s_hist[hpad((k4[i] >> shift) & ((1u << W) - 1u), W)], 1);
                }
            }
            __syncthreads();
            digit_select(s_hist, W, remaining, s_sel);
            if (s_sel[0] == 0xFFFFFFFFu) {
                bad = true;
                break;
            }
            prefix |= s_sel[0] << shift;
            pbits += W;
            remaining -= (int)s_sel[1];
            eq_count = (int)s_sel[2];
            whole = eq_count == remaining && pbits < 32;
        }
        if (bad) {
            // fewer candidates than the count asks for (counts[] does not match
            // idx): take none; the row count check flags it
            prefix = 0xFFFFFFFFu;
            remaining = 0;
            eq_count = 0;
        } else if (whole) {
            // every key of the bin is taken: the threshold is the bin's lowest key
            prefix = prefix == 0 ? 0u : prefix - 1u;
            remaining = 0;
            eq_count = 0;
        }
    }
    const uint32_t v = prefix;
    const bool all_eq = remaining >= eq_count;

    // ordered pass: threshold ties go to the lowest tokens, then the kept tokens
    // are numbered in token order
    int eq_before = 0;
    if (need_sel && !all_eq) {
        int eq_local = 0;
        FOR_RUN(g) {
            const uint4 q = key4(g);
            eq_local += (q.x != 0 && q.x == v) + (q.y != 0 && q.y == v) + (q.z != 0 && q.z == v) +
                        (q.w != 0 && q.w == v);
        }
        int tot;
        eq_before = block_excl_sum(eq_local, s_ws, &tot);
    }
    auto kept = [&](uint32_t key, int t, int &eq_seen) -> bool {
        if (t >= T) return false;
        const bool cand = key != 0;
        if (mode == kKeep) return cand;
        bool chosen = false;
        if (cand && need_sel) {
            if (key > v) chosen = true;
            else if (key == v && remaining > 0) chosen = all_eq || (eq_before + eq_seen++ < remaining);
        }
        return mode == kDown ? chosen : (!cand || chosen);
    };
    // keep flags of this thread's run, as a bit mask when the run has <= 32 tokens
    const bool use_bits = G <= 8;
    uint32_t kbits = 0;
    int keep_local = 0;
    {
        int eq_seen = 0;
        FOR_RUN(g) {
            const uint4 q = key4(g);
            const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool k = kept(k4[i], 4 * (q0 + g) + i, eq_seen);
                keep_local += k;
                if (use_bits && k) kbits |= 1u << (4 * g + i);
            }
        }
    }
    int total;
    int row = base + block_excl_sum(keep_local, s_ws, &total);
    auto emit = [&](int t) {
        if (row < base + ce && (int64_t)row < a.cap) {
            a.perm_token[row] = t;
            a.row_map[(size_t)t * E + e] = row;
        }
        ++row;
    };
    if (use_bits) {
        while (kbits != 0) {
            const int j2 = __ffs(kbits) - 1;
            kbits &= kbits - 1;
            emit(4 * q0 + j2);
        }
    } else {
        int eq_seen = 0;
        FOR_RUN(g) {
            const uint4 q = key4(g);
            const uint32_t k4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * (q0 + g) + i;
                if (kept(k4[i], t, eq_seen)) emit(t);
            }
        }
    }
    if (tid == 0 && (total != ce || (int64_t)base + ce > a.cap || s_members != f))
        atomicOr(a.err, MOE_DEVERR_COUNT_MISMATCH);
}

constexpr int kWThreads = 256;
constexpr int kWWarps = kWThreads / 32;
constexpr int kPerLane = kMaxE / 32;
static_assert(kPerLane == 8, "the 16-byte layout covers 256 experts in two halves");

// s + c += x with the rounding error of the addition kept in c (Knuth's TwoSum).
__device__ __forceinline__ void two_sum_acc(float &s, float &c, float x) {
    const float t = __fadd_rn(s, x);
    const float bp = __fsub_rn(t, s);
    const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(x, bp));
    s = t;
    c = __fadd_rn(c, err);
}

__global__ void __launch_bounds__(kWThreads)
round_weights_kernel(const float *__restrict__ L, const int32_t *__restrict__ row_map, int T,
                     int E, int renorm, bool vec, float *__restrict__ row_w,
                     int32_t *__restrict__ tok_rows, int32_t *__restrict__ tok_n) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * kWWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    // this lane's experts: e(i) = lane + 32 i, or with 16-byte loads
    // e(i) = 128 (i / 4) + 4 lane + i % 4
    float l[kPerLane];
    int r[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        l[i] = -INFINITY;
        r[i] = -1;
    }
    if (vec) {
#pragma unroll
        for (int h = 0; h < kPerLane / 4; ++h) {
            const int e = 128 * h + 4 * lane;
            if (e < E) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(L + t * E + e));
                const int4 q = __ldg(reinterpret_cast<const int4 *>(row_map + t * E + e));
                l[4 * h] = v.x, l[4 * h + 1] = v.y, l[4 * h + 2] = v.z, l[4 * h + 3] = v.w;
                r[4 * h] = q.x, r[4 * h + 1] = q.y, r[4 * h + 2] = q.z, r[4 * h + 3] = q.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                l[i] = __ldg(L + t * E + e);
                r[i] = __ldg(row_map + t * E + e);
            }
        }
    }
    if (tok_rows != nullptr) {
        // the token's rows in ascending expert order (at most kTokCap stored)
        int n = 0;
        if (vec) {
#pragma unroll
            for (int h = 0; h < kPerLane / 4; ++h) {
                int cnt = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) cnt += r[4 * h + j] >= 0;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += x;
                }
                int pos = n + incl - cnt;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (r[4 * h + j] >= 0) {
                        if (pos < kTokCap) tok_rows[t * kTokCap + pos] = r[4 * h + j];
                        ++pos;
                    }
                n += __shfl_sync(0xffffffffu, incl, 31);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const unsigned bal = __ballot_sync(0xffffffffu, r[i] >= 0);
                const int pos = n + __popc(bal & ((1u << lane) - 1u));
                if (r[i] >= 0 && pos < kTokCap) tok_rows[t * kTokCap + pos] = r[i];
                n += __popc(bal);
            }
        }
        if (lane == 0) tok_n[t] = n;
    }
    float m_all = -INFINITY, m_kept = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        m_all = fmaxf(m_all, l[i]);
        if (r[i] >= 0) m_kept = fmaxf(m_kept, l[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        m_all = fmaxf(m_all, __shfl_xor_sync(0xffffffffu, m_all, o));
        m_kept = fmaxf(m_kept, __shfl_xor_sync(0xffffffffu, m_kept, o));
    }
    if (m_kept == -INFINITY) return;  // no expert kept this token
    // renormalised: exp(l - max over kept) / sum over kept; else the softmax over
    // all. The sum is compensated (each addition's rounding error is carried in
    // c), so it is accurate to a few fp32 ulps for any E.
    const float mref = renorm ? m_kept : m_all;
    float ex[kPerLane];
    float s = 0.f, c = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        ex[i] = expf(l[i] - mref);  // 0 for the padding slots (l = -inf)
        if (!renorm || r[i] >= 0) two_sum_acc(s, c, ex[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        two_sum_acc(s, c, s2);
        c = __fadd_rn(c, c2);
    }
    const float denom = __fadd_rn(s, c);
#pragma unroll
    for (int i = 0; i < kPerLane; ++i)
        if (r[i] >= 0) row_w[r[i]] = __fdiv_rn(ex[i], denom);
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

// Y row = bf16( sum of the n rows of Z listed in rows[], in that order ), fp32.
__device__ __forceinline__ void sum_rows(const __nv_bfloat16 *__restrict__ Z, const int *rows, int n,
                                         int d, int lane, __nv_bfloat16 *__restrict__ y) {
    const int nv = d / 8;
    uint4 *dst = reinterpret_cast<uint4 *>(y);
    for (int c = lane; c < nv; c += 32) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
        // batches of 8 rows, every load of a batch issued before the first add
        for (int i = 0; i < n; i += 8) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i + j < n)
                    v[j] = __ldg(reinterpret_cast<const uint4 *>(Z + (int64_t)rows[i + j] * d) + c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i + j < n) add_bf16x8(acc, v[j]);
        }
        uint4 out;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
        for (int u = 0; u < 4; ++u) o2[u] = __floats2bfloat162_rn(acc[2 * u], acc[2 * u + 1]);
        dst[c] = out;
    }
}

__global__ void __launch_bounds__(kCThreads)
combine_rows_kernel(const __nv_bfloat16 *__restrict__ Z, const int32_t *__restrict__ row_map,
                    const int32_t *__restrict__ tok_rows, const int32_t *__restrict__ tok_n,
                    int T, int E, int d, int64_t rows_cap, __nv_bfloat16 *__restrict__ Y) {
    pdl_wait();
    pdl_trigger();
    __shared__ int s_rows[kCWarps][kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCWarps + warp;
    if (t >= T) return;
    int *rows = s_rows[warp];
    const int nl = tok_rows != nullptr ? __ldg(tok_n + t) : kTokCap + 1;
    if (nl <= kTokCap) {
        // the compact list (already in ascending expert order)
        int r = lane < nl ? __ldg(tok_rows + t * kTokCap + lane) : -1;
        if (r >= rows_cap) r = -1;
        const unsigned bal = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) rows[__popc(bal & ((1u << lane) - 1u))] = r;
        __syncwarp();
        sum_rows(Z, rows, __popc(bal), d, lane, Y + t * d);
        return;
    }
    int rr[kMaxE / 32];
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        rr[i] = e < E ? __ldg(row_map + t * E + e) : -1;
    }
    int n = 0;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
        const int r = rr[i] < rows_cap ? rr[i] : -1;  // out of range: treated as not kept
        const unsigned bal = __ballot_sync(0xffffffffu, r >= 0);
        if (r >= 0) rows[n + __popc(bal & ((1u << lane) - 1u))] = r;
        n += __popc(bal);
    }
    __syncwarp();
    sum_rows(Z, rows, n, d, lane, Y + t * d);
}

}  // namespace

size_t round_scratch_bytes(int T, int E) { return (size_t)4 * E * key_stride(T); }

cudaError_t launch_round(const float *L, const int32_t *idx, const int32_t *counts, int T, int E,
                         int K, int M, int renorm, int32_t *counts_out, int32_t *offsets,
                         int32_t *perm_token, int32_t *row_map, float *row_w, int32_t *tiles,
                         int32_t *num_tiles, int32_t *tok_rows, int32_t *tok_n, void *scratch,
                         uint32_t *err, cudaStream_t s) {
    uint32_t *keyT = static_cast<uint32_t *>(scratch);
    // 16-byte accesses when every row of L and row_map starts 16-byte aligned
    const bool vec = (E % 4) == 0 && ((reinterpret_cast<uintptr_t>(L) |
                                       reinterpret_cast<uintptr_t>(row_map)) & 15u) == 0;
    cudaError_t e = launch_k(round_prep_kernel, dim3((unsigned)(key_stride(T) / kPT)),
                             dim3(kPThreads), 0, s, L, idx, counts, T, E, K, M, vec, keyT, row_map,
                             err);
    if (e != cudaSuccess) return e;
    RoundArgs a{};
    a.keyT = keyT;
    a.counts = counts;
    a.T = T;
    a.E = E;
    a.M = M;
    a.cap = round_capacity(T, E, K, M);
    a.max_tiles = (int)(a.cap / kTileM) + E;
    a.counts_out = counts_out;
    a.offsets = offsets;
    a.perm_token = perm_token;
    a.row_map = row_map;
    a.tiles = tiles;
    a.num_tiles = num_tiles;
    a.err = err;
    auto sel = key_stride(T) <= 4 * 4 * kRThreads ? round_select_kernel<4> : round_select_kernel<0>;
    if ((e = launch_k(sel, dim3(E), dim3(kRThreads), 0, s, a)) != cudaSuccess) return e;
    return launch_k(round_weights_kernel, dim3((unsigned)((T + kWWarps - 1) / kWWarps)),
                    dim3(kWThreads), 0, s, L, static_cast<const int32_t *>(row_map), T, E, renorm,
                    vec, row_w, tok_rows, tok_n);
}

cudaError_t launch_combine_rows(const __nv_bfloat16 *Z, const int32_t *row_map,
                                const int32_t *tok_rows, const int32_t *tok_n, int T, int E,
                                int d, int64_t rows_cap, __nv_bfloat16 *Y, cudaStream_t s) {
    return launch_k(combine_rows_kernel, dim3((unsigned)((T + kCWarps - 1) / kCWarps)),
                    dim3(kCThreads), 0, s, Z, row_map, tok_rows, tok_n, T, E, d, rows_cap, Y);
}

}  // namespace moe
