// Grouping of routed slots by expert: counts, CSR-style offsets, a stable
// permutation (rows of one expert in ascending token order) and the row-tile
// schedule of the grouped GEMMs.
//
// Pages: "混合专家模型(MoE)架构优化与SonicMoE实践" §1 (Gather by routing result;
// tiles of fixed size pad experts whose row count is not a multiple of the tile),
// §2.2 (intermediates stored grouped by expert), §3.1 (per-expert counts over
// every (t,k) choice); "稀疏矩阵乘法（SpMM）在MoE中的应用：利用Triton内核加速稀疏专家
// 的计算" §2 (CSR row offsets); "Оптимизация Triton ускоряет матричные вычисления
// для моделей Mixture-of-Experts" (persistent kernel pulling tiles from a list).
//
// Three small kernels, all deterministic (no atomics decide a position):
//  1. rank:    one warp per chunk of 32 tokens builds, for every expert, a
//              32-bit mask of the chunk's tokens that chose it; a slot's rank in
//              its chunk is the popcount of the mask below its lane, and the
//              chunk's count per expert is the mask's popcount. A slot whose
//              expert is out of range, or repeats an expert listed earlier in
//              its token's row, gets no row (rank -1) and is flagged.
//  2. scan:    one block per expert turns the chunk counts into exclusive
//              prefix sums; the last block to finish (ticket counter) scans the
//              expert totals into offsets, tile bases and the tile list (the
//              list is skipped when tiles is NULL: the whole-layer call's
//              GEMMs decode their units from the offsets).
//  3. scatter: p = offsets[e] + chunk prefix + rank; writes perm_token,
//              perm_slot and row_of_slot.
//
// For T <= kGroupMaxBlocks * kGroupMaxCpb * 32 tokens one kernel does all of it
// (group_kernel): each block takes a run of chunks, counts them per expert,
// publishes its block counts with a flag, then reads every block's counts
// (bounded waits on their flags; every block publishes before it waits and all
// blocks are resident at once, so none waits on one that cannot run). The
// expert totals give the offsets (and are checked against counts when given),
// the earlier blocks' counts each block's start within every expert; then it
// scatters. The positions are the three kernels' own.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// One warp, one chunk of 32 tokens: masks m[e] of the chunk's tokens choosing
// expert e (slots with a bad or repeated expert get none and are flagged), and
// the experts of this lane's token's slots in ek (-1: no row).
__device__ __forceinline__ void chunk_masks(const int32_t *__restrict__ idx, int T, int E, int K,
                                            int chunk, uint32_t *m, int (&ek)[kMaxK],
                                            uint32_t *ctrl) {
    const int lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) m[e] = 0u;
    __syncwarp();
    const int64_t t = (int64_t)chunk * kChunk + lane;
    const bool valid = t < T;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        ek[k] = -1;
        if (k < K && valid) {
            const int e = __ldg(idx + t * K + k);
            if (e >= 0 && e < E) {
                bool repeat = false;
#pragma unroll
                for (int k2 = 0; k2 < k; ++k2) repeat |= ek[k2] == e;
                if (repeat) {
                    if (ctrl != nullptr) atomicOr(&ctrl[kWordErr], MOE_DEVERR_REPEATED_EXPERT);
                } else {
                    ek[k] = e;
                    atomicOr(&m[e], 1u << lane);
                }
            } else if (ctrl != nullptr) {
                atomicOr(&ctrl[kWordErr], MOE_DEVERR_BAD_EXPERT);
            }
        }
    }
    __syncwarp();
}


__global__ void __launch_bounds__(kThreads)
rank_kernel(const int32_t *__restrict__ idx, int T, int E, int K, int nchunks,
            int32_t *__restrict__ rank, int32_t *__restrict__ chunk_cnt,
            uint32_t *__restrict__ ctrl) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t masks[kThreads / 32][kMaxE];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0) ctrl[kWordDone] = 0;  // ticket for the scan
    const int chunk = blockIdx.x * (kThreads / 32) + warp;
    if (chunk >= nchunks) return;
    uint32_t *m = masks[warp];
    int ek[kMaxK];
    chunk_masks(idx, T, E, K, chunk, m, ek, ctrl);
    const int64_t t = (int64_t)chunk * kChunk + lane;
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
        if (k < K && t < T) rank[t * K + k] = ek[k] >= 0 ? __popc(m[ek[k]] & below) : -1;
    for (int e = lane; e < E; e += 32) chunk_cnt[(int64_t)e * nchunks + chunk] = __popc(m[e]);
}

// Exclusive block-wide scan of one value per thread (256 threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int ws = lane < kThreads / 32 ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < kThreads / 32) warp_sums[lane] = wi - ws;  // exclusive warp offsets
        if (lane == kThreads / 32 - 1) warp_sums[kThreads / 32] = wi;
    }
    __syncthreads();
    int excl = warp_sums[warp] + incl - v;
    total = warp_sums[kThreads / 32];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kThreads)
scan_kernel(int32_t *__restrict__ chunk_cnt, int nchunks, int E, const int32_t *counts_in,
            int32_t *__restrict__ totals, int32_t *__restrict__ offsets,
            int32_t *__restrict__ tile_base, int32_t *__restrict__ tiles,
            int32_t *__restrict__ num_tiles, uint32_t *__restrict__ ctrl) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_sums[kThreads / 32 + 1];
    __shared__ bool is_last;
    const int e = blockIdx.x;
    int32_t *row = chunk_cnt + (int64_t)e * nchunks;
    int carry = 0;
    for (int c0 = 0; c0 < nchunks; c0 += kThreads) {
        const int c = c0 + threadIdx.x;
        const int v = c < nchunks ? row[c] : 0;
        int tot;
        const int ex = block_exclusive_scan(v, warp_sums, tot);
        if (c < nchunks) row[c] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) {
        totals[e] = carry;
        __threadfence();
        const uint32_t ticket = atomicAdd(&ctrl[kWordDone], 1u);
        is_last = (ticket == (uint32_t)E - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // last block: offsets, tile bases, tile list over all experts (E <= 256)
    const int ee = threadIdx.x;
    const int c = ee < E ? *((volatile int32_t *)totals + ee) : 0;
    const int ntile = (c + kTileM - 1) / kTileM;
    int tot_rows, tot_tiles;
    const int off = block_exclusive_scan(c, warp_sums, tot_rows);
    const int tb = block_exclusive_scan(ntile, warp_sums, tot_tiles);
    if (ee < E) {
        offsets[ee] = off;
        tile_base[ee] = tb;
        if (counts_in != nullptr && counts_in[ee] != c)
            atomicOr(&ctrl[kWordErr], MOE_DEVERR_COUNT_MISMATCH);
        for (int i = 0; tiles != nullptr && i < ntile; ++i) {
            int4 tv;
            tv.x = ee;
            tv.y = off + i * kTileM;
            tv.z = min(kTileM, c - i * kTileM);
            tv.w = 0;
            reinterpret_cast<int4 *>(tiles)[tb + i] = tv;
        }
    }
    if (ee == 0) {
        offsets[E] = tot_rows;
        tile_base[E] = tot_tiles;
        if (num_tiles != nullptr) num_tiles[0] = tot_tiles;
        ctrl[kWordDone] = 0;
    }
}

__global__ void __launch_bounds__(kThreads)
scatter_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ rank,
               const int32_t *__restrict__ chunk_base, const int32_t *__restrict__ offsets,
               int T, int E, int K, int nchunks, int32_t *__restrict__ perm_token,
               int32_t *__restrict__ perm_slot, int32_t *__restrict__ row_of_slot,
               uint32_t *__restrict__ ctrl) {
    pdl_wait();
    pdl_trigger();
    const int64_t slot = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t R = (int64_t)T * K;
    if (slot >= R) return;
    const int e = idx[slot];
    const int r = rank[slot];
    if (e < 0 || e >= E || r < 0) {
        row_of_slot[slot] = -1;
        return;
    }
    const int64_t t = slot / K;
    const int64_t p = (int64_t)offsets[e] + chunk_base[(int64_t)e * nchunks + t / kChunk] + r;
    if (p < 0 || p >= R) {
        atomicOr(&ctrl[kWordErr], MOE_DEVERR_BAD_EXPERT);
        row_of_slot[slot] = -1;
        return;
    }
    perm_token[p] = (int32_t)t;
    perm_slot[p] = (int32_t)slot;
    row_of_slot[slot] = (int32_t)p;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The one-kernel grouping. Block b takes chunks [b*cpb, (b+1)*cpb).
__global__ void __launch_bounds__(kThreads)
group_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ counts, int T, int E,
             int K, int nchunks, int cpb, int32_t *__restrict__ offsets,
             int32_t *__restrict__ perm_token, int32_t *__restrict__ perm_slot,
             int32_t *__restrict__ row_of_slot, int32_t *__restrict__ tiles,
             int32_t *__restrict__ num_tiles, uint32_t *__restrict__ flags,
             int32_t *__restrict__ agg, uint32_t *__restrict__ ctrl) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t masks[kThreads / 32][kMaxE];
    __shared__ int32_t pre[kGroupMaxCpb][kMaxE];  // per chunk of the block: counts, then prefixes
    __shared__ int32_t base[kMaxE];               // offsets[e] + this block's prefix over blocks
    __shared__ int warp_sums[kThreads / 32 + 1];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x;
    const int c0 = b * cpb, c1 = min(nchunks, c0 + cpb);
    const uint32_t tag = __ldcg(ctrl + kWordGroupEpoch) + 1u;
    const int64_t R = (int64_t)T * K;
    int ek[kMaxK];
    // 1. each chunk's counts per expert
    for (int c = c0 + warp; c < c1; c += kThreads / 32) {
        uint32_t *m = masks[warp];
        chunk_masks(idx, T, E, K, c, m, ek, ctrl);
        for (int e = lane; e < E; e += 32) pre[c - c0][e] = __popc(m[e]);
        __syncwarp();
    }
    __syncthreads();
    // 2. per expert: prefixes over the block's chunks, the block's count published
    int blk = 0;
    if (tid < E) {
        for (int i = 0; i < c1 - c0; ++i) {
            const int v = pre[i][tid];
            pre[i][tid] = blk;
            blk += v;
        }
        agg[(int64_t)b * E + tid] = blk;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_u32(flags + b, tag);
    // 3. every block's counts (their flags first, bounded): the expert totals
    //    give the offsets, the blocks before this one its start within each expert
    bool late = false;
    if (warp == 0) {
        const uint64_t t_start = ptx::globaltimer_ns();
        for (int j = lane; j < (int)gridDim.x; j += 32) {
            uint32_t spin = 0;
            while (ld_acquire_u32(flags + j) != tag) {
                if ((++spin & 63u) == 0 && ptx::globaltimer_ns() - t_start > 1000000000ull) {
                    late = true;
                    break;
                }
            }
        }
    }
    if (__syncthreads_or(late)) {
        if (tid == 0) atomicOr(&ctrl[kWordErr], MOE_DEVERR_TIMEOUT);
    }
    int tot_e = 0, before = 0;
    if (tid < E) {
        // (integer sums: any order gives the same result; unrolled so that the
        // loads of several blocks' counts are in flight together)
#pragma unroll 8
        for (int j = 0; j < (int)gridDim.x; ++j) {
            const int v = j == b ? blk : __ldcg(agg + (int64_t)j * E + tid);
            before += j < b ? v : 0;
            tot_e += v;
        }
    }
    int total = 0;
    const int off = block_exclusive_scan(tot_e, warp_sums, total);
    if (tid < E) {
        base[tid] = off + before;
        if (b == 0) {
            offsets[tid] = off;
            if (counts != nullptr && __ldg(counts + tid) != tot_e)
                atomicOr(&ctrl[kWordErr], MOE_DEVERR_COUNT_MISMATCH);
        }
    }
    if (b == 0 && tid == 0) offsets[E] = total;
    // tile list (only when asked for): block 0
    if (b == 0 && tiles != nullptr) {
        const int ntile = tid < E ? (tot_e + kTileM - 1) / kTileM : 0;
        int tot_tiles = 0;
        const int tb = block_exclusive_scan(ntile, warp_sums, tot_tiles);
        for (int i = 0; i < ntile; ++i) {
            int4 tv;
            tv.x = tid;
            tv.y = off + i * kTileM;
            tv.z = min(kTileM, tot_e - i * kTileM);
            tv.w = 0;
            reinterpret_cast<int4 *>(tiles)[tb + i] = tv;
        }
        if (tid == 0 && num_tiles != nullptr) num_tiles[0] = tot_tiles;
    }
    __syncthreads();
    // 4. scatter: p = offsets[e] + blocks before + chunks before + rank in the chunk
    //    (a warp with one chunk still holds its masks and experts from step 1)
    const bool one_each = c1 - c0 <= kThreads / 32;
    for (int c = c0 + warp; c < c1; c += kThreads / 32) {
        uint32_t *m = masks[warp];
        if (!one_each) chunk_masks(idx, T, E, K, c, m, ek, nullptr);
        const int64_t t = (int64_t)c * kChunk + lane;
        const uint32_t below = (1u << lane) - 1u;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
            if (k >= K || t >= T) continue;
            const int64_t slot = t * K + k;
            const int e = ek[k];
            if (e < 0) {
                row_of_slot[slot] = -1;
                continue;
            }
            const int64_t p = (int64_t)base[e] + pre[c - c0][e] + __popc(m[e] & below);
            if (p < 0 || p >= R) {  // cannot happen after a complete recount
                atomicOr(&ctrl[kWordErr], MOE_DEVERR_BAD_EXPERT);
                row_of_slot[slot] = -1;
                continue;
            }
            perm_token[p] = (int32_t)t;
            perm_slot[p] = (int32_t)slot;
            row_of_slot[slot] = (int32_t)p;
        }
        __syncwarp();
    }
    // the last block to finish moves the epoch on for the next call
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t ticket = atomicAdd(&ctrl[kWordGroupTicket], 1u);
        if (ticket == gridDim.x - 1) {
            atomicExch(&ctrl[kWordGroupTicket], 0u);
            atomicAdd(&ctrl[kWordGroupEpoch], 1u);
        }
    }
}

}  // namespace

int permute_launch_count(int T) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    return nchunks <= kGroupMaxBlocks * kGroupMaxCpb ? 1 : 3;
}

cudaError_t launch_permute(const int32_t *idx, const int32_t *counts_in, int T, int E, int K,
                           int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                           int32_t *row_of_slot, int32_t *tiles, int32_t *num_tiles,
                           const WsLayout &L, char *ws, cudaStream_t s, bool one_kernel) {
    uint32_t *ctrl = reinterpret_cast<uint32_t *>(ws + L.err);
    int32_t *rank = reinterpret_cast<int32_t *>(ws + L.rank);
    int32_t *chunk = reinterpret_cast<int32_t *>(ws + L.chunk_base);
    int32_t *totals = reinterpret_cast<int32_t *>(ws + L.totals);
    int32_t *tile_base = reinterpret_cast<int32_t *>(ws + L.tile_base);
    const int nchunks = L.nchunks;
    const int64_t R = (int64_t)T * K;
    if (one_kernel && permute_launch_count(T) == 1) {
        // blocks of at least 8 chunks (one per warp) while there are enough chunks
        int nb = std::min(kGroupMaxBlocks, std::max(1, nchunks / 8));
        int cpb = (nchunks + nb - 1) / nb;
        nb = (nchunks + cpb - 1) / cpb;
        return launch_k(group_kernel, dim3(nb), dim3(kThreads), 0, s, idx, counts_in, T, E, K,
                        nchunks, cpb, offsets, perm_token, perm_slot, row_of_slot, tiles,
                        num_tiles, reinterpret_cast<uint32_t *>(ws + L.group_flags),
                        reinterpret_cast<int32_t *>(ws + L.group_agg), ctrl);
    }
    cudaError_t err = launch_k(rank_kernel, dim3((nchunks + kThreads / 32 - 1) / (kThreads / 32)),
                               dim3(kThreads), 0, s, idx, T, E, K, nchunks, rank, chunk, ctrl);
    if (err != cudaSuccess) return err;
    err = launch_k(scan_kernel, dim3(E), dim3(kThreads), 0, s, chunk, nchunks, E, counts_in, totals,
                   offsets, tile_base, tiles, num_tiles, ctrl);
    if (err != cudaSuccess) return err;
    return launch_k(scatter_kernel, dim3((unsigned)((R + kThreads - 1) / kThreads)), dim3(kThreads),
                    0, s, idx, static_cast<const int32_t *>(rank), static_cast<const int32_t *>(chunk),
                    static_cast<const int32_t *>(offsets), T, E, K, nchunks, perm_token, perm_slot,
                    row_of_slot, ctrl);
}

}  // namespace moe
