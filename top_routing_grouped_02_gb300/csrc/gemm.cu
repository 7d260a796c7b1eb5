// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// Pages: "混合专家模型(MoE)架构优化与SonicMoE实践" §1 (two-layer expert MLP over the
// gathered rows; tile padding when a count is not a multiple of the tile),
// §2.1 (producer warps move tiles with TMA while the MMA side computes),
// §2.2 (SwiGLU fused into the GEMM epilogue), §4.2 (MMA issued by one thread,
// accumulators in TMEM, two TMEM accumulator stages so the epilogue drains one
// while the MMA fills the other); "Оптимизация Triton ускоряет матричные
// вычисления для моделей Mixture-of-Experts" (one launch covers every expert;
// persistent CTAs, one per SM, take tiles from a schedule; expert-grouped tile
// order for L2 reuse of expert weights; TMA loads of expert weights).
//
// One kernel template serves both GEMMs of the expert MLP:
//   gate/up:  acc[128 x 256] = Xg[rows, d] . [W1[e][:, 128 cols] | W3[e][:, 128 cols]]
//             H[rows, 128 cols] = bf16( SiLU(gate) * up )
//   down:     acc[128 x 256] = H[rows, n] . W2[e][:, 256 cols]
//             Z[rows, 256 cols] = bf16( w_row * acc )
// A unit of work is (expert, 128-row tile of that expert, 256-column block).
// Units are ordered expert-major, then column block, then row tile, and CTA b
// takes units b, b + gridDim.x, ...: CTAs running at the same time share one
// expert's weight block through L2 while its few activation tiles stay hot.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: A tile 128x64 (K-major) and B tile 64x256
//               (MN-major, four 64-column boxes) per stage, 128-byte swizzle.
//   warp 1      MMA issuer: one thread issues 4 x tcgen05.mma (M128 N256 K16)
//               per stage into the current TMEM accumulator, commits the stage
//               back to the producer and, after the last stage, the
//               accumulator to the epilogue.
//   warp 2      allocates / frees 512 TMEM columns (2 accumulators x 256).
//   warps 4-7   epilogue: tcgen05.ld of their 32 TMEM lanes (= tile rows),
//               activation or scaling in fp32, bf16 stores.
// Every wait is bounded (about one second); a wait that gives up sets
// MOE_DEVERR_TIMEOUT in the error word and that role stops. Before the TMEM is
// released, in-flight MMAs and TMA loads of a stopped role are drained.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int BM = kTileM;  // 128 rows
constexpr int BK = 64;      // reduction depth per stage (128 bytes of bf16)
constexpr int BN = 256;     // accumulator columns per unit
constexpr int kStages = 4;
constexpr uint32_t kABytes = BM * BK * 2;               // 16 KB
constexpr uint32_t kBBox = BK * 64 * 2;                 // 8 KB: 64 k-rows x 64 columns
constexpr uint32_t kBBytes = 4 * kBBox;                 // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;     // 48 KB
constexpr uint32_t kTmemCols = 2 * BN;                  // two accumulators
constexpr uint32_t kIdesc = ptx::idesc_bf16(BM, BN, /*A MN-major*/ false, /*B MN-major*/ true);
constexpr uint64_t kWaitLimitNs = 1000000000ull;

enum Mode : int { kGateUp = 0, kDown = 1 };

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t tile_base[kMaxE + 1];
    int32_t offsets[kMaxE + 1];
    int32_t scan[kThreads / 32 + 1];
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + sizeof(Ctl);

struct GemmArgs {
    const int32_t *offsets;  // [E+1] grouped row offsets
    int E;
    int R;                   // rows of A / out (T*K)
    int Kdim;                // reduction length (d for gate/up, n for down)
    int NB;                  // column blocks per row tile
    __nv_bfloat16 *out;      // H [R, n] or Z [R, d]
    int out_ld;              // row length of out (elements)
    const float *topk_w;     // down only: routing weights [T*K]
    const int32_t *perm_slot;// down only: slot of each grouped row
    uint32_t *err;           // device error word
};

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, uint32_t *err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0 && ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, MOE_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Unit u -> (expert, column block, first row, rows). tile_base[e] counts the
// 128-row tiles of experts before e; empty experts own no units.
__device__ __forceinline__ void decode_unit(int u, int NB, int E, const int32_t *tb,
                                            const int32_t *off, int &e, int &nb, int &row0,
                                            int &rows) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb[mid] * NB <= u) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int m_e = tb[e + 1] - tb[e];
    const int local = u - tb[e] * NB;
    nb = local / m_e;
    const int mt = local - nb * m_e;
    row0 = off[e] + mt * BM;
    rows = min(BM, off[e + 1] - row0);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + (size_t)kStages * kStageBytes);
    const uint32_t smem_base = ptx::smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = args.E;

    // ---- setup: barriers, TMEM, tile bases --------------------------------
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&ctl->tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->tempty[a]), 4);
        }
        ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB0);
        if (MODE == kGateUp) ptx::prefetch_tensormap(&tmB1);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    {
        // tile bases: exclusive scan of ceil(rows_e / 128) over experts
        const int e = tid;
        int c = 0;
        bool bad = false;
        if (e < E) {
            const int o0 = args.offsets[e], o1 = args.offsets[e + 1];
            ctl->offsets[e] = o0;
            bad = o0 < 0 || o1 < o0 || o1 > args.R || (e == 0 && o0 != 0);
            c = bad ? 0 : (o1 - o0 + BM - 1) / BM;
        }
        if (e == 0) ctl->offsets[E] = args.offsets[E];
        // offsets must be a non-decreasing split of [0, R); otherwise do no work
        if (__syncthreads_or(bad)) {
            if (tid == 0) atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
            c = 0;
        }
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) ctl->scan[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int ws = lane < kThreads / 32 ? ctl->scan[lane] : 0;
            int wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += v;
            }
            if (lane < kThreads / 32) ctl->scan[lane] = wi - ws;
            if (lane == kThreads / 32 - 1) ctl->scan[kThreads / 32] = wi;
        }
        __syncthreads();
        if (e < E) ctl->tile_base[e] = ctl->scan[warp] + incl - c;
        if (e == 0) ctl->tile_base[E] = ctl->scan[kThreads / 32];
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int NB = args.NB;
    const int total_units = ctl->tile_base[E] * NB;
    const int KB = args.Kdim / BK;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer --
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            int e, nb, row0, rows;
            decode_unit(u, NB, E, ctl->tile_base, ctl->offsets, e, nb, row0, rows);
            const int wrow = e * args.Kdim;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!bounded_wait(ptx::smem_addr(&ctl->empty[s]), ph ^ 1u, args.err)) {
                    ok = false;
                    break;
                }
                const uint32_t full = ptx::smem_addr(&ctl->full[s]);
                const uint32_t sA = smem_base + s * kStageBytes, sB = sA + kABytes;
                ptx::mbar_arrive_expect_tx(full, kStageBytes);
                ptx::tma_load_2d(sA, &tmA, full, kb * BK, row0);
                if (MODE == kGateUp) {
                    ptx::tma_load_2d(sB + 0 * kBBox, &tmB0, full, nb * 128, wrow + kb * BK);
                    ptx::tma_load_2d(sB + 1 * kBBox, &tmB0, full, nb * 128 + 64, wrow + kb * BK);
                    ptx::tma_load_2d(sB + 2 * kBBox, &tmB1, full, nb * 128, wrow + kb * BK);
                    ptx::tma_load_2d(sB + 3 * kBBox, &tmB1, full, nb * 128 + 64, wrow + kb * BK);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        ptx::tma_load_2d(sB + q * kBBox, &tmB0, full, nb * BN + q * 64,
                                         wrow + kb * BK);
                }
            }
        }
        if (!ok) {
            // drain the loads that may still be landing in shared memory
            const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
            for (uint32_t j = first; j < it; ++j)
                bounded_wait(ptx::smem_addr(&ctl->full[j % kStages]), (j / kStages) & 1u, args.err);
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------------ MMA issuer --
        uint32_t it = 0, uc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++uc) {
            const uint32_t a = uc & 1u, aph = (uc >> 1) & 1u;
            if (!bounded_wait(ptx::smem_addr(&ctl->tempty[a]), aph ^ 1u, args.err)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + a * BN;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const uint32_t s = it % kStages, ph = (it / kStages) & 1u;
                if (!bounded_wait(ptx::smem_addr(&ctl->full[s]), ph, args.err)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sA = smem_base + s * kStageBytes, sB = sA + kABytes;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    const uint64_t adesc = ptx::desc_sw128(sA + k * 32, 16, 1024);
                    const uint64_t bdesc = ptx::desc_sw128(sB + k * 2048, kBBox, 1024);
                    ptx::tc_mma_f16(d_tmem, adesc, bdesc, kIdesc, (kb | k) != 0);
                }
                ptx::tc_commit(ptx::smem_addr(&ctl->empty[s]));
            }
            if (!ok) break;
            ptx::tc_commit(ptx::smem_addr(&ctl->tfull[a]));
        }
        if (!ok) {
            ptx::tc_commit(ptx::smem_addr(&ctl->drain));
            bounded_wait(ptx::smem_addr(&ctl->drain), 0, args.err);
        }
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue --
        const int q = warp - 4;  // TMEM lanes 32q..32q+31 = tile rows
        const int r = q * 32 + lane;
        uint32_t uc = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++uc) {
            int e, nb, row0, rows;
            decode_unit(u, NB, E, ctl->tile_base, ctl->offsets, e, nb, row0, rows);
            const uint32_t a = uc & 1u, aph = (uc >> 1) & 1u;
            if (!bounded_wait(ptx::smem_addr(&ctl->tfull[a]), aph, args.err)) break;
            ptx::tc_fence_after();
            const bool valid = r < rows;
            const int64_t p = (int64_t)row0 + r;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * BN;
            if (MODE == kGateUp) {
                __nv_bfloat16 *dst = args.out + p * args.out_ld + nb * 128;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], v[32];
                    ptx::tmem_ld32(taddr + c * 32, g);
                    ptx::tmem_ld32(taddr + 128 + c * 32, v);
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                        const float u0 = __uint_as_float(v[2 * i]), u1 = __uint_as_float(v[2 * i + 1]);
                        const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
                        const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
                        packed[i] = pack_bf16x2(h0, h1);
                    }
                    if (valid) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                               packed[4 * i + 3]);
                    }
                }
            } else {
                float w = 0.f;
                if (valid) {
                    const int slot = __ldg(args.perm_slot + p);
                    if (slot >= 0 && slot < args.R) w = __ldg(args.topk_w + slot);
                    else atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
                }
                __nv_bfloat16 *dst = args.out + p * args.out_ld + nb * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(taddr + c * 32, v);
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]),
                                                w * __uint_as_float(v[2 * i + 1]));
                    if (valid) {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                               packed[4 * i + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl->tempty[a]));
        }
    }

    // ---- teardown -----------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 2) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------ host side --

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box box_cols x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                        const GemmArgs &args, int max_units, cudaStream_t s) {
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int grid = max(1, min(sm_count(), max_units));
    grouped_gemm_kernel<MODE><<<grid, kThreads, kSmemBytes, s>>>(a, b0, b1, args);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gate_up(const __nv_bfloat16 *Xg, const __nv_bfloat16 *W1,
                                const __nv_bfloat16 *W3, const int32_t *offsets, int R, int d,
                                int E, int n, __nv_bfloat16 *H, uint32_t *err, cudaStream_t s) {
    CUtensorMap ta, tb0, tb1;
    if (!make_map(&ta, Xg, d, R, 64, BM) || !make_map(&tb0, W1, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&tb1, W3, n, (uint64_t)E * d, 64, BK))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = d;
    args.NB = n / 128;
    args.out = H;
    args.out_ld = n;
    args.err = err;
    const int max_units = (R / BM + E) * args.NB;
    return launch_gemm<kGateUp>(ta, tb0, tb1, args, max_units, s);
}

cudaError_t launch_gemm_down(const __nv_bfloat16 *H, const __nv_bfloat16 *W2,
                             const float *topk_w, const int32_t *perm_slot,
                             const int32_t *offsets, int R, int d, int E, int n,
                             __nv_bfloat16 *Z, uint32_t *err, cudaStream_t s) {
    CUtensorMap ta, tb0;
    if (!make_map(&ta, H, n, R, 64, BM) || !make_map(&tb0, W2, d, (uint64_t)E * n, 64, BK))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = n;
    args.NB = d / BN;
    args.out = Z;
    args.out_ld = d;
    args.topk_w = topk_w;
    args.perm_slot = perm_slot;
    args.err = err;
    const int max_units = (R / BM + E) * args.NB;
    return launch_gemm<kDown>(ta, tb0, tb0, args, max_units, s);
}

}  // namespace moe
