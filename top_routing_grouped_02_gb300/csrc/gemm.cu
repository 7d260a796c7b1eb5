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
// One kernel template serves both GEMMs of the expert MLP (and, fused, both at once):
//   gate/up:  acc[128 x 256] = X[perm_token[rows], d] . [W1[e][:, 128 cols] | W3[e][:, 128 cols]]
//             H[rows, 128 cols] = bf16( SiLU(gate) * up )
//   down:     acc[128 x 256] = H[rows, n] . W2[e][:, 256 cols]
//             Z[rows, 256 cols] = bf16( w_row * acc )
// A unit of work is (expert, 128-row tile of that expert, 256-column block).
// Units are ordered expert-major, then by groups of up to 16 row tiles, then
// column block, then row tile within the group, and CTA b takes units b,
// b + gridDim.x, ...: CTAs running at the same time share one expert's weight
// block through L2 while the group's activation tiles stay hot. The units are
// decoded from the offsets on the device (no host synchronisation and no tile
// list); this static stride leaves each SM busy to within 2.3% (gate/up) and
// 6.5% (down) of the busiest one on the DeepSeek-V3-shaped layer, the most that
// taking tiles dynamically from a device list could recover.
// Experts with at most two tiles (one pair) read a weight block per one or two
// units, faster than HBM delivers at tensor-core pace; their units are spread
// evenly through the sequence of the others, so each wave of CTAs mixes
// weight-streaming units with compute-bound ones.
//
// Two variants share the code. Single CTA: M=128 tiles, B tile 64x256 per stage
// (48 KB stages, 4 deep). CTA pair (a cluster of 2 CTAs on one SM pair,
// tcgen05 cta_group::2): the even CTA issues M=256 MMAs over both CTAs' 128 A
// rows, each CTA loads half of B (32 KB stages, 6 deep), both CTAs' TMA loads
// complete on the even CTA's barrier, MMA completion is multicast to both, and
// both CTAs' epilogues release the accumulator to the even CTA.
//
// Warp roles (128 + 32 * EW threads):
//   warp 0      TMA producer: B tile 64x256 (MN-major, four 64-column boxes;
//               two per CTA of a pair) per stage, 128-byte swizzle, and the A
//               tile 128x64 (K-major) unless the A rows are gathered.
//   warps 2-3   single-CTA gate/up only: gather the A tile's 128 token rows
//               straight from X (cp.async into the same 128-byte-swizzled K-major
//               layout), so no gathered copy of X goes through HBM. The token
//               indices of the next unit are loaded while the current unit is
//               copied, so no unit boundary waits on them. (CTA pairs load A by
//               TMA from rows gathered beforehand: measured faster.)
//   warp 1      MMA issuer: one thread issues 4 x tcgen05.mma (M128 N256 K16)
//               per stage into the current TMEM accumulator, commits the stage
//               back to the producer and, after the last stage, the
//               accumulator to the epilogue.
//   warp 2      allocates / frees 512 TMEM columns (2 accumulators x 256).
//   warps 4..    epilogue, EW = 4, 8 or 12 warps: warp w reads TMEM lanes
//               32(w%4)..+31 (= tile rows); with 8 or 12 the 2 or 3 warps of
//               each lane quadrant split the columns: tcgen05.ld of the lanes,
//               activation or scaling in fp32, bf16 packing; each 32 x 32
//               chunk goes through a swizzled shared-memory buffer and one TMA
//               store (whole 64-byte row segments instead of 32 half-sector
//               writes per store instruction); a warp whose 32 rows cross the
//               end of the expert's rows stores its valid rows directly.
//
// Fused expert MLP (MODE kFused, single CTA, on request only): one persistent
// launch runs the units of both GEMMs, so that on every SM the down units'
// short main loops and long epilogues (Z writes) can overlap the gate/up units'
// long main loops through the two TMEM accumulators. On the SonicMoE-shaped
// layer it measured slower than the two launches: both unit kinds wait on the
// same operand latency, which interleaving does not hide. The unit sequence is a list of rounds, one unit per CTA in each, every
// round drawn from one GEMM, so that all CTAs run the same kind of unit at the
// same time. A down unit reads the H tile that the n/128 gate/up units of its
// row tile wrote; each of their epilogue warps, once its TMA stores of that tile
// are complete, adds one to the tile's counter word in the workspace, and the
// producer of the down unit waits (bounded) for the full count before it loads
// H. The schedule places a down round only after the gate/up round holding its
// last dependency, a few rounds back, so these waits are rare. A unit only
// waits on units placed earlier in the sequence, which every CTA takes in
// order, and all CTAs are resident together (one per SM), so the waits always
// end. Counter words carry the launch's epoch (a control word the last CTA to
// finish advances), so they are never cleared.
//
// Every wait is bounded (about one second); a wait that gives up sets
// MOE_DEVERR_TIMEOUT in the error word and that role stops. Before the TMEM is
// released, in-flight MMAs and TMA loads of a stopped role are drained.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// Epilogue warps: 4, or 8 when a tile's main loop is short (see choose_ew).
// A launch has 128 + 32 * EW threads.
constexpr int kMaxThreads = 128 + 32 * 12;
template <int EW>
constexpr int threads_of() { return 128 + 32 * EW; }
constexpr int BM = kTileM;  // 128 rows per CTA
constexpr int BK = 64;      // reduction depth per stage (128 bytes of bf16)
constexpr int BN = 256;     // accumulator columns per unit
#ifndef MOE_GEMM_STAGES
#define MOE_GEMM_STAGES 4
#endif
#ifndef MOE_GEMM_PAIR_STAGES
#define MOE_GEMM_PAIR_STAGES 6
#endif
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBox = BK * 64 * 2;    // 8 KB: 64 k-rows x 64 columns
constexpr uint32_t kTmemCols = 2 * BN;     // two accumulators
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kMaxStages = MOE_GEMM_STAGES > MOE_GEMM_PAIR_STAGES ? MOE_GEMM_STAGES
                                                                   : MOE_GEMM_PAIR_STAGES;

// Per-variant geometry. Single CTA: B tile 64 x 256 (four boxes), 48 KB stages.
// CTA pair: each CTA holds its own 128 A rows and half of B (64 x 128, two
// boxes), 32 KB stages, so the same shared memory holds more stages.
template <bool PAIR>
struct Geo {
    static constexpr int kStages = PAIR ? MOE_GEMM_PAIR_STAGES : MOE_GEMM_STAGES;
    static constexpr int kBBoxes = PAIR ? 2 : 4;
    static constexpr uint32_t kStageBytes = kABytes + kBBoxes * kBBox;

};

// kGateUpPre: gate/up that also keeps the pre-activations A1 = x W1[e] and
// A3 = x W3[e] (fp32, the accumulators as they are) beside H, for the backward. kDH: the backward's
// dH' = dY[t_p] W2[e]^T (B = W2[e] read K-major, rows of dY gathered like X),
// whose epilogue forms dA1, dA3 and the routing-weight gradient's partial sums.
// kDX: the backward's dXg = dA1 W1[e]^T + dA3 W3[e]^T over the grouped rows,
// one reduction of 2n (dA1 against W1[e], then dA3 against W3[e], both weights
// read K-major), stored as bf16 like Z.
// kDW13, kDW2: the weight gradients, one unit per (expert, 128 output rows,
// output columns) with the expert's rows as the reduction (64 per k-block);
// both operands MN-major, loaded by TMA:
//   kDW13: dW1[e] | dW3[e] (d x n, 128 + 128 columns) = Xg^T [dA1 | dA3]
//   kDW2:  dW2[e] (n x d, 256 columns) = H^T (w dY)g
// One operand of each is a row-padded copy (each expert's rows start on a
// 64-row boundary, zeros after its last row): Xg for kDW13, w-scaled dY rows
// for kDW2, so the k-block past an expert's last row adds nothing although its
// other operand then reads the next expert's rows. Outputs are fp32.
enum Mode : int {
    kGateUp = 0, kDown = 1, kFused = 2, kGateUpPre = 3, kDH = 4, kDX = 5, kDW13 = 6, kDW2 = 7
};

// Instruction descriptor: B is MN-major (the forward's weights, K rows of N
// contiguous columns) except for kDH, whose W2[e] rows are n-major with the
// reduction dimension d contiguous (K-major).
template <int MODE, bool PAIR>
constexpr uint32_t idesc_of() {
    return ptx::idesc_bf16(PAIR ? 2 * BM : BM, BN, /*A MN-major*/ MODE == kDW13 || MODE == kDW2,
                           /*B MN-major*/ MODE != kDH && MODE != kDX);
}

// Single-CTA gate/up A rows are gathered by warps 2 and 3 with 16-byte cp.async.
// Each lane waits for its own copies and fences them for the async proxy, the
// warp synchronises, and one lane arrives on the stage barrier (release); the
// warps signal kGatherLag stages behind their issue so several stages are in
// flight.
constexpr int kGatherWarps = 2;
#ifndef MOE_GEMM_GATHER_LAG
#define MOE_GEMM_GATHER_LAG 2
#endif
constexpr int kGatherLag = MOE_GEMM_GATHER_LAG;

// An expert's work tiles run in groups of kGroupTiles: a group takes every
// column block before the next group starts, so the A rows live in L2 at once
// are a group's (at most 16 x 128 rows) instead of all of a heavy expert's,
// at the price of reading that expert's weight blocks once per group. With a
// gathered A, its copies also carry an L2 evict-last policy: every X row is
// read once per column block of every expert that chose it, the weights once
// per group. Measured on the DeepSeek-V3-shaped layer (Zipf-skewed experts of
// up to about 40 tiles): gate/up DRAM reads 16.17 -> 14.03 GB, 3.32 -> 3.13 ms;
// layers whose experts hold at most 16 tiles (Mixtral, SonicMoE) are unchanged.
// (An evict-first policy on the weights and an evict-last one on TMA-loaded A
// rows measured slower on every shape.)
#ifndef MOE_GEMM_GROUP_TILES
#define MOE_GEMM_GROUP_TILES 16
#endif
constexpr int kGroupTiles = MOE_GEMM_GROUP_TILES;
#ifndef MOE_GEMM_GATHER_HINT
#define MOE_GEMM_GATHER_HINT 1
#endif

// Most rounds (unit positions / CTAs) a fused launch may have; the host runs
// the two GEMMs apart when the bound on its units exceeds them.
constexpr int kMaxRounds = 256;

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t tile_base[2][kMaxE + 1];  // work-tile bases: [0] heavy experts, [1] light
    int32_t offsets[kMaxE + 1];
    uint64_t scan[kMaxThreads / 32 + 1];
    uint32_t tag;  // fused: this launch's epoch, shifted into counter-word position
    int nrounds;   // fused: rounds of the unit sequence
    int32_t sched[kMaxRounds];  // fused: per round, bit 30 = down, low bits = round in its stream
    int16_t need[kMaxRounds];   // fused: per down round, the gate/up round of its last dependency
    int16_t gpos[kMaxRounds];   // fused: round at which each gate/up round was placed
};

// Epilogue staging: 32-row x 32-column bf16 buffers (64-byte rows, 64-byte
// swizzle) that TMA stores write out: two per warp with 4 epilogue warps, one
// per warp with 8 or 12.
constexpr uint32_t kEpiBuf = 32 * 32 * 2;
template <int EW>
constexpr int epi_bufs() { return EW > 8 ? EW : 8; }
template <bool PAIR, int EW>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)Geo<PAIR>::kStages * Geo<PAIR>::kStageBytes +
           (size_t)epi_bufs<EW>() * kEpiBuf + sizeof(Ctl);
}

struct GemmArgs {
    const __nv_bfloat16 *X;     // gate/up only: token rows [T, d], gathered in-kernel
    const int32_t *perm_token;  // gate/up only: token of each grouped row
    int T;                      // gate/up only: number of tokens
    const int32_t *offsets;   // [E+1] grouped row offsets
    int E;
    int R;                    // rows of A / out (T*K)
    int Kdim;                 // reduction length (d for gate/up, n for down)
    int NB;                   // column blocks per row tile
    __nv_bfloat16 *out;       // H [R, n] or Z [R, d]
    int out_ld;               // row length of out (elements)
    const float *topk_w;      // down only: routing weights [T*K]
    const int32_t *perm_slot; // down only: slot of each grouped row (NULL: the row itself)
    uint32_t *err;            // device error word, followed by the control words
    // fused only: the down units' reduction length (n), column blocks (d / 256)
    // and output Z [R, d]; the row-tile counters; the rounds kept between a
    // gate/up round and the first down round that reads its H tiles
    int Kdim2;
    int NB2;
    __nv_bfloat16 *out2;
    int out2_ld;
    uint32_t *dep;
    int gap_rounds;
    float *outf;  // kDX with f32_out: fp32 outputs [rows, out_ld] (tmOut is an fp32 map)
    int f32_out;
    // kGateUpPre: the pre-activation outputs A1, A3 [R, n] fp32; kDH: dA3 (dA1
    // goes to out)
    float *pre_out1;
    float *pre_out3;
    __nv_bfloat16 *out3;
    // kDH: the pre-activations A1, A3 [R, n] fp32 (row length out_ld), rows of
    // W2[e] per expert (n), and the per-(row, 32-column chunk) partial sums of
    // dS [R, ds_ld]
    const float *pre1;
    const float *pre3;
    int bn_rows;  // kDH, kDX: rows of the K-major weight per expert
    int kb_half;  // kDX: k-blocks of the first half of the reduction (n / 64)
    // kDW13 / kDW2: 128-row output tiles per expert and the output rows per
    // expert (the outputs go through the output tensor maps)
    int MT;
    int wout_rows;
    float *dspart;
    int ds_ld;
    // nonzero: the output's TMA stores carry an L2 evict-first hint (outputs no
    // later kernel reads soon, such as the weight gradients)
    int out_evict_first;
};

// Counter words of the fused kernel: the launch's epoch in the high 24 bits, the
// arrivals of this launch in the low 8.
constexpr uint32_t kDepCountBits = 8;

// Polls one of this CTA's barriers (acquire at CTA scope; arrivals from the
// peer CTA of a pair are made with cluster-scope release).
template <bool PAIR>
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

// Experts with few work tiles share each weight block among few units, so their
// units need more weight bytes per FLOP than HBM delivers at tensor-core pace;
// experts with many tiles are compute-bound. Position p of the unit sequence
// therefore interleaves two streams: the light experts' units sit at evenly
// spread positions (a Bresenham split of the N positions, L of them light) and
// the heavy experts' units fill the rest, so every wave of CTAs mixes both.
// With no light expert the sequence is the heavy stream itself.
// An expert is light when it has at most light_tiles<PAIR>() work tiles (two
// 128-row tiles, or one tile pair).
template <bool PAIR>
constexpr int light_tiles() { return PAIR ? 1 : 2; }

// Position p -> (expert, column block, first row, rows). Within a stream,
// tile_base[st][e] counts the work tiles of that stream's experts before e
// (128-row tiles, or pairs of them for a CTA pair, whose CTA `rank` takes the
// pair's tile 2*pt + rank); units run expert-major, then column block, then row
// tile, and experts outside the stream own no units in it. `rows` can be <= 0
// for the second tile of an odd pair.
__device__ __forceinline__ void decode_unit(int p, int NB, int E, const int32_t (*tbs)[kMaxE + 1],
                                            const int32_t *off, int per_tile, int rank, int &e,
                                            int &nb, int &row0, int &rows) {
    const uint64_t L = (uint64_t)tbs[1][E] * NB;
    int st = 0, u = p;
    if (L != 0) {
        const uint64_t N = (uint64_t)tbs[0][E] * NB + L;
        const uint64_t pl = (uint64_t)p * L;
        uint64_t a, a1;  // light positions before p and before p + 1
        if (N * L <= 0xffffffffull) {
            a = (uint32_t)pl / (uint32_t)N;
            a1 = (uint32_t)(pl + L) / (uint32_t)N;
        } else {
            a = pl / N;
            a1 = (pl + L) / N;
        }
        st = a1 != a ? 1 : 0;
        u = st ? (int)a : p - (int)a;
    }
    const int32_t *tb = tbs[st];
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb[mid] * NB <= u) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int m_e = tb[e + 1] - tb[e];
    const int local = u - tb[e] * NB;
    // groups of kGroupTiles work tiles: a group runs all column blocks before
    // the next group starts (the last group holds the remainder)
    const int nfull = m_e / kGroupTiles;
    const int k = min(local / (kGroupTiles * NB), nfull);
    const int gs = k < nfull ? kGroupTiles : m_e - nfull * kGroupTiles;
    const int go = local - k * kGroupTiles * NB;
    nb = go / gs;
    const int pt = k * kGroupTiles + (go - nb * gs);
    row0 = off[e] + (pt * per_tile + rank) * BM;
    rows = min(BM, off[e + 1] - row0);
}

// A unit as every role sees it: which GEMM (down or gate/up), expert, column
// block, first row, rows, and (fused) the row tile's index among all tiles.
struct Unit {
    bool valid;  // false: an empty position of the fused sequence
    bool down;
    int e, nb, row0, rows, tile;
    int kbs;       // k-blocks of the unit's main loop
    int poff, off;  // weight gradients: the expert's first padded row and first row
};

// Fused sequence. Each stream (gate/up units, down units) runs expert-major,
// then column block, then row tile. The sequence is a list of rounds of
// gridDim.x positions, one per CTA, each round taken from one stream, so all
// CTAs run the same kind of unit at the same time and progress alike; position
// p = round * gridDim.x + CTA. sched[r] names round r's stream and its round
// within the stream; a position past the end of its stream is empty.
// tb: row-tile bases of all experts.
__device__ __forceinline__ Unit decode_sched(int p, int NBg, int NBd, int E,
                                             const int32_t *sched, const int32_t *tb,
                                             const int32_t *off) {
    Unit u;
    const int G = (int)gridDim.x;
    const int r = p / G;
    const int32_t sr = sched[r];
    u.down = (sr >> 30) & 1;
    const int NBs = u.down ? NBd : NBg;
    const int i = (sr & 0x3fffffff) * G + (p - r * G);
    u.valid = i < tb[E] * NBs;
    if (!u.valid) return u;
    int lo = 0, hi = E - 1;  // the last expert whose units start at or before i
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tb[mid] * NBs <= i) lo = mid; else hi = mid - 1;
    }
    u.e = lo;
    const int m = tb[lo + 1] - tb[lo];
    const int local = i - tb[lo] * NBs;
    u.nb = local / m;
    const int rt = local - u.nb * m;
    u.tile = tb[lo] + rt;
    u.row0 = off[lo] + rt * BM;
    u.rows = min(BM, off[lo + 1] - u.row0);
    return u;
}

// Fused: one epilogue warp's H stores of a row tile are complete (release; the
// caller fences first). A word of this launch's epoch takes one atomic add; one
// still carrying an older epoch is replaced by this epoch's first arrival
// (compare-and-swap, which fails, and the add follows, once another warp has).
__device__ __forceinline__ void dep_arrive(uint32_t *w, uint32_t tag) {
    uint32_t old = *reinterpret_cast<volatile uint32_t *>(w);
    while ((old >> kDepCountBits) != (tag >> kDepCountBits)) {
        const uint32_t prev = atomicCAS(w, old, tag | 1u);
        if (prev == old) return;
        old = prev;
    }
    atomicAdd(w, 1u);
}

// Fused: waits (bounded) until a row tile's counter word reads `want`.
__device__ __forceinline__ bool dep_wait(const uint32_t *w, uint32_t want, uint32_t *err) {
    if (ptx::ld_acquire_gpu(w) == want) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        __nanosleep(32);
        if (ptx::ld_acquire_gpu(w) == want) return true;
        if ((spin & 15u) == 0 && ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(err, MOE_DEVERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int MODE, bool PAIR, int EW>
__global__ void __launch_bounds__(threads_of<EW>(), 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmOut,
                    const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmOut2,
                    const GemmArgs args) {
    using G = Geo<PAIR>;
    constexpr int S = G::kStages;
    constexpr int kThreads = threads_of<EW>();
    // epilogue warps signalling an accumulator release (both CTAs of a pair)
    constexpr uint32_t kTemptyCount = PAIR ? 2 * EW : EW;
    constexpr int kNBuf = epi_bufs<EW>() / EW;  // staging buffers per epilogue warp
    // fused: both GEMMs' units in one launch (single CTA only); the maps are
    // tmA = H (A of down units), tmB0/tmB1 = W1/W3, tmOut = H (stores),
    // tmB2 = W2, tmOut2 = Z (stores)
    constexpr bool FUSED = MODE == kFused;
    static_assert(!(FUSED && PAIR), "the fused kernel runs single CTAs");
    // A rows gathered in the kernel (single-CTA gate/up units) or loaded by TMA
    constexpr bool GATHER = (MODE == kGateUp || MODE == kGateUpPre || MODE == kDH || FUSED) && !PAIR;
    constexpr bool GATE = MODE == kGateUp || MODE == kGateUpPre;  // gate/up B boxes (W1 | W3)
    constexpr bool WGRAD = MODE == kDW13 || MODE == kDW2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + (size_t)S * G::kStageBytes +
                                       (size_t)epi_bufs<EW>() * kEpiBuf);
    const uint32_t smem_base = ptx::smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = args.E;
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int first_unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int unit_stride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    // ---- setup: barriers, TMEM, tile bases --------------------------------
    if (tid == 0) {
        // full[s]: the TMA producer's arrive (+ one per gatherer warp)
        const uint32_t full_count = 1 + (GATHER ? kGatherWarps : 0);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), full_count);
            ptx::mbar_init(ptx::smem_addr(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&ctl->tfull[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->tempty[a]), kTemptyCount);
        }
        ptx::mbar_init(ptx::smem_addr(&ctl->drain), 1);
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        if (!GATHER) ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB0);
        if (GATE || FUSED || MODE == kDX || MODE == kDW13) ptx::prefetch_tensormap(&tmB1);
        if (MODE == kDX || MODE == kGateUpPre) ptx::prefetch_tensormap(&tmB2);
        if (MODE == kGateUpPre) ptx::prefetch_tensormap(&tmOut2);
        ptx::prefetch_tensormap(&tmOut);
        if (MODE == kDH || MODE == kDW13) ptx::prefetch_tensormap(&tmOut2);
        if (FUSED) {
            ptx::prefetch_tensormap(&tmA);
            ptx::prefetch_tensormap(&tmB2);
            ptx::prefetch_tensormap(&tmOut2);
        }
    }
    if (warp == 2) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    // barriers, TMEM and tensor maps are set up; from here on global memory
    // written by the previous kernel is read
    pdl_wait();
    pdl_trigger();
    {
        // work-tile bases: exclusive scan over experts of ceil(rows_e / 128)
        // tiles (single CTA) or of ceil(tiles_e / 2) tile pairs (CTA pair)
        const int e = tid;
        int c = 0;
        bool bad = false;
        if (e < E) {
            const int o0 = args.offsets[e], o1 = args.offsets[e + 1];
            ctl->offsets[e] = o0;
            bad = o0 < 0 || o1 < o0 || o1 > args.R || (e == 0 && o0 != 0);
            // weight gradients: the expert's 64-row k-blocks (their prefix gives
            // the padded row offsets); otherwise its 128-row tiles
            c = bad ? 0 : WGRAD ? (o1 - o0 + BK - 1) / BK : (o1 - o0 + BM - 1) / BM;
            if (PAIR && !WGRAD) c = (c + 1) / 2;  // tile pairs (k-blocks stay k-blocks)
        }
        if (e == 0) ctl->offsets[E] = args.offsets[E];
        // offsets must be a non-decreasing split of [0, R); otherwise do no work
        if (__syncthreads_or(bad)) {
            if (tid == 0) atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
            c = 0;
        }
        // both streams in one scan: heavy tiles in the low 32 bits, light in the
        // high 32 (the sums stay below 2^31, so the halves never carry)
        // (the fused sequence keeps every expert in one stream)
        const bool light = !FUSED && !WGRAD && c <= light_tiles<PAIR>();
        const uint64_t cs = light ? (uint64_t)c << 32 : (uint64_t)c;
        uint64_t incl = cs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) ctl->scan[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint64_t ws = lane < kThreads / 32 ? ctl->scan[lane] : 0ull;
            uint64_t wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint64_t v = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += v;
            }
            if (lane < kThreads / 32) ctl->scan[lane] = wi - ws;
            if (lane == kThreads / 32 - 1) ctl->scan[kThreads / 32] = wi;
        }
        __syncthreads();
        if (e < E) {
            const uint64_t ex = ctl->scan[warp] + incl - cs;
            ctl->tile_base[0][e] = (int32_t)(uint32_t)ex;
            ctl->tile_base[1][e] = (int32_t)(ex >> 32);
        }
        if (e == 0) {
            const uint64_t tot = ctl->scan[kThreads / 32];
            ctl->tile_base[0][E] = (int32_t)(uint32_t)tot;
            ctl->tile_base[1][E] = (int32_t)(tot >> 32);
            if (FUSED) ctl->tag = (__ldcg(args.err + kWordEpoch) & 0xffffffu) << kDepCountBits;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // peer barriers initialised, TMEM allocated
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const int NB = args.NB;
    if constexpr (FUSED) {
        // The round schedule. Down round k may run once the gate/up round holding
        // the last unit of its last expert lies more than `gap` rounds back;
        // among ready rounds, down rounds keep to their share of the rounds so
        // far, at most ceil(down rounds / gate/up rounds) in a row, so that each
        // CTA alternates long gate/up main loops with epilogue-bound down units.
        const int G = (int)gridDim.x;
        const int nt = ctl->tile_base[0][E];
        const int ngr = (nt * NB + G - 1) / G, ndr = (nt * args.NB2 + G - 1) / G;
        const bool fits = ngr + ndr <= kMaxRounds;
        if (fits) {
            for (int k = tid; k < ndr; k += kThreads) {
                const int j = min(nt * args.NB2, (k + 1) * G) - 1;
                int lo = 0, hi = E - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (ctl->tile_base[0][mid] * args.NB2 <= j) lo = mid; else hi = mid - 1;
                }
                ctl->need[k] = (int16_t)((ctl->tile_base[0][lo + 1] * NB - 1) / G);
            }
        }
        __syncthreads();
        if (tid == 0) {
            if (!fits) atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
            const int nr = fits ? ngr + ndr : 0;
            const int gap = args.gap_rounds;
            const int maxrun = (ndr + max(ngr, 1) - 1) / max(ngr, 1);
            int gi = 0, di = 0, run = 0;
            for (int r = 0; r < nr; ++r) {
                bool take_d = false;
                if (di < ndr) {
                    if (gi == ngr) {
                        take_d = true;
                    } else {
                        const int gr = ctl->need[di];
                        const bool ready = gr < gi && r - ctl->gpos[gr] > gap;
                        take_d = ready && (int64_t)di * ngr <= (int64_t)gi * ndr && run < maxrun;
                    }
                }
                if (take_d) {
                    ctl->sched[r] = (1 << 30) | di++;
                    ++run;
                } else {
                    ctl->gpos[gi] = (int16_t)r;
                    ctl->sched[r] = gi++;
                    run = 0;
                }
            }
            ctl->nrounds = nr;
        }
        __syncthreads();
    }
    const int total_units =
        FUSED   ? ctl->nrounds * (int)gridDim.x
        : WGRAD ? E * (PAIR ? args.MT / 2 : args.MT) * NB
                : (ctl->tile_base[0][E] + ctl->tile_base[1][E]) * NB;
    const int per_tile = PAIR ? 2 : 1;
    // k-blocks of a unit: d / 64 for gate/up, n / 64 for down (weight gradients:
    // the expert's rows / 64, rounded up)
    const int KB = args.Kdim / BK;
    const int KB2 = FUSED ? args.Kdim2 / BK : KB;
    auto unit_at = [&](int u) -> Unit {
        if constexpr (FUSED) {
            Unit x = decode_sched(u, NB, args.NB2, E, ctl->sched, ctl->tile_base[0], ctl->offsets);
            x.kbs = x.down ? KB2 : KB;
            return x;
        } else if constexpr (WGRAD) {
            // expert-major, then 128-row output tile (a pair of them on CTA pairs,
            // CTA `rank` taking the pair's tile 2*mt + rank), then output column block
            Unit x;
            x.valid = true;
            x.down = false;
            x.tile = -1;
            const int per_e = (PAIR ? args.MT / 2 : args.MT) * NB;
            x.e = u / per_e;
            const int rem = u - x.e * per_e;
            const int mt = rem / NB;
            x.nb = rem - mt * NB;
            x.row0 = (PAIR ? 2 * mt + (int)rank : mt) * BM;
            x.rows = BM;
            x.kbs = ctl->tile_base[0][x.e + 1] - ctl->tile_base[0][x.e];
            x.poff = BK * ctl->tile_base[0][x.e];
            x.off = ctl->offsets[x.e];
            return x;
        } else {
            Unit x;
            x.valid = true;
            x.down = MODE == kDown;
            x.tile = -1;
            x.kbs = KB;
            decode_unit(u, NB, E, ctl->tile_base, ctl->offsets, per_tile, rank, x.e, x.nb, x.row0,
                        x.rows);
            return x;
        }
    };
    // fused: arrivals that complete a row tile's H (epilogue warps x column blocks)
    const uint32_t dep_full = (uint32_t)(NB * EW);

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer --
        uint32_t it = 0;
        bool ok = true;
        for (int u = first_unit; u < total_units && ok; u += unit_stride) {
            const Unit un = unit_at(u);
            if (!un.valid) continue;
            const int e = un.e, nb = un.nb, row0 = un.row0;
            // fused down unit: its A is the H tile, loaded once every gate/up
            // unit of the row tile has completed its stores
            const bool fdown = FUSED && un.down;
            if (fdown) {
                if (!dep_wait(args.dep + un.tile, ctl->tag | dep_full, args.err)) {
                    ok = false;
                    break;
                }
                ptx::fence_proxy_async_global();
            }
            const int wrow = e * (fdown ? args.Kdim2 : args.Kdim);
            const int kbs = un.kbs;
            for (int kb = 0; kb < kbs; ++kb, ++it) {
                const uint32_t s = it % S, ph = (it / S) & 1u;
                if (!bounded_wait<PAIR>(ptx::smem_addr(&ctl->empty[s]), ph ^ 1u, args.err)) {
                    ok = false;
                    break;
                }
                const uint32_t full = ptx::smem_addr(&ctl->full[s]);
                const uint32_t sA = smem_base + s * G::kStageBytes, sB = sA + kABytes;
                const int ky = wrow + kb * BK;
                // TMA bytes per CTA and stage: B always, A only when not gathered
                constexpr uint32_t kTx = G::kStageBytes - (GATHER ? kABytes : 0);
                if constexpr (PAIR) {
                    // both CTAs' loads complete on the even CTA's barrier
                    if (leader) ptx::mbar_arrive_expect_tx(full, 2 * kTx);
                    const uint32_t fullc = ptx::mapa(full, 0);
                    if constexpr (WGRAD) {
                        // A (MN-major): this CTA's 128 output rows, two 64-column slabs;
                        // B: its half of the 256 output columns (dW1|dW3: dA1 on the even
                        // CTA, dA3 on the odd; dW2: 128 of the w dY columns)
                        const int ya = (MODE == kDW13 ? un.poff : un.off) + kb * BK;
                        const int yb = (MODE == kDW13 ? un.off : un.poff) + kb * BK;
                        ptx::tma_load_2d_pair(sA, &tmA, fullc, row0, ya);
                        ptx::tma_load_2d_pair(sA + kBBox, &tmA, fullc, row0 + 64, ya);
                        const CUtensorMap *mb =
                            MODE == kDW13 ? (leader ? &tmB0 : &tmB1) : &tmB0;
                        const int x0 = MODE == kDW13 ? nb * 128 : nb * BN + (int)rank * 128;
                        ptx::tma_load_2d_pair(sB, mb, fullc, x0, yb);
                        ptx::tma_load_2d_pair(sB + kBBox, mb, fullc, x0 + 64, yb);
                        continue;
                    }
                    if constexpr (MODE == kDX) {
                        // A: this CTA's 128 rows of dA1 (first n/64 k-blocks) or dA3;
                        // B: its 128 of the tile's 256 output columns, W1[e] or W3[e]
                        // rows (K-major), two 64-row boxes
                        const bool second = kb >= args.kb_half;
                        const int kx = (second ? kb - args.kb_half : kb) * BK;
                        ptx::tma_load_2d_pair(sA, second ? &tmB2 : &tmA, fullc, kx, row0);
                        const int brow = e * args.bn_rows + nb * BN + (int)rank * 128;
                        const CUtensorMap *mb = second ? &tmB1 : &tmB0;
                        ptx::tma_load_2d_pair(sB, mb, fullc, kx, brow);
                        ptx::tma_load_2d_pair(sB + kBBox, mb, fullc, kx, brow + 64);
                        continue;
                    }
                    ptx::tma_load_2d_pair(sA, &tmA, fullc, kb * BK, row0);
                    if constexpr (MODE == kDH) {
                        // its 128 of the tile's 256 hidden columns: W2[e] rows (K-major,
                        // d contiguous), two 64-row boxes
                        const int brow = e * args.bn_rows + nb * BN + (int)rank * 128;
                        ptx::tma_load_2d_pair(sB, &tmB0, fullc, kb * BK, brow);
                        ptx::tma_load_2d_pair(sB + kBBox, &tmB0, fullc, kb * BK, brow + 64);
                    } else if (GATE) {
                        // even CTA: gate columns (W1), odd CTA: up columns (W3)
                        const CUtensorMap *mb = leader ? &tmB0 : &tmB1;
                        ptx::tma_load_2d_pair(sB, mb, fullc, nb * 128, ky);
                        ptx::tma_load_2d_pair(sB + kBBox, mb, fullc, nb * 128 + 64, ky);
                    } else {
                        const int x0 = nb * BN + (int)rank * 128;
                        ptx::tma_load_2d_pair(sB, &tmB0, fullc, x0, ky);
                        ptx::tma_load_2d_pair(sB + kBBox, &tmB0, fullc, x0 + 64, ky);
                    }
                } else if (fdown) {
                    ptx::mbar_arrive_expect_tx(full, G::kStageBytes);
                    ptx::tma_load_2d(sA, &tmA, full, kb * BK, row0);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        ptx::tma_load_2d(sB + q * kBBox, &tmB2, full, nb * BN + q * 64, ky);
                } else if constexpr (WGRAD) {
                    // A: two 64-column slabs of the 128 output rows, k-rows = the
                    // expert's rows kb*64 .. +63; B: four 64-column boxes of the same
                    // k-rows. The padded operand's rows start at poff, the other's at off.
                    ptx::mbar_arrive_expect_tx(full, kTx);
                    const int ya = (MODE == kDW13 ? un.poff : un.off) + kb * BK;
                    const int yb = (MODE == kDW13 ? un.off : un.poff) + kb * BK;
                    ptx::tma_load_2d(sA, &tmA, full, un.row0, ya);
                    ptx::tma_load_2d(sA + kBBox, &tmA, full, un.row0 + 64, ya);
                    if constexpr (MODE == kDW13) {
                        ptx::tma_load_2d(sB + 0 * kBBox, &tmB0, full, nb * 128, yb);
                        ptx::tma_load_2d(sB + 1 * kBBox, &tmB0, full, nb * 128 + 64, yb);
                        ptx::tma_load_2d(sB + 2 * kBBox, &tmB1, full, nb * 128, yb);
                        ptx::tma_load_2d(sB + 3 * kBBox, &tmB1, full, nb * 128 + 64, yb);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::tma_load_2d(sB + q * kBBox, &tmB0, full, nb * BN + q * 64, yb);
                    }
                } else if constexpr (MODE == kDX) {
                    // k-blocks 0 .. n/64-1: dA1 rows against W1[e]; then dA3 against W3[e].
                    // W rows e*d + nb*256 .. +255 (d), columns kx .. kx+63 (n): K-major
                    ptx::mbar_arrive_expect_tx(full, kTx);
                    const bool second = kb >= args.kb_half;
                    const int kx = (second ? kb - args.kb_half : kb) * BK;
                    ptx::tma_load_2d(sA, second ? &tmB2 : &tmA, full, kx, row0);
                    const int brow = e * args.bn_rows + nb * BN;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        ptx::tma_load_2d(sB + q * kBBox, second ? &tmB1 : &tmB0, full, kx, brow + q * 64);
                } else {
                    ptx::mbar_arrive_expect_tx(full, kTx);
                    if (!GATHER) ptx::tma_load_2d(sA, &tmA, full, kb * BK, row0);
                    if constexpr (MODE == kDH) {
                        // W2[e] rows nb*256 .. +255 (n), columns kb*64 .. +63 (d):
                        // four 64-row boxes stacked into one K-major 256-row tile
                        const int brow = e * args.bn_rows + nb * BN;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::tma_load_2d(sB + q * kBBox, &tmB0, full, kb * BK, brow + q * 64);
                    } else if (MODE != kDown) {
                        ptx::tma_load_2d(sB + 0 * kBBox, &tmB0, full, nb * 128, ky);
                        ptx::tma_load_2d(sB + 1 * kBBox, &tmB0, full, nb * 128 + 64, ky);
                        ptx::tma_load_2d(sB + 2 * kBBox, &tmB1, full, nb * 128, ky);
                        ptx::tma_load_2d(sB + 3 * kBBox, &tmB1, full, nb * 128 + 64, ky);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ptx::tma_load_2d(sB + q * kBBox, &tmB0, full, nb * BN + q * 64, ky);
                    }
                }
            }
        }
        if (!ok && (!PAIR || leader)) {
            // drain the loads that may still be landing in shared memory
            const uint32_t first = it > (uint32_t)S ? it - S : 0u;
            for (uint32_t j = first; j < it; ++j)
                bounded_wait<PAIR>(ptx::smem_addr(&ctl->full[j % S]), (j / S) & 1u, args.err);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer --
        uint32_t it = 0, uc = 0;
        bool ok = true;
        for (int u = first_unit; u < total_units && ok; u += unit_stride) {
            const Unit un = unit_at(u);
            if (!un.valid) continue;
            const uint32_t a = uc & 1u, aph = (uc >> 1) & 1u;
            ++uc;
            if (!bounded_wait<PAIR>(ptx::smem_addr(&ctl->tempty[a]), aph ^ 1u, args.err)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + a * BN;
            const int kbs = un.kbs;
            for (int kb = 0; kb < kbs; ++kb, ++it) {
                const uint32_t s = it % S, ph = (it / S) & 1u;
                if (!bounded_wait<PAIR>(ptx::smem_addr(&ctl->full[s]), ph, args.err)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sA = smem_base + s * G::kStageBytes, sB = sA + kABytes;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    // A K-major: the next 16 k-columns are 32 bytes on; MN-major (weight
                    // gradients): the next 16 k-rows are 2048 bytes on, slabs 8 KB apart
                    const uint64_t adesc = WGRAD ? ptx::desc_sw128(sA + k * 2048, kBBox, 1024)
                                                 : ptx::desc_sw128(sA + k * 32, 16, 1024);
                    // B MN-major: the next 16 k-rows are 2048 bytes on; K-major (kDH):
                    // the next 16 k-columns are 32 bytes on within each row
                    const uint64_t bdesc = (MODE == kDH || MODE == kDX)
                                               ? ptx::desc_sw128(sB + k * 32, 16, 1024)
                                               : ptx::desc_sw128(sB + k * 2048, kBBox, 1024);
                    constexpr uint32_t kId = idesc_of<MODE, PAIR>();
                    if constexpr (PAIR)
                        ptx::tc_mma_f16_pair(d_tmem, adesc, bdesc, kId, (kb | k) != 0);
                    else
                        ptx::tc_mma_f16(d_tmem, adesc, bdesc, kId, (kb | k) != 0);
                }
                if constexpr (PAIR)
                    ptx::tc_commit_pair(ptx::smem_addr(&ctl->empty[s]), 0x3);
                else
                    ptx::tc_commit(ptx::smem_addr(&ctl->empty[s]));
            }
            if (!ok) break;
            if constexpr (PAIR)
                ptx::tc_commit_pair(ptx::smem_addr(&ctl->tfull[a]), 0x3);
            else
                ptx::tc_commit(ptx::smem_addr(&ctl->tfull[a]));
        }
        // every MMA this thread issued (and its barrier arrivals) has completed
        if constexpr (PAIR)
            ptx::tc_commit_pair(ptx::smem_addr(&ctl->drain), 0x1);
        else
            ptx::tc_commit(ptx::smem_addr(&ctl->drain));
        bounded_wait<PAIR>(ptx::smem_addr(&ctl->drain), 0, args.err);
    } else if (GATHER && (warp == 2 || warp == 3)) {
        // ------------------------------------------------- A-row gatherers --
        // Lane (rr, c) copies 16-byte chunk c of rows gw*4 + rr + 8i (i < 16) of
        // the stage's 128-row A tile, placed at the 128-byte-swizzle position
        // row*128 + ((c ^ (row & 7)) << 4) the MMA descriptor expects.
        const int gw = warp - 2;
        const int c = lane & 7, rr = lane >> 3;
        const uint32_t full0 = ptx::smem_addr(&ctl->full[0]);
        auto signal = [&](uint32_t j) {  // this warp's rows of stage j have landed
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full0 + (j % S) * (uint32_t)sizeof(uint64_t));
        };
        uint32_t it = 0;
        bool ok = true;
        // token indices of a unit's rows, loaded one unit ahead so that their
        // latency hides behind the current unit's copies (-2: past the rows)
        // (fused down units: no rows, and the warps only arrive for their stages)
        auto load_tok = [&](int uu, int (&raw)[16]) {
            const Unit un = unit_at(uu);
            const int rows = !un.valid || (FUSED && un.down) ? 0 : un.rows;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = gw * 4 + rr + 8 * i;
                raw[i] = r < rows ? __ldg(args.perm_token + un.row0 + r) : -2;
            }
        };
        int nxt[16];
#if MOE_GEMM_GATHER_HINT
        const uint64_t gpol = ptx::policy_evict_last();
#endif
        if (first_unit < total_units) load_tok(first_unit, nxt);
        for (int u = first_unit; u < total_units && ok; u += unit_stride) {
            const Unit cur = unit_at(u);
            const int kbs = !cur.valid ? 0 : cur.kbs;
            int tok[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int t = nxt[i];
                tok[i] = -1;
                if (t != -2) {
                    if (t >= 0 && t < args.T) tok[i] = t;
                    else atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
                }
            }
            if (u + unit_stride < total_units) load_tok(u + unit_stride, nxt);
            for (int kb = 0; kb < kbs; ++kb, ++it) {
                const uint32_t s = it % S, ph = (it / S) & 1u;
                if (!bounded_wait<PAIR>(ptx::smem_addr(&ctl->empty[s]), ph ^ 1u, args.err)) {
                    ok = false;
                    break;
                }
                const uint32_t sA = smem_base + s * G::kStageBytes;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = gw * 4 + rr + 8 * i;
                    if (tok[i] >= 0) {
#if MOE_GEMM_GATHER_HINT
                        ptx::cp_async_16_hint(sA + r * 128 + ((c ^ (r & 7)) << 4),
                                              args.X + (int64_t)tok[i] * args.Kdim + kb * BK + c * 8,
                                              gpol);
#else
                        ptx::cp_async_16(sA + r * 128 + ((c ^ (r & 7)) << 4),
                                         args.X + (int64_t)tok[i] * args.Kdim + kb * BK + c * 8);
#endif
                    }
                }
                ptx::cp_async_commit_group();
                if (it >= (uint32_t)kGatherLag) {
                    ptx::cp_async_wait_group<kGatherLag>();
                    ptx::fence_proxy_async_smem();
                    signal(it - kGatherLag);
                }
            }
        }
        // the last stages still in flight
        ptx::cp_async_wait_group<0>();
        ptx::fence_proxy_async_smem();
        for (uint32_t j = it >= (uint32_t)kGatherLag ? it - kGatherLag : 0u; j < it; ++j) signal(j);
    } else if (warp >= 4) {
        // -------------------------------------------------------- epilogue --
        // TMEM lanes 32q..32q+31 (= tile rows) belong to warps with warp % 4 == q;
        // with 8 or 12 epilogue warps the warps of a quadrant split the tile's
        // 32-column chunks (warp `half` of nhalf takes chunks half*C/nhalf ..)
        const int q = warp & 3, half = (warp - 4) >> 2, nhalf = EW / 4;
        const int r = q * 32 + lane;
        const uint32_t tempty0 = PAIR ? ptx::mapa(ptx::smem_addr(&ctl->tempty[0]), 0)
                                      : ptx::smem_addr(&ctl->tempty[0]);
        // this warp's output staging buffers
        const uint32_t epi_base =
            smem_base + (uint32_t)S * G::kStageBytes + (uint32_t)(warp - 4) * kNBuf * kEpiBuf;
        uint32_t epi_groups = 0;  // TMA store groups this warp has committed
        uint32_t uc = 0;
        for (int u = first_unit; u < total_units; u += unit_stride) {
            const Unit un = unit_at(u);
            if (!un.valid) continue;
            const int nb = un.nb, row0 = un.row0, rows = un.rows;
            const bool dn = MODE == kDown || MODE == kDX || (FUSED && un.down);
            const CUtensorMap *omap = FUSED && un.down ? &tmOut2 : &tmOut;
            const uint32_t a = uc & 1u, aph = (uc >> 1) & 1u;
            ++uc;
            const bool valid = r < rows;
            const int64_t p = (int64_t)row0 + r;
            // kDH: the row's stored pre-activations, one 32-column chunk ahead of
            // their use; the first chunk's loads go out before the accumulator wait
            const int c_lo = half * (BN / 32) / nhalf, c_hi = (half + 1) * (BN / 32) / nhalf;
            float4 x1[8], x3[8];
            auto load_pre = [&](int c, float4 (&l1)[8], float4 (&l3)[8]) {
                const int64_t off = p * args.out_ld + nb * BN + c * 32;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    l1[i] = valid ? __ldg(reinterpret_cast<const float4 *>(args.pre1 + off) + i)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                    l3[i] = valid ? __ldg(reinterpret_cast<const float4 *>(args.pre3 + off) + i)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            };
            if constexpr (MODE == kDH) load_pre(c_lo, x1, x3);
            if (!bounded_wait<PAIR>(ptx::smem_addr(&ctl->tfull[a]), aph, args.err)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * BN;
            // A warp whose 32 rows all belong to the tile writes each 32-column
            // chunk through shared memory and a TMA store (whole 64-byte row
            // segments); otherwise each valid row is stored directly.
            const bool whole = q * 32 + 31 < rows;
            // 32 rows x 64 bytes (each lane's 16 words) through a staging buffer
            // (64-byte swizzle) and one TMA store at (x, y)
            auto store_box = [&](const uint32_t (&packed)[16], int x, int y,
                                 const CUtensorMap *map) {
                // buffers rotate with the store groups, so the group that last
                // read this buffer is the kNBuf-th most recent one
                const uint32_t buf = epi_base + (epi_groups % kNBuf) * kEpiBuf;
                if (lane == 0 && epi_groups >= (uint32_t)kNBuf)
                    ptx::bulk_wait_group_read<kNBuf - 1>();
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    ptx::st_shared_v4(buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4),
                                      packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                      packed[4 * i + 3]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (args.out_evict_first)
                        ptx::tma_store_2d_hint(map, buf, x, y, ptx::policy_evict_first());
                    else
                        ptx::tma_store_2d(map, buf, x, y);
                    ptx::bulk_commit_group();
                }
                ++epi_groups;
            };
            auto emit = [&](const uint32_t (&packed)[16], __nv_bfloat16 *dst, int col,
                            const CUtensorMap *map) {
                if (whole) {
                    store_box(packed, col, row0 + q * 32, map);
                } else if (valid) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                           packed[4 * i + 3]);
                }
            };
            if constexpr (WGRAD) {
                // output rows row0 + 32q .. +31 of expert e (fp32 [E * wout_rows,
                // wout_ld]; kDW13: dW1 by tmOut, dW3 by tmOut2): each 32-column chunk
                // as two 16-column TMA boxes. An expert with no rows ran no MMA, so
                // its gradient is written as zeros.
                const int oy = un.e * args.wout_rows + un.row0 + q * 32;
#pragma unroll 1
                for (int c = half * (BN / 32) / nhalf; c < (half + 1) * (BN / 32) / nhalf; ++c) {
                    uint32_t v[32], lo[16], hi[16];
                    if (un.kbs > 0) {
                        ptx::tmem_ld32(taddr + c * 32, v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0u;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        lo[i] = v[i];
                        hi[i] = v[16 + i];
                    }
                    const CUtensorMap *map = MODE == kDW13 && c >= 4 ? &tmOut2 : &tmOut;
                    const int x0 = MODE == kDW13 ? nb * 128 + (c & 3) * 32 : nb * BN + c * 32;
                    store_box(lo, x0, oy, map);
                    store_box(hi, x0 + 16, oy, map);
                }
            } else if constexpr (MODE == kDH) {
                // g = dY[t_p] W2[e]^T for 256 columns j of the expert's hidden
                // layer; with the stored pre-activations a1, a3 of row p:
                //   dA1 = w g a3 s (1 + a1 (1 - s)), dA3 = w g SiLU(a1), s = sigmoid(a1)
                // and the routing weight's gradient gets sum_j g SiLU(a1) a3, summed
                // here per 32-column chunk (ascending j) into dS partials
                float w = 0.f;
                if (valid) {
                    const int slot = args.perm_slot != nullptr ? __ldg(args.perm_slot + p) : (int)p;
                    if (slot >= 0 && slot < args.R) w = __ldg(args.topk_w + slot);
                    else atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
                }
                const int64_t rowoff = p * args.out_ld + nb * BN;
#pragma unroll 1
                for (int c = c_lo; c < c_hi; ++c) {
                    float4 n1[8], n3[8];
                    if (c + 1 < c_hi) load_pre(c + 1, n1, n3);
                    uint32_t gv[32];
                    ptx::tmem_ld32(taddr + c * 32, gv);
                    float part = 0.f;
                    uint32_t pa[16], pb[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float r1[2], r3[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const float a1 = (&x1[i >> 1].x)[2 * (i & 1) + hh];
                            const float a3 = (&x3[i >> 1].x)[2 * (i & 1) + hh];
                            const float g = __uint_as_float(gv[2 * i + hh]);
                            const float sg = __fdividef(1.0f, 1.0f + __expf(-a1));
                            const float silu = a1 * sg;
                            part += g * (silu * a3);
                            r1[hh] = w * g * a3 * sg * (1.0f + a1 * (1.0f - sg));
                            r3[hh] = w * g * silu;
                        }
                        pa[i] = pack_bf16x2(r1[0], r1[1]);
                        pb[i] = pack_bf16x2(r3[0], r3[1]);
                    }
                    emit(pa, args.out + rowoff + c * 32, nb * BN + c * 32, &tmOut);
                    emit(pb, args.out3 + rowoff + c * 32, nb * BN + c * 32, &tmOut2);
                    if (valid) args.dspart[p * args.ds_ld + nb * (BN / 32) + c] = part;
                    if (c + 1 < c_hi) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            x1[i] = n1[i];
                            x3[i] = n3[i];
                        }
                    }
                }
            } else if (!dn) {
                __nv_bfloat16 *dst = args.out + p * args.out_ld + nb * 128;
#pragma unroll 1
                for (int c = half * 4 / nhalf; c < (half + 1) * 4 / nhalf; ++c) {
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
                    emit(packed, dst + c * 32, nb * 128 + c * 32, omap);
                    if constexpr (MODE == kGateUpPre) {
                        // the pre-activations as they are (fp32): A1 (gate), A3 (up).
                        // Whole 32-row warps: four 16-column TMA boxes through the
                        // staging buffers (maps in tmB2, tmOut2); else each valid lane
                        // writes its row's 128 bytes of the chunk
                        if (whole) {
                            uint32_t lo[16], hi[16];
                            const int x0 = nb * 128 + c * 32, y0 = row0 + q * 32;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                lo[i] = g[i];
                                hi[i] = g[16 + i];
                            }
                            store_box(lo, x0, y0, &tmB2);
                            store_box(hi, x0 + 16, y0, &tmB2);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                lo[i] = v[i];
                                hi[i] = v[16 + i];
                            }
                            store_box(lo, x0, y0, &tmOut2);
                            store_box(hi, x0 + 16, y0, &tmOut2);
                        } else if (valid) {
                            const int64_t off = p * args.out_ld + nb * 128 + c * 32;
                            float4 *d1 = reinterpret_cast<float4 *>(args.pre_out1 + off);
                            float4 *d3 = reinterpret_cast<float4 *>(args.pre_out3 + off);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                d1[i] = make_float4(__uint_as_float(g[4 * i]), __uint_as_float(g[4 * i + 1]),
                                                    __uint_as_float(g[4 * i + 2]), __uint_as_float(g[4 * i + 3]));
                                d3[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                            }
                        }
                    }
                }
            } else if (MODE == kDX && args.f32_out) {
                // fp32 outputs (the router's share dL Wr^T): 16-column TMA boxes for
                // whole 32-row warps, else direct stores of the valid rows
                float *dst = args.outf + p * args.out_ld + nb * BN;
#pragma unroll 1
                for (int c = half * (BN / 32) / nhalf; c < (half + 1) * (BN / 32) / nhalf; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(taddr + c * 32, v);
                    if (whole) {
                        uint32_t lo[16], hi[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            lo[i] = v[i];
                            hi[i] = v[16 + i];
                        }
                        store_box(lo, nb * BN + c * 32, row0 + q * 32, omap);
                        store_box(hi, nb * BN + c * 32 + 16, row0 + q * 32, omap);
                    } else if (valid) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                    }
                }
            } else {
                float w = 0.f;
                if (MODE == kDX) {
                    w = 1.f;  // dXg carries no routing weight (dA1, dA3 already do)
                } else if (valid) {
                    const int slot = args.perm_slot != nullptr ? __ldg(args.perm_slot + p) : (int)p;
                    if (slot >= 0 && slot < args.R) w = __ldg(args.topk_w + slot);
                    else atomicOr(args.err, MOE_DEVERR_BAD_EXPERT);
                }
                __nv_bfloat16 *dst = FUSED ? args.out2 + p * args.out2_ld + nb * BN
                                           : args.out + p * args.out_ld + nb * BN;
#pragma unroll 1
                for (int c = half * (BN / 32) / nhalf; c < (half + 1) * (BN / 32) / nhalf; ++c) {
                    uint32_t v[32];
                    ptx::tmem_ld32(taddr + c * 32, v);
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        packed[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]),
                                                w * __uint_as_float(v[2 * i + 1]));
                    emit(packed, dst + c * 32, nb * BN + c * 32, omap);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // the accumulator stage is free again (the even CTA's MMA waits on it)
                const uint32_t bar = tempty0 + a * (uint32_t)sizeof(uint64_t);
                if constexpr (PAIR) ptx::mbar_arrive_cluster(bar);
                else ptx::mbar_arrive(bar);
            }
            if (FUSED && !dn) {
                // this warp's share of the H tile is written: direct stores are
                // fenced by each lane, TMA stores waited for to completion
                __threadfence();
                __syncwarp();
                if (lane == 0) {
                    ptx::bulk_wait_group<0>();
                    ptx::fence_proxy_async_global();
                    __threadfence();
                    dep_arrive(args.dep + un.tile, ctl->tag);
                }
                __syncwarp();
            }
        }
        // this warp's TMA stores have completed before the CTA exits
        if (lane == 0) ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    // ---- teardown -----------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // no remote arrival can still target us
    ptx::tc_fence_after();
    if (warp == 2) {
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
        else ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
    if (FUSED && tid == 0) {
        // the last CTA to finish advances the epoch for the next launch
        __threadfence();
        const uint32_t ticket = atomicAdd(args.err + kWordTicket, 1u);
        if (ticket == gridDim.x - 1) {
            atomicExch(args.err + kWordTicket, 0u);
            atomicAdd(args.err + kWordEpoch, 1u);
        }
    }
}

// Failure-detection self-test: one thread waits, through the pipeline's own
// bounded wait, on a shared-memory barrier that nothing arrives at. After the
// time limit the wait gives up, sets MOE_DEVERR_TIMEOUT and the kernel returns.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = ptx::smem_addr(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_barrier_init();
    bounded_wait<false>(b, 0, err);  // phase 0 never completes
}

// ------------------------------------------------------------ host side --

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    // looked up once (a function-local static is initialised thread-safely)
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box box_cols x box_rows,
// 128-byte swizzle unless given, zero fill outside the tensor.
bool make_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, cols] row-major (the weight gradients' TMA stores)
bool make_map_f32(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                  uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// b2 and out2 are read by the fused kernel only (the others get copies of b0, out)
template <int MODE, bool PAIR, int EW>
cudaError_t launch_ew(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                      const CUtensorMap &out, const CUtensorMap &b2, const CUtensorMap &out2,
                      const GemmArgs &args, int max_units, cudaStream_t s) {
    constexpr size_t kSmem = smem_bytes<PAIR, EW>();
    constexpr int kThreads = threads_of<EW>();
    {
        const cudaError_t e = ensure_dynamic_smem(
            reinterpret_cast<const void *>(grouped_gemm_kernel<MODE, PAIR, EW>), (int)kSmem);
        if (e != cudaSuccess) return e;
    }
    if constexpr (!PAIR) {
        const int grid = max(1, min(sm_count(), max_units));
        return launch_k(grouped_gemm_kernel<MODE, false, EW>, dim3(grid), dim3(kThreads), kSmem, s,
                        a, b0, b1, out, b2, out2, args);
    } else {
        // one cluster of 2 CTAs (an SM pair) per unit slot
        const int pairs = max(1, min(sm_count() / 2, max_units));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl_enabled() ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE, true, EW>, a, b0, b1, out, b2,
                                  out2, args);
    }
}

// Eight epilogue warps when a tile's main loop is at most 8 k-blocks (the
// epilogue then dominates: measured on the SonicMoE-shaped down GEMM, n = 256,
// 0.082 -> 0.072 ms), twelve for the single-CTA down GEMM there (0.0764 ->
// 0.0708 ms; the backward's dX GEMM measured no faster with them); four
// otherwise (with longer main loops the extra warps cost slightly: DeepSeek-V3-
// shaped GEMMs about 1% slower).
template <int MODE, bool PAIR>
cudaError_t launch_variant(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                           const CUtensorMap &out, const GemmArgs &args, int max_units,
                           cudaStream_t s) {
    if constexpr (MODE == kDown && !PAIR) {
        if (args.Kdim / BK <= 8)
            return launch_ew<MODE, PAIR, 12>(a, b0, b1, out, b0, out, args, max_units, s);
    }
    if (args.Kdim / BK <= 8)
        return launch_ew<MODE, PAIR, 8>(a, b0, b1, out, b0, out, args, max_units, s);
    return launch_ew<MODE, PAIR, 4>(a, b0, b1, out, b0, out, args, max_units, s);
}

// CTA pairs halve the B bytes each SM receives per MMA and so allow a deeper
// ring; they pay off when experts have many 128-row tiles (an expert with an odd
// tile count wastes half of one pair, and few-tile experts are HBM-bound anyway):
// measured faster at 8 tiles per expert on average, slower at 2 and 4.
// MOE_GEMM_CTA_PAIR=0/1 forces a choice (tests run both kernels this way).
bool use_pair(int R, int E) {
    const char *env = getenv("MOE_GEMM_CTA_PAIR");
    if (env != nullptr && (env[0] == '0' || env[0] == '1')) return env[0] == '1';
    return (int64_t)R >= (int64_t)8 * BM * E;
}

template <int MODE>
cudaError_t launch_gemm(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                        const CUtensorMap &out, const GemmArgs &args, cudaStream_t s) {
    // (gate/up chooses its variant itself: the A source differs)
    const int tiles = args.R / BM + args.E;  // upper bound of the 128-row tiles
    if (use_pair(args.R, args.E))
        return launch_variant<MODE, true>(a, b0, b1, out, args, (tiles / 2 + args.E) * args.NB, s);
    return launch_variant<MODE, false>(a, b0, b1, out, args, tiles * args.NB, s);
}

}  // namespace

cudaError_t launch_gemm_gate_up(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                                const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                                const int32_t *offsets, int R, int d, int E, int n,
                                __nv_bfloat16 *H, __nv_bfloat16 *xg, uint32_t *err,
                                cudaStream_t s) {
    CUtensorMap ta, tb0, tb1, th;
    if (!make_map(&tb0, W1, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&tb1, W3, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&th, H, n, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.X = X;
    args.perm_token = perm_token;
    args.T = T;
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = d;
    args.NB = n / 128;
    args.out = H;
    args.out_ld = n;
    args.err = err;
    const int tiles = R / BM + E;  // upper bound of the 128-row tiles
    if (use_pair(R, E)) {
        // CTA pairs load A by TMA from rows gathered into xg beforehand
        // the grouped rows in use end at offsets[E]
        cudaError_t e = launch_gather_rows(X, perm_token, T, R, offsets + E, d, xg, err, s);
        if (e != cudaSuccess) return e;
        if (!make_map(&ta, xg, d, R, 64, BM)) return cudaErrorInvalidValue;
        return launch_variant<kGateUp, true>(ta, tb0, tb1, th, args, (tiles / 2 + E) * args.NB, s);
    }
    // single CTAs gather their A rows themselves; the A map argument is not read
    return launch_variant<kGateUp, false>(tb0, tb0, tb1, th, args, tiles * args.NB, s);
}

namespace {
// Epilogue warps as launch_variant chooses them, with the extra maps b2/out2.
template <int MODE, bool PAIR>
cudaError_t launch_ew_auto(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                           const CUtensorMap &out, const CUtensorMap &b2, const CUtensorMap &out2,
                           const GemmArgs &args, int max_units, cudaStream_t s) {
    if (args.Kdim / BK <= 8)
        return launch_ew<MODE, PAIR, 8>(a, b0, b1, out, b2, out2, args, max_units, s);
    return launch_ew<MODE, PAIR, 4>(a, b0, b1, out, b2, out2, args, max_units, s);
}

// dS[p] = sum of the row's partials (rows in use) in a fixed order: g lanes per
// row (a power of two, from the row length), lane i of the group adding
// partials i, i + g, ... ascending, then a butterfly of fixed shape over the
// group. Reads are coalesced along the row.
__global__ void __launch_bounds__(256)
ds_reduce_kernel(const float *__restrict__ part, int ld, int R, const int32_t *__restrict__ rows_used,
                 int g, float *__restrict__ dS) {
    pdl_wait();
    pdl_trigger();
    const int64_t p = ((int64_t)blockIdx.x * 256 + threadIdx.x) / g;
    const int sub = threadIdx.x & (g - 1);
    const bool valid = p < R && p < __ldg(rows_used);
    float acc = 0.f;
    if (valid) {
        const float *row = part + p * ld;
        for (int i = sub; i < ld; i += g) acc = __fadd_rn(acc, __ldg(row + i));
    }
    for (int o = g >> 1; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    if (valid && sub == 0) dS[p] = acc;
}
}  // namespace

cudaError_t launch_gemm_gate_up_train(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                                      const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                                      const int32_t *offsets, int R, int d, int E, int n,
                                      __nv_bfloat16 *H, float *A1, float *A3,
                                      __nv_bfloat16 *xg, uint32_t *err, cudaStream_t s) {
    // (A1, A3: fp32 boxes of 16 columns x 32 rows, one epilogue warp's rows)
    CUtensorMap ta, tb0, tb1, th, tp1, tp3;
    if (!make_map(&tb0, W1, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&tb1, W3, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&th, H, n, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_f32(&tp1, A1, n, R, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_f32(&tp3, A3, n, R, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.X = X;
    args.perm_token = perm_token;
    args.T = T;
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = d;
    args.NB = n / 128;
    args.out = H;
    args.out_ld = n;
    args.pre_out1 = A1;
    args.pre_out3 = A3;
    args.err = err;
    const int tiles = R / BM + E;  // upper bound of the 128-row tiles
    if (use_pair(R, E)) {
        cudaError_t e = launch_gather_rows(X, perm_token, T, R, offsets + E, d, xg, err, s);
        if (e != cudaSuccess) return e;
        if (!make_map(&ta, xg, d, R, 64, BM)) return cudaErrorInvalidValue;
        return launch_ew_auto<kGateUpPre, true>(ta, tb0, tb1, th, tp1, tp3, args,
                                                (tiles / 2 + E) * args.NB, s);
    }
    return launch_ew_auto<kGateUpPre, false>(tb0, tb0, tb1, th, tp1, tp3, args, tiles * args.NB, s);
}

cudaError_t launch_backward_dh(const __nv_bfloat16 *dY, const int32_t *perm_token, int T,
                               const __nv_bfloat16 *W2, const float *A1,
                               const float *A3, const float *topk_w,
                               const int32_t *perm_slot, const int32_t *offsets, int R, int d,
                               int E, int n, __nv_bfloat16 *dA1, __nv_bfloat16 *dA3,
                               __nv_bfloat16 *xg, float *dspart, float *dS, uint32_t *err,
                               cudaStream_t s) {
    CUtensorMap ta, tb, t1, t3;
    // W2 as [E*n rows, d columns]: 64 x 64 boxes, K-major (d contiguous)
    if (!make_map(&tb, W2, d, (uint64_t)E * n, 64, 64) ||
        !make_map(&t1, dA1, n, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&t3, dA3, n, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.X = dY;
    args.perm_token = perm_token;
    args.T = T;
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = d;
    args.NB = n / BN;
    args.out = dA1;
    args.out_ld = n;
    args.out3 = dA3;
    args.topk_w = topk_w;
    args.perm_slot = perm_slot;
    args.err = err;
    args.pre1 = A1;
    args.pre3 = A3;
    args.bn_rows = n;
    args.dspart = dspart;
    args.ds_ld = n / 32;
    const int tiles = R / BM + E;
    cudaError_t e;
    if (use_pair(R, E)) {
        // CTA pairs, where the forward uses them: dY rows gathered into xg first
        // (the grouped rows in use end at offsets[E]), then loaded by TMA
        e = launch_gather_rows(dY, perm_token, T, R, offsets + E, d, xg, err, s);
        if (e != cudaSuccess) return e;
        if (!make_map(&ta, xg, d, R, 64, BM)) return cudaErrorInvalidValue;
        e = launch_ew_auto<kDH, true>(ta, tb, tb, t1, tb, t3, args, (tiles / 2 + E) * args.NB, s);
    } else {
        // single CTAs gather their dY rows themselves
        e = launch_ew_auto<kDH, false>(tb, tb, tb, t1, tb, t3, args, tiles * args.NB, s);
    }
    if (e != cudaSuccess) return e;
    // lanes per row: about 8 partials each, 1 .. 32
    const int ld = n / 32;
    int g = 1;
    while (g < 32 && g * 8 < ld) g *= 2;
    return launch_k(ds_reduce_kernel, dim3((unsigned)(((int64_t)R * g + 255) / 256)), dim3(256), 0,
                    s, static_cast<const float *>(dspart), ld, R, offsets + E, g, dS);
}

cudaError_t launch_backward_dx(const __nv_bfloat16 *dA1, const __nv_bfloat16 *dA3,
                               const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                               const int32_t *offsets, const int32_t *row_of_slot, int T, int K,
                               int R, int d, int E, int n, __nv_bfloat16 *dXg,
                               __nv_bfloat16 *dX, uint32_t *err, cudaStream_t s) {
    CUtensorMap ta1, ta3, tw1, tw3, tout;
    // A: rows of dA1 / dA3 [R, n], boxes of 64 columns x 128 rows; B: W1 / W3
    // as [E*d rows, n columns], 64 x 64 boxes (n contiguous: K-major)
    if (!make_map(&ta1, dA1, n, R, 64, BM) || !make_map(&ta3, dA3, n, R, 64, BM) ||
        !make_map(&tw1, W1, n, (uint64_t)E * d, 64, 64) ||
        !make_map(&tw3, W3, n, (uint64_t)E * d, 64, 64) ||
        !make_map(&tout, dXg, d, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = 2 * n;
    args.NB = d / BN;
    args.out = dXg;
    args.out_ld = d;
    args.err = err;
    args.bn_rows = d;
    args.kb_half = n / BK;
    const int tiles = R / BM + E;
    // CTA pairs (M = 256, each CTA half of B) where the forward GEMMs use them
    cudaError_t e =
        use_pair(R, E)
            ? launch_ew_auto<kDX, true>(ta1, tw1, tw3, tout, ta3, tout, args,
                                        (tiles / 2 + E) * args.NB, s)
            : launch_ew_auto<kDX, false>(ta1, tw1, tw3, tout, ta3, tout, args, tiles * args.NB, s);
    if (e != cudaSuccess) return e;
    return launch_combine(dXg, row_of_slot, T, K, d, dX, s);
}

cudaError_t launch_backward_dw(const __nv_bfloat16 *X, const __nv_bfloat16 *dY,
                               const __nv_bfloat16 *H, const __nv_bfloat16 *dA1,
                               const __nv_bfloat16 *dA3, const float *topk_w,
                               const int32_t *perm_token, const int32_t *perm_slot,
                               const int32_t *offsets, int T, int R, int d, int E, int n,
                               float *dW1, float *dW3, float *dW2, __nv_bfloat16 *pad,
                               int32_t *poff, uint32_t *err, cudaStream_t s) {
    const int64_t cap = (int64_t)R + 64 * E;
    // dW1 | dW3 = Xg^T [dA1 | dA3]: padded gathered X rows against dA1, dA3
    cudaError_t e = launch_gather_padded(X, perm_token, T, offsets, E, d, nullptr, nullptr, R, cap,
                                         poff, pad, false, s);
    if (e != cudaSuccess) return e;
    // outputs: fp32 boxes of 16 columns x 32 rows (one epilogue warp's rows)
    CUtensorMap tx, t1, t3, to1, to3;
    if (!make_map(&tx, pad, d, cap, 64, 64) || !make_map(&t1, dA1, n, R, 64, 64) ||
        !make_map(&t3, dA3, n, R, 64, 64) ||
        !make_map_f32(&to1, dW1, n, (uint64_t)E * d, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_f32(&to3, dW3, n, (uint64_t)E * d, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs a{};
    a.offsets = offsets;
    a.E = E;
    a.R = R;
    a.NB = n / 128;
    a.MT = d / BM;
    a.wout_rows = d;
    a.err = err;
    a.out_evict_first = 1;  // 4 d n E bytes that nothing reads back here
    // CTA pairs (256 output rows a unit) where the forward uses them
    const bool pair13 = use_pair(R, E) && a.MT % 2 == 0;
    e = pair13 ? launch_ew<kDW13, true, 4>(tx, t1, t3, to1, tx, to3, a, E * (a.MT / 2) * a.NB, s)
               : launch_ew<kDW13, false, 4>(tx, t1, t3, to1, tx, to3, a, E * a.MT * a.NB, s);
    if (e != cudaSuccess) return e;
    // dW2 = H^T (w dY)g: H rows against padded, w-scaled gathered dY rows
    e = launch_gather_padded(dY, perm_token, T, offsets, E, d, topk_w, perm_slot, R, cap, poff, pad,
                             true, s);
    if (e != cudaSuccess) return e;
    CUtensorMap th, ty, to2;
    if (!make_map(&th, H, n, R, 64, 64) || !make_map(&ty, pad, d, cap, 64, 64) ||
        !make_map_f32(&to2, dW2, d, (uint64_t)E * n, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs b{};
    b.offsets = offsets;
    b.E = E;
    b.R = R;
    b.NB = d / BN;
    b.MT = n / BM;
    b.wout_rows = n;
    b.err = err;
    b.out_evict_first = 1;
    const bool pair2 = use_pair(R, E) && b.MT % 2 == 0;
    return pair2 ? launch_ew<kDW2, true, 4>(th, ty, ty, to2, th, to2, b, E * (b.MT / 2) * b.NB, s)
                 : launch_ew<kDW2, false, 4>(th, ty, ty, to2, th, to2, b, E * b.MT * b.NB, s);
}

cudaError_t launch_router_dwr_tc(const __nv_bfloat16 *X, const __nv_bfloat16 *dLc,
                                 const int32_t *offsets, int T, int d, int E, int nchunks,
                                 float *P, uint32_t *err, cudaStream_t s) {
    // the weight-gradient GEMM with the token chunks as its groups: A = X rows
    // (MN-major over d), B = dLc rows (2E columns), outputs [chunk][d][2E] fp32
    CUtensorMap ta, tb, to;
    if (!make_map(&ta, X, d, T, 64, 64) || !make_map(&tb, dLc, 2 * (uint64_t)E, T, 64, 64) ||
        !make_map_f32(&to, P, 2 * (uint64_t)E, (uint64_t)nchunks * d, 16, 32,
                      CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs b{};
    b.offsets = offsets;
    b.E = nchunks;
    b.R = T;
    b.NB = 2 * E / BN;
    b.MT = d / BM;
    b.wout_rows = d;
    b.err = err;
    return launch_ew<kDW2, false, 4>(ta, tb, tb, to, ta, to, b, nchunks * b.MT * b.NB, s);
}

cudaError_t launch_router_dx_tc(const __nv_bfloat16 *dLc, const __nv_bfloat16 *WrA,
                                const __nv_bfloat16 *WrB, const int32_t *offsets, int T, int d,
                                int E, float *dXr, uint32_t *err, cudaStream_t s) {
    // the dX GEMM mode over the tokens as one group: A = dLc [T, 2E] in both
    // halves of the 4E reduction, B = WrA then WrB ([d, 2E], K-major); fp32 out
    CUtensorMap ta, tb0, tb1, to;
    if (!make_map(&ta, dLc, 2 * (uint64_t)E, T, 64, BM) ||
        !make_map(&tb0, WrA, 2 * (uint64_t)E, d, 64, 64) ||
        !make_map(&tb1, WrB, 2 * (uint64_t)E, d, 64, 64) ||
        !make_map_f32(&to, dXr, d, T, 16, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs a{};
    a.offsets = offsets;
    a.E = 1;
    a.R = T;
    a.Kdim = 4 * E;
    a.NB = d / BN;
    a.out_ld = d;
    a.outf = dXr;
    a.f32_out = 1;
    a.err = err;
    a.bn_rows = d;
    a.kb_half = 2 * E / BK;
    const int tiles = T / BM + 1;
    return launch_ew_auto<kDX, false>(ta, tb0, tb1, to, ta, to, a, tiles * a.NB, s);
}

cudaError_t launch_wait_timeout_selftest(uint32_t *err, cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err);
    return cudaGetLastError();
}

bool gemm_uses_pair(int R, int E) { return use_pair(R, E); }

namespace {
// CTAs of a fused launch and the most rounds its units can take.
int fused_grid(int R, int d, int E, int n) {
    const int64_t tiles = R / BM + E;  // upper bound of the 128-row tiles
    return (int)std::max<int64_t>(1, std::min<int64_t>(sm_count(), tiles * (n / 128 + d / BN)));
}
int64_t fused_rounds_bound(int R, int d, int E, int n) {
    const int64_t tiles = R / BM + E, G = fused_grid(R, d, E, n);
    return (tiles * (n / 128) + G - 1) / G + (tiles * (d / BN) + G - 1) / G;
}
}  // namespace

// The fused kernel runs on request only (MOE_GEMM_FUSED=1): measured on the
// SonicMoE-shaped layer it takes 0.183-0.191 ms against 0.170 ms for the two
// launches, and on the 512-token layer it ties. It needs n <= 2048 (a counter
// target, epilogue warps x gate/up column blocks, that fits a counter word) and
// units that fit kMaxRounds rounds; otherwise the two launches run.
bool use_fused_mlp(int R, int d, int E, int n) {
    const char *env = getenv("MOE_GEMM_FUSED");
    if (env == nullptr || env[0] != '1') return false;
    return n % 128 == 0 && d % BN == 0 && n <= 2048 && (n / 128) * 8 < (1 << kDepCountBits) &&
           fused_rounds_bound(R, d, E, n) <= kMaxRounds;
}

cudaError_t launch_gemm_down(const __nv_bfloat16 *H, const __nv_bfloat16 *W2,
                             const float *topk_w, const int32_t *perm_slot,
                             const int32_t *offsets, int R, int d, int E, int n,
                             __nv_bfloat16 *Z, uint32_t *err, cudaStream_t s) {
    CUtensorMap ta, tb0, tz;
    if (!make_map(&ta, H, n, R, 64, BM) || !make_map(&tb0, W2, d, (uint64_t)E * n, 64, BK) ||
        !make_map(&tz, Z, d, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
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
    return launch_gemm<kDown>(ta, tb0, tb0, tz, args, s);
}

cudaError_t launch_expert_mlp(const __nv_bfloat16 *X, const int32_t *perm_token, int T,
                              const __nv_bfloat16 *W1, const __nv_bfloat16 *W3,
                              const __nv_bfloat16 *W2, const float *topk_w,
                              const int32_t *perm_slot, const int32_t *offsets, int R, int d,
                              int E, int n, __nv_bfloat16 *H, __nv_bfloat16 *Z,
                              __nv_bfloat16 *xg, uint32_t *dep, uint32_t *err, cudaStream_t s) {
    if (!use_fused_mlp(R, d, E, n)) {
        cudaError_t e = launch_gemm_gate_up(X, perm_token, T, W1, W3, offsets, R, d, E, n, H, xg,
                                            err, s);
        if (e != cudaSuccess) return e;
        return launch_gemm_down(H, W2, topk_w, perm_slot, offsets, R, d, E, n, Z, err, s);
    }
    CUtensorMap th_in, tb0, tb1, th_out, tw2, tz;
    if (!make_map(&th_in, H, n, R, 64, BM) || !make_map(&tb0, W1, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&tb1, W3, n, (uint64_t)E * d, 64, BK) ||
        !make_map(&th_out, H, n, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&tw2, W2, d, (uint64_t)E * n, 64, BK) ||
        !make_map(&tz, Z, d, R, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    GemmArgs args{};
    args.X = X;
    args.perm_token = perm_token;
    args.T = T;
    args.offsets = offsets;
    args.E = E;
    args.R = R;
    args.Kdim = d;
    args.NB = n / 128;
    args.out = H;
    args.out_ld = n;
    args.topk_w = topk_w;
    args.perm_slot = perm_slot;
    args.err = err;
    args.Kdim2 = n;
    args.NB2 = d / BN;
    args.out2 = Z;
    args.out2_ld = d;
    args.dep = dep;
    int gap = 2;
    if (const char *v = getenv("MOE_FUSED_GAP_ROUNDS")) gap = max(0, atoi(v));
    args.gap_rounds = gap;
    return launch_ew<kFused, false, 8>(th_in, tb0, tb1, th_out, tw2, tz, args,
                                       fused_grid(R, d, E, n), s);
}

}  // namespace moe
