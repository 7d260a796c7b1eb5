// C ABI of libmoe.so: argument checking, workspace layout and the sequence of
// kernel launches for each entry point declared in include/moe.h.
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {
namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per device, filled on first use under a mutex and published with a
// release store, so host threads calling at once see either nothing or all of it.
struct DeviceInfo {
    std::atomic<bool> init{false};
    std::mutex m;
    bool arch_ok = false;
    int sms = 0;
};
DeviceInfo g_dev[64];

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    DeviceInfo &di = g_dev[dev];
    if (!di.init.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(di.m);
        if (!di.init.load(std::memory_order_relaxed)) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return nullptr;
            di.arch_ok = (major == 10 && minor == 3);
            di.sms = sms;
            di.init.store(true, std::memory_order_release);
        }
    }
    return &di;
}

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Router-level shape rules.
moe_status_t check_route_shape(int T, int d, int E, int K) {
    if (T < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
    if (d < 0) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || K > kMaxK || K > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d != -1 && (d < 8 || d % 8 != 0)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)T * K >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// Expert-GEMM shape rules.
moe_status_t check_mlp_shape(int T, int d, int E, int K, int n) {
    moe_status_t s = check_route_shape(T, d, E, K);
    if (s != MOE_OK) return s;
    if (n < 1) return MOE_ERR_INVALID_ARG;
    if (d % 256 != 0 || n % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int64_t R = (int64_t)T * K;
    if (R * (d > n ? d : n) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Records a caller's timing event on st. Inside a stream capture the record
// becomes an external event node, so each replay of the graph records it.
bool record_event(void *event, cudaStream_t st) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
    const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u;
    return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(event), st, flags) == cudaSuccess;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

}  // namespace

moe_status_t check_arch() {
    // a failed call made by someone else earlier must not be reported as ours
    (void)cudaGetLastError();
    const DeviceInfo *di = device_info();
    if (di == nullptr) return MOE_ERR_CUDA;
    return di->arch_ok ? MOE_OK : MOE_ERR_ARCH;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = getenv("MOE_PDL");
        return !(v != nullptr && v[0] == '0');
    }();
    return on;
}

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}
}  // namespace

bool current_context_id(unsigned long long *id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

cudaError_t ensure_dynamic_smem(const void *kernel, int bytes) {
    struct Done {
        const void *kernel;
        unsigned long long ctx;
        int bytes;
    };
    static std::mutex m;
    static std::vector<Done> done;
    unsigned long long id = 0;
    bool known = current_context_id(&id);
    if (known) {
        std::lock_guard<std::mutex> lock(m);
        for (const Done &x : done)
            if (x.kernel == kernel && x.ctx == id && x.bytes >= bytes) return cudaSuccess;
    }
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (!known) known = current_context_id(&id);  // the call made the context current
    if (known) {
        std::lock_guard<std::mutex> lock(m);
        done.push_back({kernel, id, bytes});
    }
    return cudaSuccess;
}

int sm_count() {
    const DeviceInfo *di = device_info();
    return (di != nullptr && di->sms > 0) ? di->sms : 1;
}

int64_t round_capacity(int T, int E, int K, int M) {
    const int64_t a = (int64_t)T * E, b = (int64_t)T * K + (int64_t)E * (M / 2);
    return a < b ? a : b;
}

namespace {

WsLayout layout_impl(int T, int d, int E, int K, int n, size_t R, bool rounded) {
    WsLayout L{};
    L.rows = R;
    L.nchunks = (T + kChunk - 1) / kChunk;
    L.max_tiles = (int)(R / kTileM) + E;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.err = take(64);
    // right after the control words at the same offset in every shape: only the
    // one-kernel grouping writes these flags (a call's tag could otherwise meet a
    // stale value another kernel left there)
    L.group_flags = take(4 * (size_t)kGroupMaxBlocks);
    L.group_agg = take(4 * (size_t)kGroupMaxBlocks * E);
    L.counts = take(4 * (size_t)E);
    L.offsets = take(4 * (size_t)(E + 1));
    L.tile_base = take(4 * (size_t)(E + 1));
    L.totals = take(4 * (size_t)E);
    L.chunk_base = take(4 * (size_t)E * L.nchunks);
    L.rank = take(4 * R);
    L.perm_token = take(4 * R);
    L.perm_slot = take(4 * R);
    L.row_of_slot = take(4 * R);
    L.topk_idx = take(4 * R);
    L.topk_w = take(4 * R);
    L.tiles = take(16 * (size_t)L.max_tiles);
    L.num_tiles = take(4);
    L.grouping_end = off;
    L.dep = take(4 * (size_t)L.max_tiles);
    L.xg = take(2 * R * (size_t)d);
    L.h = take(2 * R * (size_t)n);
    L.z = take(2 * R * (size_t)d);
    L.logits = take(4 * (size_t)T * E);
    if (rounded) {
        L.counts_round = take(4 * (size_t)E);
        L.row_map = take(4 * (size_t)T * E);
        L.row_w = take(4 * R);
        L.round_scratch = take(round_scratch_bytes(T, E));
        L.tok_rows = take(4 * (size_t)T * kTokCap);
        L.tok_n = take(4 * (size_t)T);
    }
    L.total = off;
    return L;
}

}  // namespace

WsLayout ws_layout(int T, int d, int E, int K, int n) {
    return layout_impl(T, d, E, K, n, (size_t)T * K, false);
}

WsLayout ws_layout_rounded(int T, int d, int E, int K, int n) {
    return layout_impl(T, d, E, K, n, (size_t)round_capacity(T, E, K, kTileM), true);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
        case MOE_ERR_ARCH: return "MOE_ERR_ARCH";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
        default: return "MOE_ERR_UNKNOWN";
    }
}

int moe_abi_version(void) { return 101; }

int moe_expert_mlp_launches(int T, int d, int E, int K, int n, int rounded) {
    if ((rounded != 0 && rounded != 1) || check_mlp_shape(T, d, E, K, n) != MOE_OK) return -1;
    const int R = rounded ? (int)ws_layout_rounded(T, d, E, K, n).rows : T * K;
    return use_fused_mlp(R, d, E, n) ? 1 : (gemm_uses_pair(R, E) ? 3 : 2);
}

int moe_forward_launches(int T, int d, int E, int K, int n, int rounded) {
    const int gemms = moe_expert_mlp_launches(T, d, E, K, n, rounded);
    if (gemms < 0) return -1;
    // router 1 or 2 (with 16-byte-aligned router weights), grouping 1 (3 for
    // T > 65536) or rounding 3, combine 1, and the expert GEMMs
    const int grouping = rounded ? 3 : permute_launch_count(T);
    return (route_is_one_kernel(d, E, true) ? 1 : 2) + grouping + gemms + 1;
}

size_t moe_workspace_bytes(int T, int d, int E, int K, int n) {
    if (T < 1 || E < 1 || K < 1 || d < 0 || n < 0 || E > kMaxE || K > kMaxK || K > E) return 0;
    return ws_layout(T, d, E, K, n).total;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (ws == nullptr || ws_bytes < 64) return MOE_ERR_INVALID_ARG;
    // the control words and the one-kernel grouping's block flags, which sit at
    // the same offset in every shape (the first 512 bytes)
    const size_t n = ws_bytes < 512 ? ws_bytes : 512;
    return from_cuda(cudaMemsetAsync(ws, 0, n, as_stream(stream)));
}

moe_status_t moe_route(const moe_bf16 *X, const float *Wr, const float *bias, int T, int d, int E,
                       int K, int renorm, float *logits, int32_t *topk_idx, float *topk_w,
                       int32_t *counts, void *stream) {
    if (!X || !Wr || !logits || !topk_idx || !topk_w || !counts || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, d, E, K);
    if (s != MOE_OK) return s;
    if (!aligned16(X)) return MOE_ERR_INVALID_ARG;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_route(reinterpret_cast<const __nv_bfloat16 *>(X), Wr, bias, T, d, E, K,
                                  renorm, logits, topk_idx, topk_w, counts, as_stream(stream)));
}

moe_status_t moe_route_logits(const float *logits, int T, int E, int K, int renorm,
                              int32_t *topk_idx, float *topk_w, int32_t *counts, void *stream) {
    if (!logits || !topk_idx || !topk_w || !counts || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, 8, E, K);
    if (s != MOE_OK) return s;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(
        launch_route_logits(logits, T, E, K, renorm, topk_idx, topk_w, counts, as_stream(stream)));
}

moe_status_t moe_permute(const int32_t *topk_idx, const int32_t *counts, int T, int E, int K,
                         int32_t *offsets, int32_t *perm_token, int32_t *perm_slot,
                         int32_t *row_of_slot, int32_t *tiles, int32_t *num_tiles, void *ws,
                         size_t ws_bytes, void *stream) {
    if (!topk_idx || !offsets || !perm_token || !perm_slot || !row_of_slot || !tiles ||
        !num_tiles || !ws)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, 8, E, K);
    if (s != MOE_OK) return s;
    if (!aligned16(tiles)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, 0, E, K, 0);
    if (ws_bytes < L.grouping_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_permute(topk_idx, counts, T, E, K, offsets, perm_token, perm_slot,
                                    row_of_slot, tiles, num_tiles, L, static_cast<char *>(ws),
                                    as_stream(stream)));
}

moe_status_t moe_gemm_gate_up(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                              const int32_t *perm_token, const int32_t *offsets, int T, int d,
                              int E, int K, int n, moe_bf16 *H, void *ws, size_t ws_bytes,
                              void *stream) {
    if (!X || !W1 || !W3 || !perm_token || !offsets || !H || !ws) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(H))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, K, n);
    if (ws_bytes < L.h) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_gemm_gate_up(reinterpret_cast<const __nv_bfloat16 *>(X), perm_token, T,
                                         reinterpret_cast<const __nv_bfloat16 *>(W1),
                                         reinterpret_cast<const __nv_bfloat16 *>(W3), offsets,
                                         T * K, d, E, n, reinterpret_cast<__nv_bfloat16 *>(H),
                                         at<__nv_bfloat16>(ws, L.xg), at<uint32_t>(ws, L.err),
                                         as_stream(stream)));
}

moe_status_t moe_gemm_gate_up_train(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                                    const int32_t *perm_token, const int32_t *offsets, int T,
                                    int d, int E, int K, int n, moe_bf16 *H, float *A1,
                                    float *A3, void *ws, size_t ws_bytes, void *stream) {
    if (!X || !W1 || !W3 || !perm_token || !offsets || !H || !A1 || !A3 || !ws)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(H) || !aligned16(A1) ||
        !aligned16(A3))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, K, n);
    if (ws_bytes < L.h) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_gemm_gate_up_train(
        reinterpret_cast<const __nv_bfloat16 *>(X), perm_token, T,
        reinterpret_cast<const __nv_bfloat16 *>(W1), reinterpret_cast<const __nv_bfloat16 *>(W3),
        offsets, T * K, d, E, n, reinterpret_cast<__nv_bfloat16 *>(H), A1, A3,
        at<__nv_bfloat16>(ws, L.xg), at<uint32_t>(ws, L.err), as_stream(stream)));
}

moe_status_t moe_backward_dh(const moe_bf16 *dY, const moe_bf16 *W2, const float *A1,
                             const float *A3, const float *topk_w, const int32_t *perm_token,
                             const int32_t *perm_slot, const int32_t *offsets, int T, int d,
                             int E, int K, int n, moe_bf16 *dA1, moe_bf16 *dA3, float *dS,
                             void *ws, size_t ws_bytes, void *stream) {
    if (!dY || !W2 || !A1 || !A3 || !topk_w || !perm_token || !offsets || !dA1 || !dA3 || !dS ||
        !ws)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    // 256 hidden columns per unit; the dS partials (n/32 floats per row) live in
    // the workspace's H region (2*n bytes per row), the gathered dY rows of the
    // CTA-pair path in its gathered-rows region
    if (n % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(dY) || !aligned16(W2) || !aligned16(A1) || !aligned16(A3) || !aligned16(dA1) ||
        !aligned16(dA3))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, K, n);
    if (ws_bytes < L.z) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_backward_dh(
        reinterpret_cast<const __nv_bfloat16 *>(dY), perm_token, T,
        reinterpret_cast<const __nv_bfloat16 *>(W2), A1, A3, topk_w, perm_slot, offsets, T * K, d, E, n,
        reinterpret_cast<__nv_bfloat16 *>(dA1), reinterpret_cast<__nv_bfloat16 *>(dA3),
        at<__nv_bfloat16>(ws, L.xg), at<float>(ws, L.h), dS, at<uint32_t>(ws, L.err),
        as_stream(stream)));
}

moe_status_t moe_backward_dx(const moe_bf16 *dA1, const moe_bf16 *dA3, const moe_bf16 *W1,
                             const moe_bf16 *W3, const int32_t *offsets,
                             const int32_t *row_of_slot, int T, int d, int E, int K, int n,
                             moe_bf16 *dXg, moe_bf16 *dX, void *ws, size_t ws_bytes,
                             void *stream) {
    if (!dA1 || !dA3 || !W1 || !W3 || !offsets || !row_of_slot || !dXg || !dX || !ws)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(dA1) || !aligned16(dA3) || !aligned16(W1) || !aligned16(W3) ||
        !aligned16(dXg) || !aligned16(dX))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < 64) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_backward_dx(
        reinterpret_cast<const __nv_bfloat16 *>(dA1), reinterpret_cast<const __nv_bfloat16 *>(dA3),
        reinterpret_cast<const __nv_bfloat16 *>(W1), reinterpret_cast<const __nv_bfloat16 *>(W3),
        offsets, row_of_slot, T, K, T * K, d, E, n, reinterpret_cast<__nv_bfloat16 *>(dXg),
        reinterpret_cast<__nv_bfloat16 *>(dX), at<uint32_t>(ws, 0), as_stream(stream)));
}

moe_status_t moe_backward_router(const moe_bf16 *X, const float *Wr, const float *logits,
                                 const int32_t *topk_idx, const float *dS,
                                 const int32_t *row_of_slot, int T, int d, int E, int K,
                                 int renorm, const moe_bf16 *dXg, moe_bf16 *dX, float *dL,
                                 float *dWr, float *dbias, void *ws, size_t ws_bytes,
                                 void *stream) {
    if (!X || !Wr || !logits || !topk_idx || !dS || !row_of_slot || !dXg || !dX || !dL || !dWr ||
        !dbias || !ws || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, d, E, K);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(dXg) || !aligned16(dX)) return MOE_ERR_INVALID_ARG;
    // the partial sums of dWr (at most T * d floats) live in the workspace from
    // the gathered-rows region on (that region and the ones after it hold >= 4*T*d bytes)
    const WsLayout L = ws_layout(T, d, E, K, 0);
    const size_t need = L.xg + (size_t)T * d * sizeof(float);
    if (ws_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    // the region after the gathered rows serves as a second scratch (the
    // tensor-core path's split operands) when the first one, T * d floats, ends
    // before it (K >= 2)
    const bool s2 = ws_bytes > L.z && L.z >= need;
    return from_cuda(launch_backward_router(
        reinterpret_cast<const __nv_bfloat16 *>(X), Wr, logits, topk_idx, dS, row_of_slot, T, d, E,
        K, renorm, reinterpret_cast<const __nv_bfloat16 *>(dXg), dL, dWr, dbias,
        at<float>(ws, L.xg), s2 ? at<char>(ws, L.z) : nullptr, s2 ? ws_bytes - L.z : 0,
        reinterpret_cast<__nv_bfloat16 *>(dX),
        at<uint32_t>(ws, L.err), as_stream(stream)));
}

size_t moe_backward_dw_scratch_bytes(int T, int d, int E, int K) {
    if (T < 1 || E < 1 || K < 1 || d < 1 || E > kMaxE || K > kMaxK || K > E) return 0;
    const size_t pad = ((size_t)T * K + 64 * (size_t)E) * d * 2;
    return 256 + (pad + 255) / 256 * 256 + 4 * (size_t)(E + 1);
}

moe_status_t moe_backward_dw(const moe_bf16 *X, const moe_bf16 *dY, const moe_bf16 *H,
                             const moe_bf16 *dA1, const moe_bf16 *dA3, const float *topk_w,
                             const int32_t *perm_token, const int32_t *perm_slot,
                             const int32_t *offsets, int T, int d, int E, int K, int n,
                             float *dW1, float *dW3, float *dW2, void *scratch,
                             size_t scratch_bytes, void *stream) {
    if (!X || !dY || !H || !dA1 || !dA3 || !topk_w || !perm_token || !perm_slot || !offsets ||
        !dW1 || !dW3 || !dW2 || !scratch)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(dY) || !aligned16(H) || !aligned16(dA1) || !aligned16(dA3) ||
        !aligned16(dW1) || !aligned16(dW3) || !aligned16(dW2) ||
        (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
        return MOE_ERR_INVALID_ARG;
    if (scratch_bytes < moe_backward_dw_scratch_bytes(T, d, E, K)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    const size_t pad = ((size_t)T * K + 64 * (size_t)E) * d * 2;
    char *base = static_cast<char *>(scratch);
    return from_cuda(launch_backward_dw(
        reinterpret_cast<const __nv_bfloat16 *>(X), reinterpret_cast<const __nv_bfloat16 *>(dY),
        reinterpret_cast<const __nv_bfloat16 *>(H), reinterpret_cast<const __nv_bfloat16 *>(dA1),
        reinterpret_cast<const __nv_bfloat16 *>(dA3), topk_w, perm_token, perm_slot, offsets, T,
        T * K, d, E, n, dW1, dW3, dW2, reinterpret_cast<__nv_bfloat16 *>(base + 256),
        reinterpret_cast<int32_t *>(base + 256 + (pad + 255) / 256 * 256),
        reinterpret_cast<uint32_t *>(base), as_stream(stream)));
}

moe_status_t moe_gemm_down(const moe_bf16 *H, const moe_bf16 *W2, const float *topk_w,
                           const int32_t *perm_slot, const int32_t *offsets, int T, int d, int E,
                           int K, int n, moe_bf16 *Z, void *ws, size_t ws_bytes, void *stream) {
    if (!H || !W2 || !topk_w || !offsets || !Z || !ws) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(H) || !aligned16(W2) || !aligned16(Z)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < 64) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    const WsLayout L = ws_layout(T, d, E, K, n);
    return from_cuda(launch_gemm_down(reinterpret_cast<const __nv_bfloat16 *>(H),
                                      reinterpret_cast<const __nv_bfloat16 *>(W2), topk_w,
                                      perm_slot, offsets, T * K, d, E, n,
                                      reinterpret_cast<__nv_bfloat16 *>(Z),
                                      at<uint32_t>(ws, L.err), as_stream(stream)));
}

moe_status_t moe_expert_mlp(const moe_bf16 *X, const moe_bf16 *W1, const moe_bf16 *W3,
                            const moe_bf16 *W2, const float *topk_w, const int32_t *perm_token,
                            const int32_t *perm_slot, const int32_t *offsets, int T, int d, int E,
                            int K, int n, moe_bf16 *H, moe_bf16 *Z, void *ws, size_t ws_bytes,
                            void *stream) {
    if (!X || !W1 || !W3 || !W2 || !topk_w || !perm_token || !offsets || !H || !Z || !ws)
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(H) ||
        !aligned16(Z))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, K, n);
    if (ws_bytes < L.h) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_expert_mlp(
        reinterpret_cast<const __nv_bfloat16 *>(X), perm_token, T,
        reinterpret_cast<const __nv_bfloat16 *>(W1), reinterpret_cast<const __nv_bfloat16 *>(W3),
        reinterpret_cast<const __nv_bfloat16 *>(W2), topk_w, perm_slot, offsets, T * K, d, E, n,
        reinterpret_cast<__nv_bfloat16 *>(H), reinterpret_cast<__nv_bfloat16 *>(Z),
        at<__nv_bfloat16>(ws, L.xg), at<uint32_t>(ws, L.dep), at<uint32_t>(ws, L.err),
        as_stream(stream)));
}

moe_status_t moe_combine(const moe_bf16 *Z, const int32_t *row_of_slot, int T, int K, int d,
                         moe_bf16 *Y, void *stream) {
    if (!Z || !row_of_slot || !Y) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, d, K, K);
    if (s != MOE_OK) return s;
    if (!aligned16(Z) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_combine(reinterpret_cast<const __nv_bfloat16 *>(Z), row_of_slot, T, K,
                                    d, reinterpret_cast<__nv_bfloat16 *>(Y), as_stream(stream)));
}

moe_status_t moe_forward_traced(const moe_bf16 *X, const float *Wr, const float *bias,
                                const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2, int T,
                                int d, int E, int K, int n, int renorm, moe_bf16 *Y,
                                int32_t *topk_idx_out, float *topk_w_out, void *ws,
                                size_t ws_bytes, void *stream, void *const *events,
                                int n_events) {
    if (!X || !Wr || !W1 || !W3 || !W2 || !Y || !ws || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    if (n_events < 0 || (n_events > 0 && events == nullptr)) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(Y))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, K, n);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    cudaStream_t st = as_stream(stream);
    int ev = 0;
    auto mark = [&]() -> bool {
        if (ev < n_events && !record_event(events[ev], st)) return false;
        ++ev;
        return true;
    };
    const int R = T * K;
    uint32_t *err = at<uint32_t>(ws, L.err);
    int32_t *idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.topk_idx);
    float *w = topk_w_out ? topk_w_out : at<float>(ws, L.topk_w);
    int32_t *counts = at<int32_t>(ws, L.counts);
    int32_t *offsets = at<int32_t>(ws, L.offsets);
    int32_t *perm_token = at<int32_t>(ws, L.perm_token);
    int32_t *perm_slot = at<int32_t>(ws, L.perm_slot);
    int32_t *row_of_slot = at<int32_t>(ws, L.row_of_slot);
    __nv_bfloat16 *h = at<__nv_bfloat16>(ws, L.h);
    __nv_bfloat16 *z = at<__nv_bfloat16>(ws, L.z);
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(X);

    if (!mark()) return MOE_ERR_CUDA;
    if (launch_route(x, Wr, bias, T, d, E, K, renorm, at<float>(ws, L.logits), idx, w, counts,
                     st) != cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    // the expert GEMMs decode their units from the offsets, so the tile list is
    // not written here (moe_permute writes it for callers that schedule tiles)
    if (launch_permute(idx, counts, T, E, K, offsets, perm_token, perm_slot, row_of_slot, nullptr,
                       nullptr, L, static_cast<char *>(ws), st) != cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    if (use_fused_mlp(R, d, E, n)) {
        // one launch for both GEMMs: its time is the gate/up stage, the down
        // stage's events are adjacent
        if (launch_expert_mlp(x, perm_token, T, reinterpret_cast<const __nv_bfloat16 *>(W1),
                              reinterpret_cast<const __nv_bfloat16 *>(W3),
                              reinterpret_cast<const __nv_bfloat16 *>(W2), w, perm_slot, offsets,
                              R, d, E, n, h, z, at<__nv_bfloat16>(ws, L.xg),
                              at<uint32_t>(ws, L.dep), err, st) != cudaSuccess ||
            !mark() || !mark())
            return MOE_ERR_CUDA;
    } else {
        if (launch_gemm_gate_up(x, perm_token, T, reinterpret_cast<const __nv_bfloat16 *>(W1),
                                reinterpret_cast<const __nv_bfloat16 *>(W3), offsets, R, d, E, n,
                                h, at<__nv_bfloat16>(ws, L.xg), err, st) != cudaSuccess ||
            !mark())
            return MOE_ERR_CUDA;
        if (launch_gemm_down(h, reinterpret_cast<const __nv_bfloat16 *>(W2), w, perm_slot,
                             offsets, R, d, E, n, z, err, st) != cudaSuccess ||
            !mark())
            return MOE_ERR_CUDA;
    }
    if (launch_combine(z, row_of_slot, T, K, d, reinterpret_cast<__nv_bfloat16 *>(Y), st) !=
            cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t moe_forward(const moe_bf16 *X, const float *Wr, const float *bias,
                         const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2, int T, int d,
                         int E, int K, int n, int renorm, moe_bf16 *Y, int32_t *topk_idx_out,
                         float *topk_w_out, void *ws, size_t ws_bytes, void *stream) {
    return moe_forward_traced(X, Wr, bias, W1, W3, W2, T, d, E, K, n, renorm, Y, topk_idx_out,
                              topk_w_out, ws, ws_bytes, stream, nullptr, 0);
}

moe_status_t moe_forward_host(const moe_bf16 *X_host, moe_bf16 *Y_host, moe_bf16 *X_dev,
                              moe_bf16 *Y_dev, const float *Wr, const float *bias,
                              const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2, int T,
                              int d, int E, int K, int n, int renorm, void *ws, size_t ws_bytes,
                              void *stream) {
    if (!X_host || !Y_host || !X_dev || !Y_dev) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    cudaStream_t st = as_stream(stream);
    const size_t bytes = (size_t)T * d * sizeof(moe_bf16);
    if (cudaMemcpyAsync(X_dev, X_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    s = moe_forward(X_dev, Wr, bias, W1, W3, W2, T, d, E, K, n, renorm, Y_dev, nullptr, nullptr, ws,
                    ws_bytes, stream);
    if (s != MOE_OK) return s;
    if (cudaMemcpyAsync(Y_host, Y_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return from_cuda(cudaStreamSynchronize(st));
}

moe_status_t moe_forward_host_stream(const moe_bf16 *X_host, moe_bf16 *Y_host, int n_batches,
                                     moe_bf16 *X_dev2, moe_bf16 *Y_dev2, const float *Wr,
                                     const float *bias, const moe_bf16 *W1, const moe_bf16 *W3,
                                     const moe_bf16 *W2, int T, int d, int E, int K, int n,
                                     int renorm, void *ws, size_t ws_bytes, void *stream,
                                     void *h2d_stream, void *d2h_stream) {
    if (!X_host || !Y_host || !X_dev2 || !Y_dev2 || n_batches < 0) return MOE_ERR_INVALID_ARG;
    if (stream == h2d_stream || stream == d2h_stream || h2d_stream == d2h_stream)
        return MOE_ERR_INVALID_ARG;  // the overlap needs three distinct streams
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    if (n_batches == 0) return MOE_OK;
    cudaStream_t sc = as_stream(stream), sin = as_stream(h2d_stream), sout = as_stream(d2h_stream);
    const size_t elems = (size_t)T * d, bytes = elems * sizeof(moe_bf16);
    // per device buffer b: X landed / X free again (layer done) / Y written / Y copied out
    cudaEvent_t x_in[2], x_free[2], y_done[2], y_out[2];
    int created = 0;
    cudaError_t ce = cudaSuccess;
    for (int b = 0; b < 2 && ce == cudaSuccess; ++b) {
        cudaEvent_t *evs[4] = {&x_in[b], &x_free[b], &y_done[b], &y_out[b]};
        for (int k = 0; k < 4 && ce == cudaSuccess; ++k) {
            ce = cudaEventCreateWithFlags(evs[k], cudaEventDisableTiming);
            if (ce == cudaSuccess) ++created;
        }
    }
    auto destroy = [&]() {
        int left = created;
        for (int b = 0; b < 2; ++b) {
            cudaEvent_t evs[4] = {x_in[b], x_free[b], y_done[b], y_out[b]};
            for (int k = 0; k < 4 && left > 0; ++k, --left) cudaEventDestroy(evs[k]);
        }
    };
    if (ce != cudaSuccess) {
        destroy();
        return MOE_ERR_CUDA;
    }
    s = MOE_OK;
    for (int i = 0; i < n_batches && s == MOE_OK; ++i) {
        const int b = i & 1;
        moe_bf16 *xd = X_dev2 + b * elems, *yd = Y_dev2 + b * elems;
        // upload batch i once the layer of batch i-2 no longer reads this buffer
        if ((i >= 2 && cudaStreamWaitEvent(sin, x_free[b], 0) != cudaSuccess) ||
            cudaMemcpyAsync(xd, X_host + (size_t)i * elems, bytes, cudaMemcpyHostToDevice, sin) !=
                cudaSuccess ||
            cudaEventRecord(x_in[b], sin) != cudaSuccess) {
            s = MOE_ERR_CUDA;
            break;
        }
        // the layer, after the upload and after batch i-2's output has left yd
        if (cudaStreamWaitEvent(sc, x_in[b], 0) != cudaSuccess ||
            (i >= 2 && cudaStreamWaitEvent(sc, y_out[b], 0) != cudaSuccess)) {
            s = MOE_ERR_CUDA;
            break;
        }
        s = moe_forward(xd, Wr, bias, W1, W3, W2, T, d, E, K, n, renorm, yd, nullptr, nullptr, ws,
                        ws_bytes, stream);
        if (s != MOE_OK) break;
        if (cudaEventRecord(x_free[b], sc) != cudaSuccess ||
            cudaEventRecord(y_done[b], sc) != cudaSuccess ||
            cudaStreamWaitEvent(sout, y_done[b], 0) != cudaSuccess ||
            cudaMemcpyAsync(Y_host + (size_t)i * elems, yd, bytes, cudaMemcpyDeviceToHost, sout) !=
                cudaSuccess ||
            cudaEventRecord(y_out[b], sout) != cudaSuccess)
            s = MOE_ERR_CUDA;
    }
    const cudaError_t e1 = cudaStreamSynchronize(sin), e2 = cudaStreamSynchronize(sc),
                      e3 = cudaStreamSynchronize(sout);
    destroy();
    if (s != MOE_OK) return s;
    return (e1 == cudaSuccess && e2 == cudaSuccess && e3 == cudaSuccess) ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, void *stream) {
    if (ws == nullptr || ws_bytes < 64) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_arch();
    if (s != MOE_OK) return s;
    return from_cuda(launch_wait_timeout_selftest(at<uint32_t>(ws, 0), as_stream(stream)));
}

moe_status_t moe_sync_check(void *ws, void *stream, uint32_t *word_out) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (word != 0 && cudaMemset(ws, 0, sizeof word) != cudaSuccess) return MOE_ERR_CUDA;
    if (word_out != nullptr) *word_out = word;
    if (word & MOE_DEVERR_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    if (word != 0) return MOE_ERR_DEVICE_CHECK;
    return MOE_OK;
}


// ------------------------------------------------------------ Token Rounding

int64_t moe_round_capacity(int T, int E, int K, int M) {
    if (T < 1 || E < 1 || K < 1 || K > E || M < 1) return -1;
    return round_capacity(T, E, K, M);
}

size_t moe_round_workspace_bytes(int T, int E) {
    if (T < 1 || E < 1 || E > kMaxE) return 0;
    return 256 + round_scratch_bytes(T, E);
}

moe_status_t moe_round_routing(const float *logits, const int32_t *topk_idx,
                               const int32_t *counts, int T, int E, int K, int M, int renorm,
                               int32_t *counts_out, int32_t *offsets, int32_t *perm_token,
                               int32_t *row_map, float *row_w, int32_t *tiles,
                               int32_t *num_tiles, void *ws, size_t ws_bytes, void *stream) {
    if (!logits || !topk_idx || !counts || !counts_out || !offsets || !perm_token || !row_map ||
        !row_w || !tiles || !num_tiles || !ws || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, 8, E, K);
    if (s != MOE_OK) return s;
    if (M < 1) return MOE_ERR_INVALID_ARG;
    if (M > kMaxRoundM || (int64_t)T * E >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(tiles)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_round_workspace_bytes(T, E)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    void *scratch = static_cast<char *>(ws) + 256;
    return from_cuda(launch_round(logits, topk_idx, counts, T, E, K, M, renorm, counts_out,
                                  offsets, perm_token, row_map, row_w, tiles, num_tiles, nullptr,
                                  nullptr, scratch, at<uint32_t>(ws, 0), as_stream(stream)));
}

moe_status_t moe_combine_rows(const moe_bf16 *Z, const int32_t *row_map, int T, int E, int d,
                              int64_t rows, moe_bf16 *Y, void *stream) {
    if (!Z || !row_map || !Y || rows < 0) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_route_shape(T, d, E, 1);
    if (s != MOE_OK) return s;
    if (!aligned16(Z) || !aligned16(Y)) return MOE_ERR_INVALID_ARG;
    if ((s = check_arch()) != MOE_OK) return s;
    return from_cuda(launch_combine_rows(reinterpret_cast<const __nv_bfloat16 *>(Z), row_map,
                                         nullptr, nullptr, T, E, d, rows,
                                         reinterpret_cast<__nv_bfloat16 *>(Y), as_stream(stream)));
}

size_t moe_workspace_bytes_rounded(int T, int d, int E, int K, int n) {
    if (T < 1 || E < 1 || K < 1 || d < 0 || n < 0 || E > kMaxE || K > kMaxK || K > E) return 0;
    return ws_layout_rounded(T, d, E, K, n).total;
}

moe_status_t moe_forward_rounded_traced(const moe_bf16 *X, const float *Wr, const float *bias,
                                        const moe_bf16 *W1, const moe_bf16 *W3,
                                        const moe_bf16 *W2, int T, int d, int E, int K, int n,
                                        int renorm, moe_bf16 *Y, int32_t *row_map_out, void *ws,
                                        size_t ws_bytes, void *stream, void *const *events,
                                        int n_events) {
    if (!X || !Wr || !W1 || !W3 || !W2 || !Y || !ws || (renorm != 0 && renorm != 1))
        return MOE_ERR_INVALID_ARG;
    if (n_events < 0 || (n_events > 0 && events == nullptr)) return MOE_ERR_INVALID_ARG;
    moe_status_t s = check_mlp_shape(T, d, E, K, n);
    if (s != MOE_OK) return s;
    const WsLayout L = ws_layout_rounded(T, d, E, K, n);
    if ((int64_t)L.rows * (d > n ? d : n) >= (1ll << 31) || (int64_t)T * E >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(Y))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((s = check_arch()) != MOE_OK) return s;
    cudaStream_t st = as_stream(stream);
    int ev = 0;
    auto mark = [&]() -> bool {
        if (ev < n_events && !record_event(events[ev], st)) return false;
        ++ev;
        return true;
    };
    const int R = (int)L.rows;
    uint32_t *err = at<uint32_t>(ws, L.err);
    float *logits = at<float>(ws, L.logits);
    int32_t *idx = at<int32_t>(ws, L.topk_idx);
    float *w = at<float>(ws, L.topk_w);
    int32_t *counts = at<int32_t>(ws, L.counts);
    int32_t *counts_r = at<int32_t>(ws, L.counts_round);
    int32_t *offsets = at<int32_t>(ws, L.offsets);
    int32_t *perm_token = at<int32_t>(ws, L.perm_token);
    int32_t *row_map = row_map_out ? row_map_out : at<int32_t>(ws, L.row_map);
    float *row_w = at<float>(ws, L.row_w);
    __nv_bfloat16 *h = at<__nv_bfloat16>(ws, L.h);
    __nv_bfloat16 *z = at<__nv_bfloat16>(ws, L.z);
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(X);
    void *scratch = static_cast<char *>(ws) + L.round_scratch;

    if (!mark()) return MOE_ERR_CUDA;
    if (launch_route(x, Wr, bias, T, d, E, K, renorm, logits, idx, w, counts, st) != cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    if (launch_round(logits, idx, counts, T, E, K, kTileM, renorm, counts_r, offsets, perm_token,
                     row_map, row_w, at<int32_t>(ws, L.tiles), at<int32_t>(ws, L.num_tiles),
                     at<int32_t>(ws, L.tok_rows), at<int32_t>(ws, L.tok_n), scratch, err,
                     st) != cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    // the weight of grouped row p is row_w[p] (no slot indirection)
    if (use_fused_mlp(R, d, E, n)) {
        if (launch_expert_mlp(x, perm_token, T, reinterpret_cast<const __nv_bfloat16 *>(W1),
                              reinterpret_cast<const __nv_bfloat16 *>(W3),
                              reinterpret_cast<const __nv_bfloat16 *>(W2), row_w, nullptr,
                              offsets, R, d, E, n, h, z, at<__nv_bfloat16>(ws, L.xg),
                              at<uint32_t>(ws, L.dep), err, st) != cudaSuccess ||
            !mark() || !mark())
            return MOE_ERR_CUDA;
    } else {
        if (launch_gemm_gate_up(x, perm_token, T, reinterpret_cast<const __nv_bfloat16 *>(W1),
                                reinterpret_cast<const __nv_bfloat16 *>(W3), offsets, R, d, E, n,
                                h, at<__nv_bfloat16>(ws, L.xg), err, st) != cudaSuccess ||
            !mark())
            return MOE_ERR_CUDA;
        if (launch_gemm_down(h, reinterpret_cast<const __nv_bfloat16 *>(W2), row_w, nullptr,
                             offsets, R, d, E, n, z, err, st) != cudaSuccess ||
            !mark())
            return MOE_ERR_CUDA;
    }
    if (launch_combine_rows(z, row_map, at<int32_t>(ws, L.tok_rows), at<int32_t>(ws, L.tok_n), T,
                            E, d, R, reinterpret_cast<__nv_bfloat16 *>(Y), st) != cudaSuccess ||
        !mark())
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status_t moe_forward_rounded(const moe_bf16 *X, const float *Wr, const float *bias,
                                 const moe_bf16 *W1, const moe_bf16 *W3, const moe_bf16 *W2, int T,
                                 int d, int E, int K, int n, int renorm, moe_bf16 *Y,
                                 int32_t *row_map_out, void *ws, size_t ws_bytes, void *stream) {
    return moe_forward_rounded_traced(X, Wr, bias, W1, W3, W2, T, d, E, K, n, renorm, Y,
                                      row_map_out, ws, ws_bytes, stream, nullptr, 0);
}

}  // extern "C"
