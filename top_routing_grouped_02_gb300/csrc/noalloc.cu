// moe_permute_noalloc: the grouping step for callers that cannot allocate
// device memory. Its scratch lives in a fixed array compiled into this library
// instead of a caller-provided workspace.
//
// Who needs it: code that is handed only its inputs and outputs and may not
// call cudaMalloc itself, e.g. a plugin inside an inference engine that owns
// every byte of device memory, or a serving loop whose memory was planned at
// start-up (cudaMalloc can synchronise the device and can fail once memory is
// fragmented, so such loops forbid it).
#include <stdint.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

// Capacity of the built-in scratch. Every GPU that loads libmoe.so holds this
// array until the process exits.
constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

// Device address of g_permute_scratch per device, looked up with that device
// current. In host code the symbol is only a host-side stand-in, so the kernels
// must be given this address. The address belongs to the CUDA context it was
// looked up in: each entry remembers that context's unique id (never reused,
// unlike a context handle), so after cudaDeviceReset or under another context
// the lookup runs again instead of handing out a stale address. A mutex per
// device serialises host threads.
struct ScratchSlot {
    std::mutex m;
    unsigned long long ctx_id = 0;
    void *addr = nullptr;
};
ScratchSlot g_slots[64];

moe_status_t scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    ScratchSlot &slot = g_slots[dev];
    std::lock_guard<std::mutex> lock(slot.m);
    unsigned long long id = 0;
    bool known = current_context_id(&id);
    if (known && slot.addr != nullptr && slot.ctx_id == id) {
        *out = slot.addr;
        return MOE_OK;
    }
    // first use in this context: the lookup also loads this part of the library
    // (and its array) onto the device under lazy module loading
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr)
        return MOE_ERR_CUDA;
    if (!known) known = current_context_id(&id);  // the lookup made the context current
    slot.addr = known ? p : nullptr;              // cache only under a known context
    slot.ctx_id = known ? id : 0;
    *out = p;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_noalloc(const int32_t *topk_idx, const int32_t *counts, int T,
                                            int E, int K, int32_t *offsets, int32_t *perm_token,
                                            int32_t *perm_slot, int32_t *row_of_slot,
                                            int32_t *tiles, int32_t *num_tiles, void *stream) {
    if (!topk_idx || !offsets || !perm_token || !perm_slot || !row_of_slot || !tiles || !num_tiles)
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || K < 1) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || K > kMaxK || K > E || (int64_t)T * K >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(tiles) & 15u) != 0) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, 0, E, K, 0);
    if (L.grouping_end > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;  // beyond the built-in scratch
    moe_status_t s = check_arch();
    if (s != MOE_OK) return s;
    void *scratch = nullptr;
    if ((s = scratch_for_current_device(&scratch)) != MOE_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the control words (error word, completion ticket) must start at zero
    if (cudaMemsetAsync(static_cast<char *>(scratch) + L.err, 0, 64, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    // (three kernels: the one-kernel grouping's call tags live in the control
    // words, which this call clears every time)
    if (launch_permute(topk_idx, counts, T, E, K, offsets, perm_token, perm_slot, row_of_slot,
                       tiles, num_tiles, L, static_cast<char *>(scratch), st,
                       /*one_kernel=*/false) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
