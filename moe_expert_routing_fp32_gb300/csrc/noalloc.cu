// noalloc.cu -- moe_init_routing_noalloc: init_routing without a caller
// workspace.
//
// Some callers cannot hand the library a scratch buffer: code that runs
// where no allocator is reachable (a plugin or runtime hook that only gets
// input and output pointers, a process whose memory pool is owned by
// someone else, or a context where calling cudaMalloc would synchronise the
// device or is simply not allowed).  For them this entry point keeps the
// routing histogram in a fixed array that lives in the library itself:
// kNoAllocScratchInts int32 values (1 MiB), reserved on every GPU that loads
// the library until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The host cannot use the array's name as a device address (on the host it
// only names a stand-in object), so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current and
// remembers it; later calls reuse it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchInts = 262144;   // 1 MiB of int32
constexpr int kMaxDev = 64;

static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

struct ScratchSlot {
    std::once_flag once;
    int32_t *ptr = nullptr;
    cudaError_t err = cudaSuccess;
};

ScratchSlot g_slots[kMaxDev];

// Device address of g_route_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(int32_t **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
    }
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    ScratchSlot &s = g_slots[dev];
    std::call_once(s.once, [&s] {
        void *p = nullptr;
        s.err = cudaGetSymbolAddress(&p, g_route_scratch);
        if (s.err == cudaSuccess)
            s.ptr = static_cast<int32_t *>(p);
        else
            cudaGetLastError();   // leave no error pending for later launches
    });
    if (s.err != cudaSuccess) return s.err;
    *out = s.ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_init_routing_noalloc(
    const int32_t *topk_idx, const moe_bf16_t *x, int32_t T, int32_t H, int32_t E, int32_t k,
    moe_bf16_t *expanded_x, int32_t *expanded_row_idx, int32_t *src_token,
    int32_t *sorted_expert_ids, int32_t *counts, int32_t *offsets, int32_t *dev_status,
    moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || E <= 0 || k <= 0 || H < 0) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(T) * k >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !expanded_row_idx || !src_token)) return MOE_ERR_INVALID_ARG;
    if (expanded_x) {
        if (!x || H <= 0) return MOE_ERR_INVALID_ARG;
        if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(expanded_x)) & 15u)
            return MOE_ERR_INVALID_ARG;
    }
    // the histogram needs ceil(T/32) * E entries of the built-in array
    const int B = static_cast<int>(ceil_div(T, kChunkTokens));
    if (static_cast<size_t>(B) * static_cast<size_t>(E) > kNoAllocScratchInts)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;   // cached per device
    int32_t *hist = nullptr;
    if (scratch_for_current_device(&hist) != cudaSuccess) return MOE_ERR_CUDA;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    // Every histogram entry that is read below is written first (by the
    // histogram kernel, or by the scan when it counts few tokens itself), so
    // the array needs no clearing between calls.
    const bool scan_hist = scan_builds_hist(T, E);
    if ((!scan_hist && launch_route_hist(topk_idx, T, k, E, hist, dev_status, s) != cudaSuccess) ||
        launch_route_scan(hist, B, E, counts, offsets, scan_hist ? topk_idx : nullptr, T, k,
                          dev_status, s) != cudaSuccess ||
        launch_route_scatter(topk_idx, hist, T, k, E, expanded_row_idx, src_token,
                             sorted_expert_ids, dev_status, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (expanded_x &&
        launch_permute(x, expanded_row_idx, T, H, k, expanded_x, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
