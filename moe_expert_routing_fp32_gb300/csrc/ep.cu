// ep.cu -- EP DoubleRouting, the steps local to one rank.
//
// "NPU HunyuanImage-3.0模型推理优化实践", "MoE EP优化": with expert
// parallelism each rank receives (token all_to_all) the rows other ranks
// routed to its experts, grouped by source rank and, within a rank, ordered
// by expert.  LocalRerouting reorders them by local expert for the grouped
// matmul; LocalFinalizeRerouting puts the expert outputs back in the
// received order for the return all_to_all.  Both are pure row moves.
//
// counts[r][e] = rows from source rank r for local expert e.  Received row s
// belongs to block b = (r, e) with src_off[b] <= s < src_off[b+1] (row-major
// prefix of counts) and goes to dst_off[b] + (s - src_off[b]), where
// dst_off[r][e] = offsets[e] + sum_{r' < r} counts[r'][e].  Every CTA builds
// both prefix tables in shared memory (ep * E_local <= 8192 entries), so no
// workspace is needed; a warp moves one row at a time with 16-byte accesses.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int EP_THREADS = 256;
constexpr int EP_MAX_BLOCKS = 8192;

__global__ void __launch_bounds__(EP_THREADS)
local_rerouting_kernel(const uint16_t *__restrict__ recv_x, const int32_t *__restrict__ counts,
                       int ep, int El, int R, int H, uint16_t *__restrict__ local_x,
                       int32_t *__restrict__ local_src, int32_t *__restrict__ local_counts,
                       int32_t *__restrict__ local_offsets, int32_t *dev_status) {
    extern __shared__ int sm[];
    const int nb = ep * El;
    int *src_off = sm;               // [nb + 1]
    int *dst_off = sm + nb + 1;      // [nb]
    int *e_off = dst_off + nb;       // [El + 1]
    __shared__ int s_warp[EP_THREADS / 32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_bad = 0;
    // ---- src_off: exclusive prefix of counts in (rank, expert) order
    const int per = (nb + EP_THREADS - 1) / EP_THREADS;
    const int b0 = tid * per, b1 = min(nb, b0 + per);
    int part = 0;
    for (int b = b0; b < b1; ++b) {
        const int c = counts[b];
        if (c < 0) s_bad = 1;
        part += c;
    }
    int inc = part;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < EP_THREADS / 32; ++w) {
            const int v = s_warp[w];
            s_warp[w] = run;
            run += v;
        }
    }
    __syncthreads();
    int run = inc - part + s_warp[warp];
    for (int b = b0; b < b1; ++b) {
        src_off[b] = run;
        run += counts[b];
    }
    if (b1 == nb && b0 < b1) src_off[nb] = run;
    if (nb == 0 && tid == 0) src_off[0] = 0;
    __syncthreads();
    // ---- per local expert: total rows (parallel column sums), then its first
    //      row (prefix over experts), then each source rank's first row
    for (int e = tid; e < El; e += EP_THREADS) {
        int c = 0;
        for (int r = 0; r < ep; ++r) c += counts[r * El + e];
        e_off[e + 1] = c;
    }
    __syncthreads();
    if (tid == 0) {
        e_off[0] = 0;
        for (int e = 0; e < El; ++e) e_off[e + 1] += e_off[e];
    }
    __syncthreads();
    for (int e = tid; e < El; e += EP_THREADS) {
        int d = e_off[e];
        for (int r = 0; r < ep; ++r) {
            dst_off[r * El + e] = d;
            d += counts[r * El + e];
        }
        if (blockIdx.x == 0) {
            local_counts[e] = e_off[e + 1] - e_off[e];
            local_offsets[e] = e_off[e];
        }
    }
    if (blockIdx.x == 0 && tid == 0) local_offsets[El] = e_off[El];
    __syncthreads();
    const int total = src_off[nb];
    if (s_bad || total > R) {
        if (blockIdx.x == 0 && tid == 0) report(dev_status, MOE_DEV_BAD_OFFSETS);
        return;
    }
    // ---- move rows: warp per received row
    const int nvec = H / 8;
    for (int s = blockIdx.x * (EP_THREADS / 32) + warp; s < R; s += gridDim.x * (EP_THREADS / 32)) {
        if (s >= total) {
            if (lane == 0) local_src[s] = -1;    // rows past the received ones
            continue;
        }
        int lo = 0, hi = nb - 1;                 // last block whose start <= s
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (src_off[mid] <= s)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int d = dst_off[lo] + (s - src_off[lo]);
        if (lane == 0) local_src[d] = s;
        if (local_x) {
            const uint4 *src = reinterpret_cast<const uint4 *>(recv_x + static_cast<size_t>(s) * H);
            uint4 *dst = reinterpret_cast<uint4 *>(local_x + static_cast<size_t>(d) * H);
            for (int v = lane; v < nvec; v += 32) dst[v] = src[v];
        }
    }
}

__global__ void __launch_bounds__(EP_THREADS)
local_finalize_kernel(const uint16_t *__restrict__ local_y, const int32_t *__restrict__ local_src,
                      int R, int H, uint16_t *__restrict__ recv_y) {
    const int lane = threadIdx.x & 31;
    const int nvec = H / 8;
    for (int d = blockIdx.x * (EP_THREADS / 32) + (threadIdx.x >> 5); d < R;
         d += gridDim.x * (EP_THREADS / 32)) {
        const int s = local_src[d];
        if (s < 0 || s >= R) continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(local_y + static_cast<size_t>(d) * H);
        uint4 *dst = reinterpret_cast<uint4 *>(recv_y + static_cast<size_t>(s) * H);
        for (int v = lane; v < nvec; v += 32) dst[v] = src[v];
    }
}

int ep_grid(int R) {
    const int64_t want = ceil_div(R, EP_THREADS / 32);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, num_sms() * 8)));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_local_rerouting(const moe_bf16_t *recv_x, const int32_t *recv_counts,
                                            int32_t ep_size, int32_t E_local, int32_t R,
                                            int32_t H, moe_bf16_t *local_x, int32_t *local_src,
                                            int32_t *local_counts, int32_t *local_offsets,
                                            int32_t *dev_status, moe_stream_t stream) {
    if (ep_size <= 0 || E_local <= 0 || R < 0 || H < 0) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(ep_size) * E_local > EP_MAX_BLOCKS) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!recv_counts || !local_counts || !local_offsets || (R > 0 && !local_src))
        return MOE_ERR_INVALID_ARG;
    if (local_x) {
        if (!recv_x || H <= 0) return MOE_ERR_INVALID_ARG;
        if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        if ((reinterpret_cast<uintptr_t>(recv_x) | reinterpret_cast<uintptr_t>(local_x)) & 15u)
            return MOE_ERR_INVALID_ARG;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_DEVICE;
    }
    const int nb = ep_size * E_local;
    const size_t smem = (2 * static_cast<size_t>(nb) + 1 + E_local + 1) * sizeof(int);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(local_rerouting_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return MOE_ERR_CUDA;
    local_rerouting_kernel<<<ep_grid(R), EP_THREADS, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
        recv_x, recv_counts, ep_size, E_local, R, H, local_x, local_src, local_counts,
        local_offsets, dev_status);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_local_finalize_rerouting(const moe_bf16_t *local_y,
                                                     const int32_t *local_src, int32_t R,
                                                     int32_t H, moe_bf16_t *recv_y,
                                                     moe_stream_t stream) {
    if (R < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (R == 0) return MOE_OK;
    if (!local_y || !local_src || !recv_y) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(local_y) | reinterpret_cast<uintptr_t>(recv_y)) & 15u)
        return MOE_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_NO_DEVICE;
    }
    local_finalize_kernel<<<ep_grid(R), EP_THREADS, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        local_y, local_src, R, H, recv_y);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
