// routing.cu -- init_routing, compute_expert_tokens and finalize_routing.
//
// "NPU HunyuanImage-3.0模型推理优化实践", "GMM使能&&Routing优化":
// init_routing sorts the tokens by expert, compute_expert_tokens gives each
// expert's token count, finalize_routing puts the expert outputs back in
// token order and forms the weighted sum.
//
// init_routing is a stable counting sort of the T*k assignments
// (a = t*k + j) by expert, in three steps over chunks of 32 tokens (the same
// chunks the router uses, so the router can emit the histogram itself):
//   hist:    per-chunk expert histogram (shared-memory atomics; counts only;
//            up to 512 tokens the scan's CTA counts it itself)
//   scan:    per expert, an exclusive scan over chunks -> each chunk's first
//            row per expert; counts and offsets
//   scatter: each chunk ranks its assignments within an expert in order of a
//            (warp match + per-warp counts), so rows are stable in a.
// The data movement (expanded_x[row] = x[token]) is a separate pass that
// reads each token row once and writes its k copies with 16-byte accesses.
// finalize gathers the k rows of a token and sums them in slot order in
// fp32, the shared-expert row last: deterministic, no atomics.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kScatterThreads = 256;

__global__ void __launch_bounds__(256)
route_hist_kernel(const int32_t *__restrict__ topk_idx, int T, int k, int E,
                  int32_t *__restrict__ hist, int32_t *dev_status) {
    extern __shared__ int s_hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int64_t N = static_cast<int64_t>(T) * k;
    const int64_t a0 = static_cast<int64_t>(blockIdx.x) * kChunkTokens * k;
    const int64_t a1_ = a0 + static_cast<int64_t>(kChunkTokens) * k;
    const int64_t a1 = a1_ < N ? a1_ : N;
    for (int64_t a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
        const int e = topk_idx[a];
        if (e >= 0 && e < E)
            atomicAdd(&s_hist[e], 1);
        else
            report(dev_status, MOE_DEV_BAD_EXPERT_ID);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        hist[static_cast<size_t>(blockIdx.x) * E + e] = s_hist[e];
}

// One CTA of 1024 threads (E <= 1024).  Thread (s, e) owns expert e's column
// of the [B][E] histogram over the chunk segment s.  Given topk_idx (few
// tokens), the CTA first counts the histogram in shared memory and stores it.
__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t *__restrict__ hist, int B, int E, int32_t *__restrict__ counts,
                  int32_t *__restrict__ offsets, const int32_t *__restrict__ topk_idx, int T,
                  int k, int32_t *dev_status) {
    __shared__ int s_seg[1024];
    __shared__ int s_cnt[1024];
    __shared__ int s_warp[32];
    extern __shared__ int s_hist[];   // [B][E], with topk_idx
    const int tid = threadIdx.x;
    if (topk_idx) {
        for (int i = tid; i < B * E; i += blockDim.x) s_hist[i] = 0;
        __syncthreads();
        const int n = T * k;
        for (int a = tid; a < n; a += blockDim.x) {
            const int e = topk_idx[a];
            if (e >= 0 && e < E)
                atomicAdd(&s_hist[(a / k) / kChunkTokens * E + e], 1);
            else
                report(dev_status, MOE_DEV_BAD_EXPERT_ID);
        }
        __syncthreads();
        for (int i = tid; i < B * E; i += blockDim.x) hist[i] = s_hist[i];
        __syncthreads();
    }
    const int S = 1024 / E;                  // segments per expert
    const int L = (B + S - 1) / S;           // chunks per segment
    const int e = tid % E;
    const int s = tid / E;
    const bool active = s < S;
    int sum = 0;
    if (active) {
        const int b1 = min(B, (s + 1) * L);
        for (int b = s * L; b < b1; ++b) sum += hist[static_cast<size_t>(b) * E + e];
    }
    s_seg[tid] = sum;
    __syncthreads();
    // exclusive prefix over the segments of each expert, and the totals
    if (tid < E) {
        int run = 0;
        for (int q = 0; q < S; ++q) {
            const int v = s_seg[q * E + tid];
            s_seg[q * E + tid] = run;
            run += v;
        }
        s_cnt[tid] = run;
        counts[tid] = run;
    }
    __syncthreads();
    // exclusive scan of the totals over experts (block-wide)
    const int lane = tid & 31, warp = tid >> 5;
    const int v = tid < E ? s_cnt[tid] : 0;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int w = s_warp[lane];
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        s_warp[lane] = wi - w;   // exclusive
    }
    __syncthreads();
    const int excl = inc - v + s_warp[warp];
    if (tid < E) {
        s_cnt[tid] = excl;
        offsets[tid] = excl;
        if (tid == E - 1) offsets[E] = excl + v;
    }
    __syncthreads();
    // rewrite the histogram as per-chunk first rows
    if (active) {
        int run = s_cnt[e] + s_seg[tid];
        const int b1 = min(B, (s + 1) * L);
        for (int b = s * L; b < b1; ++b) {
            const size_t i = static_cast<size_t>(b) * E + e;
            const int c = hist[i];
            hist[i] = run;
            run += c;
        }
    }
}

__global__ void __launch_bounds__(kScatterThreads)
route_scatter_kernel(const int32_t *__restrict__ topk_idx, const int32_t *__restrict__ base,
                     int T, int k, int E, int32_t *__restrict__ row_idx,
                     int32_t *__restrict__ src_token, int32_t *__restrict__ sorted_ids,
                     int32_t *dev_status) {
    constexpr int NW = kScatterThreads / 32;
    extern __shared__ int smem[];
    int *s_wc = smem;                 // [NW][E] per-warp counts of the current sub-chunk
    int *s_run = smem + NW * E;       // [E] rows already given out in this chunk
    int *s_base = s_run + E;          // [E] first row of this chunk per expert
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < NW * E; i += kScatterThreads) s_wc[i] = 0;
    for (int e = tid; e < E; e += kScatterThreads) {
        s_run[e] = 0;
        s_base[e] = base[static_cast<size_t>(blockIdx.x) * E + e];
    }
    __syncthreads();
    const int64_t N = static_cast<int64_t>(T) * k;
    const int64_t a0 = static_cast<int64_t>(blockIdx.x) * kChunkTokens * k;
    const int64_t a1_ = a0 + static_cast<int64_t>(kChunkTokens) * k;
    const int64_t a1 = a1_ < N ? a1_ : N;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int64_t sub = a0; sub < a1; sub += kScatterThreads) {
        const int64_t a = sub + tid;
        int e = -1;
        if (a < a1) {
            e = topk_idx[a];
            if (e < 0 || e >= E) {
                report(dev_status, MOE_DEV_BAD_EXPERT_ID);
                row_idx[a] = -1;
                e = -1;
            }
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        const int cnt = __popc(peers);
        const bool leader = (__ffs(peers) - 1) == lane;
        if (e >= 0 && leader) s_wc[warp * E + e] = cnt;
        __syncthreads();
        if (e >= 0) {
            int pre = s_run[e] + rank;
            for (int w = 0; w < warp; ++w) pre += s_wc[w * E + e];
            const int row = s_base[e] + pre;
            row_idx[a] = row;
            if (src_token) src_token[row] = static_cast<int32_t>(a / k);
            if (sorted_ids) sorted_ids[row] = e;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&s_run[e], cnt);
            s_wc[warp * E + e] = 0;
        }
        __syncthreads();
    }
}

// expanded_x[row_idx[t*k + j]] = xs[t] for every slot j: each token row is
// read once (16-byte loads) and written k times.
__global__ void __launch_bounds__(128)
permute_kernel(const uint16_t *__restrict__ xs, const int32_t *__restrict__ row_idx, int T,
               int H, int k, uint16_t *__restrict__ expanded_x) {
    const int nvec = H / 8;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(xs + static_cast<size_t>(t) * H);
        for (int v0 = 0; v0 < nvec; v0 += 4 * blockDim.x) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * blockDim.x + threadIdx.x;
                if (v < nvec) q[u] = src[v];
            }
            for (int j = 0; j < k; ++j) {
                const int row = row_idx[static_cast<size_t>(t) * k + j];
                if (row < 0) continue;
                uint4 *dst = reinterpret_cast<uint4 *>(expanded_x + static_cast<size_t>(row) * H);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + u * blockDim.x + threadIdx.x;
                    if (v < nvec) __stcs(dst + v, q[u]);   // streamed: read once, later
                }
            }
        }
    }
}

__device__ __forceinline__ int lower_bound_ids(const int32_t *ids, int n, int key) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ids[mid] < key)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Thread i checks that ids[i] <= ids[i+1] and that ids[i] is a valid expert;
// thread e <= E finds where expert e's rows start (binary search).
__global__ void __launch_bounds__(256)
expert_tokens_kernel(const int32_t *__restrict__ ids, int n, int E, int32_t *__restrict__ counts,
                     int32_t *__restrict__ offsets, int32_t *dev_status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const int v = ids[i];
        if (v < 0 || v >= E) report(dev_status, MOE_DEV_BAD_EXPERT_ID);
        if (i + 1 < n && ids[i + 1] < v) report(dev_status, MOE_DEV_UNSORTED);
    }
    if (i <= E) {
        const int lo = lower_bound_ids(ids, n, i);
        offsets[i] = i == E ? n : lo;
        if (i < E) counts[i] = lower_bound_ids(ids, n, i + 1) - lo;
    }
}

// out[t] = sum_j w[t,j] * y_exp[row_idx[t*k+j]] (+ shared[t]), fp32 in slot
// order.  The token's k row indices and weights are read once into shared
// memory; a lane then issues the loads of 8 slots' 16-byte pieces before it
// accumulates them (in slot order).  blockIdx.y splits the row's columns
// when there are few tokens.
// Y_F32: the routed rows are fp32 (the down matmul's unrounded accumulator)
template <bool Y_F32, bool SHARED_F32, bool OUT_F32>
__global__ void __launch_bounds__(128)
finalize_kernel(const void *__restrict__ y_exp, const int32_t *__restrict__ row_idx,
                const float *__restrict__ topk_w, const void *__restrict__ shared, int T, int H,
                int k, void *__restrict__ out) {
    __shared__ int s_row[32];
    __shared__ float s_w[32];
    const int nvec = H / 8;
    const int vchunk = (nvec + gridDim.y - 1) / gridDim.y;
    const int v0 = blockIdx.y * vchunk;
    const int v1 = min(nvec, v0 + vchunk);
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();                       // the previous token's slots are consumed
        if (threadIdx.x < k) {
            s_row[threadIdx.x] = row_idx[static_cast<size_t>(t) * k + threadIdx.x];
            s_w[threadIdx.x] = topk_w[static_cast<size_t>(t) * k + threadIdx.x];
        }
        __syncthreads();
        for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            for (int j0 = 0; j0 < k; j0 += 8) {
                if (Y_F32) {
                    // eight slots' loads in flight, then the sums in slot order
                    float4 qa[8], qb[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u;
                        const int row = j < k ? s_row[j] : -1;
                        if (row >= 0) {
                            const float4 *src = reinterpret_cast<const float4 *>(
                                static_cast<const float *>(y_exp) + static_cast<size_t>(row) * H);
                            qa[u] = __ldg(src + 2 * v);
                            qb[u] = __ldg(src + 2 * v + 1);
                        } else {
                            qa[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            qb[u] = qa[u];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u;
                        if (j >= k || s_row[j] < 0) continue;
                        const float w = s_w[j];
                        acc[0] = __fmaf_rn(w, qa[u].x, acc[0]);
                        acc[1] = __fmaf_rn(w, qa[u].y, acc[1]);
                        acc[2] = __fmaf_rn(w, qa[u].z, acc[2]);
                        acc[3] = __fmaf_rn(w, qa[u].w, acc[3]);
                        acc[4] = __fmaf_rn(w, qb[u].x, acc[4]);
                        acc[5] = __fmaf_rn(w, qb[u].y, acc[5]);
                        acc[6] = __fmaf_rn(w, qb[u].z, acc[6]);
                        acc[7] = __fmaf_rn(w, qb[u].w, acc[7]);
                    }
                } else {
                    uint4 q[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u;
                        const int row = j < k ? s_row[j] : -1;
                        q[u] = row >= 0
                                   ? __ldg(reinterpret_cast<const uint4 *>(
                                               static_cast<const uint16_t *>(y_exp) +
                                               static_cast<size_t>(row) * H) + v)
                                   : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u;
                        if (j >= k || s_row[j] < 0) continue;
                        const float w = s_w[j];
                        const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[2 * i] = __fmaf_rn(w, __uint_as_float(wd[i] << 16), acc[2 * i]);
                            acc[2 * i + 1] =
                                __fmaf_rn(w, __uint_as_float(wd[i] & 0xFFFF0000u), acc[2 * i + 1]);
                        }
                    }
                }
            }
            if (shared) {
                if (SHARED_F32) {
                    const float4 *sp = reinterpret_cast<const float4 *>(
                        static_cast<const float *>(shared) + static_cast<size_t>(t) * H);
                    const float4 s0 = sp[2 * v], s1 = sp[2 * v + 1];
                    acc[0] += s0.x; acc[1] += s0.y; acc[2] += s0.z; acc[3] += s0.w;
                    acc[4] += s1.x; acc[5] += s1.y; acc[6] += s1.z; acc[7] += s1.w;
                } else {
                    const uint4 q = reinterpret_cast<const uint4 *>(
                        static_cast<const uint16_t *>(shared) + static_cast<size_t>(t) * H)[v];
                    const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] += __uint_as_float(wd[i] << 16);
                        acc[2 * i + 1] += __uint_as_float(wd[i] & 0xFFFF0000u);
                    }
                }
            }
            if (OUT_F32) {
                float4 *op = reinterpret_cast<float4 *>(static_cast<float *>(out) +
                                                        static_cast<size_t>(t) * H);
                op[2 * v] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                op[2 * v + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            } else {
                uint4 *op = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) +
                                                      static_cast<size_t>(t) * H);
                op[v] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            }
        }
    }
}

int grid_for_rows(int rows, int per_sm) {
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(rows, num_sms() * per_sm)));
}

}  // namespace

cudaError_t launch_route_hist(const int32_t *topk_idx, int T, int k, int E, int32_t *hist,
                              int32_t *dev_status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int B = static_cast<int>(ceil_div(T, kChunkTokens));
    route_hist_kernel<<<B, 256, E * sizeof(int), stream>>>(topk_idx, T, k, E, hist, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_route_scan(int32_t *hist, int B, int E, int32_t *counts, int32_t *offsets,
                              const int32_t *topk_idx, int T, int k, int32_t *dev_status,
                              cudaStream_t stream) {
    if (topk_idx && !scan_builds_hist(T, E)) return cudaErrorInvalidValue;
    const size_t smem = topk_idx ? static_cast<size_t>(B) * E * sizeof(int) : 0;
    route_scan_kernel<<<1, 1024, smem, stream>>>(hist, B, E, counts, offsets, topk_idx, T, k,
                                                 dev_status);
    return cudaGetLastError();
}

cudaError_t launch_route_scatter(const int32_t *topk_idx, const int32_t *base, int T, int k,
                                 int E, int32_t *row_idx, int32_t *src_token,
                                 int32_t *sorted_ids, int32_t *dev_status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int B = static_cast<int>(ceil_div(T, kChunkTokens));
    const size_t smem = (kScatterThreads / 32 + 2) * static_cast<size_t>(E) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(route_scatter_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    route_scatter_kernel<<<B, kScatterThreads, smem, stream>>>(topk_idx, base, T, k, E, row_idx,
                                                               src_token, sorted_ids, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_permute(const uint16_t *xs, const int32_t *row_idx, int T, int H, int k,
                           uint16_t *expanded_x, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    permute_kernel<<<grid_for_rows(T, 16), 128, 0, stream>>>(xs, row_idx, T, H, k, expanded_x);
    return cudaGetLastError();
}

cudaError_t launch_expert_tokens(const int32_t *ids, int n, int E, int32_t *counts,
                                 int32_t *offsets, int32_t *dev_status, cudaStream_t stream) {
    const int64_t work = std::max<int64_t>(n, E + 1);
    expert_tokens_kernel<<<static_cast<int>(ceil_div(work, 256)), 256, 0, stream>>>(
        ids, n, E, counts, offsets, dev_status);
    return cudaGetLastError();
}

template <bool Y_F32>
void launch_finalize_t(const void *y_exp, const int32_t *row_idx, const float *topk_w,
                       const void *shared, bool shared_f32, int T, int H, int k, void *out,
                       bool out_f32, dim3 grid, cudaStream_t stream) {
    if (shared_f32 && out_f32)
        finalize_kernel<Y_F32, true, true><<<grid, 128, 0, stream>>>(y_exp, row_idx, topk_w,
                                                                     shared, T, H, k, out);
    else if (shared_f32)
        finalize_kernel<Y_F32, true, false><<<grid, 128, 0, stream>>>(y_exp, row_idx, topk_w,
                                                                      shared, T, H, k, out);
    else if (out_f32)
        finalize_kernel<Y_F32, false, true><<<grid, 128, 0, stream>>>(y_exp, row_idx, topk_w,
                                                                      shared, T, H, k, out);
    else
        finalize_kernel<Y_F32, false, false><<<grid, 128, 0, stream>>>(y_exp, row_idx, topk_w,
                                                                       shared, T, H, k, out);
}

cudaError_t launch_finalize(const void *y_exp, bool y_f32, const int32_t *row_idx,
                            const float *topk_w, const void *shared, bool shared_f32, int T,
                            int H, int k, void *out, bool out_f32, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    // few tokens: split each row's columns over blocks (>= 128 vectors each)
    // so that about two blocks per SM run
    const int nvec = H / 8;
    const int want = num_sms() * 2;
    const int ysplit = T >= want ? 1
                                 : static_cast<int>(std::max<int64_t>(
                                       1, std::min<int64_t>(ceil_div(want, T), nvec / 128)));
    const dim3 grid(static_cast<unsigned>(grid_for_rows(T, 16)), static_cast<unsigned>(ysplit));
    if (y_f32)
        launch_finalize_t<true>(y_exp, row_idx, topk_w, shared, shared_f32, T, H, k, out, out_f32,
                                grid, stream);
    else
        launch_finalize_t<false>(y_exp, row_idx, topk_w, shared, shared_f32, T, H, k, out,
                                 out_f32, grid, stream);
    return cudaGetLastError();
}

}  // namespace moe
