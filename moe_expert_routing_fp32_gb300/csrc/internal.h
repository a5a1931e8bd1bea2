// internal.h -- launchers shared between the libmoe translation units.
// Every launcher only enqueues work on `stream`; it returns the
// cudaGetLastError() of its launches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// tokens per routing chunk: the router's CTA and the routing kernels agree on it
constexpr int kChunkTokens = 32;
// largest E for which the router fuses top-k and the routing histogram
constexpr int kRouterExperts = 64;
// batches of at most this many tokens use the one-CTA-per-token router (the
// sequential fp32 gate); larger ones take the tensor-core gate unless the
// caller asks for the sequential one
constexpr int kGateSmallMaxT = 512;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int num_sms();  // of the current device (cached)
// whether the current device is of the sm_100 family (looked up once per
// device; a failed lookup leaves no CUDA error pending)
bool current_device_ok();

// ---- router.cu
// RMSNorm (optional) + fp32 gate.  If fuse_topk (requires E <= 64), also
// top-k/softmax into topk_idx/topk_w and the per-chunk expert histogram
// into hist[ceil(T/32)][E] (hist may be NULL).
cudaError_t launch_router(const uint16_t *x, const uint16_t *gamma, const float *wg,
                          const float *gate_bias, int T, int H, int E, float eps, bool rmsnorm,
                          uint16_t *xn, float *logits, bool fuse_topk, int k, bool renorm,
                          int32_t *topk_idx, float *topk_w, int32_t *hist,
                          int32_t *dev_status, cudaStream_t stream);

// output columns of the tensor-core gate's GEMM: the three parts of every
// expert's weights, padded to whole 128-column blocks
inline int gate_tc_cols(int E) { return static_cast<int>(ceil_div(3 * E, 128) * 128); }
// Tensor-core gate: RMSNorm alone (xn; H % 128 == 0), the exact three-way
// bf16 split of the gate weight (rows [0,E) part 1, [E,2E) part 2, [2E,3E)
// part 3, zero rows up to NW), and the combine of the three partial logits:
// with fuse_topk and E <= kRouterExperts the top-k and the chunk histograms
// (logits not written), else the logits.
cudaError_t launch_rmsnorm(const uint16_t *x, const uint16_t *gamma, int T, int H, float eps,
                           uint16_t *xn, int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_gate_split(const float *wg, int E, int H, uint16_t *wsplit, int NW,
                              cudaStream_t stream);
// RMSNorm's sum of squares of each row: the exact sum rounded once to fp32
cudaError_t launch_sumsq(const uint16_t *x, int T, int H, float *ss, cudaStream_t stream);
cudaError_t launch_gate_combine(const float *parts, int NW, int T, int E, const float *gate_bias,
                                float *logits, bool fuse_topk, int k, bool renorm,
                                int32_t *topk_idx, float *topk_w, int32_t *hist,
                                cudaStream_t stream);
cudaError_t launch_topk(const float *logits, int T, int E, int k, bool renorm,
                        int32_t *topk_idx, float *topk_w, cudaStream_t stream);

// ---- routing.cu
cudaError_t launch_route_hist(const int32_t *topk_idx, int T, int k, int E, int32_t *hist,
                              int32_t *dev_status, cudaStream_t stream);
// hist [B][E] -> in place per-chunk row bases; counts [E]; offsets [E+1].
// Given topk_idx ([T, k], B = ceil(T/32)), the scan's CTA first counts the
// histogram itself (scan_builds_hist(T, E) must hold); else hist holds it.
cudaError_t launch_route_scan(int32_t *hist, int B, int E, int32_t *counts, int32_t *offsets,
                              const int32_t *topk_idx, int T, int k, int32_t *dev_status,
                              cudaStream_t stream);
// few tokens: one CTA counts the histogram faster than a launch of its own
// (at most 32 KB of it, within the default 48 KB of shared memory)
inline bool scan_builds_hist(int T, int E) {
    return T <= kGateSmallMaxT && ceil_div(T, kChunkTokens) * E <= 8 * 1024;
}
cudaError_t launch_route_scatter(const int32_t *topk_idx, const int32_t *base, int T, int k,
                                 int E, int32_t *row_idx, int32_t *src_token,
                                 int32_t *sorted_ids, int32_t *dev_status, cudaStream_t stream);
cudaError_t launch_permute(const uint16_t *xs, const int32_t *row_idx, int T, int H, int k,
                           uint16_t *expanded_x, cudaStream_t stream);
cudaError_t launch_expert_tokens(const int32_t *ids, int n, int E, int32_t *counts,
                                 int32_t *offsets, int32_t *dev_status, cudaStream_t stream);
// y_exp is bf16, or fp32 with y_f32 (the routed rows kept at the matmul's
// accumulator precision)
cudaError_t launch_finalize(const void *y_exp, bool y_f32, const int32_t *row_idx,
                            const float *topk_w, const void *shared, bool shared_f32, int T,
                            int H, int k, void *out, bool out_f32, cudaStream_t stream);

// ---- gemm.cu
struct GemmSegment1 {       // an optional dense problem appended to the grouped one
    const uint16_t *A;      // [rows, K1]
    const uint16_t *B;      // SwiGLU: [2*N1, K1]; store: [N1, K1]
    int rows = 0;           // 0 = absent
    int K1 = 0;
    int N1 = 0;             // SwiGLU: I_s (act columns); store: output columns
    void *out = nullptr;    // [rows, N1] bf16 (or fp32 with out_f32)
    bool out_f32 = false;
};

// G may be 0 (segment 1 only; `offsets` must still point at one readable int).
// act[r, :] = bf16(SiLU(A W13g^T) * (A W13u^T)) per group; A [n, K], W13 [G, 2N, K]
// With gather_src, A is not read: routed row r is row gather_rows[r] of
// gather_src ([gather_n, K]), copied in by the kernel itself (only where
// gemm_can_gather holds: the wide pair kernel's shapes).
cudaError_t launch_gemm_swiglu(const uint16_t *A, const int32_t *offsets, int G, int n, int K,
                               const uint16_t *W13, int N, uint16_t *act,
                               const GemmSegment1 &seg1, int32_t *dev_status,
                               cudaStream_t stream, const uint16_t *gather_src = nullptr,
                               const int32_t *gather_rows = nullptr, int gather_n = 0);
bool gemm_can_gather(int n, int G, int K, int N, const GemmSegment1 &seg1);
// y[r, :] = bf16(A W^T) per group (fp32, unrounded, with y_f32); A [n, K], W [G, N, K]
cudaError_t launch_gemm_store(const uint16_t *A, const int32_t *offsets, int G, int n, int K,
                              const uint16_t *W, int N, void *y, const GemmSegment1 &seg1,
                              int32_t *dev_status, cudaStream_t stream, bool y_f32 = false);
bool tensor_maps_available();

}  // namespace moe
