/*
 * moe.h -- C ABI of libmoe, a single-GPU (sm_103a) Mixture-of-Experts
 * feed-forward layer.
 *
 * The layer is the one described on "NPU HunyuanImage-3.0模型推理优化实践"
 * (HunyuanImage-3.0 inference on Ascend, cf-1.com/news/2296994):
 *   RMSNorm ("RmsNorm算子优化") -> fp32 gate ("消除gate计算冗余cast算子")
 *   -> GatingTopK ("MoE EP优化") -> init_routing / compute_expert_tokens
 *   ("GMM使能&&Routing优化") -> grouped matmul over the merged gate/up weight
 *   w13 with SwiGLU ("MoE TP优化 / 计算分解") -> grouped down matmul
 *   -> finalize_routing ("GMM使能&&Routing优化"), plus an optional shared
 *   expert ("MoE多流并行优化").
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer into memory the caller owns.
 *     The library never allocates, frees or synchronises: each call only
 *     enqueues kernels on `stream` (NULL = the legacy default stream) and
 *     returns.  Outputs are valid once the caller has synchronised.
 *   - All tensors are dense, row-major, contiguous.  bf16 values are passed
 *     as their 16-bit patterns (moe_bf16_t).  Unless stated otherwise every
 *     pointer must be 16-byte aligned.
 *   - The return value reports host-side argument checks and launch errors;
 *     nothing is enqueued when it is not MOE_OK.  Errors that only the
 *     device can see are OR-ed as MOE_DEV_* bits into *dev_status (a device
 *     int32 the caller zeroes beforehand; NULL = not reported).  A kernel
 *     that detects one writes nothing out of bounds and returns early; the
 *     outputs of that call are then undefined.
 *   - Sizes: 1 <= k <= min(E, 32), E <= 1024, T*k < 2^31, H % 64 == 0
 *     (H % 128 == 0 for the grouped MLP and the layer), I % 128 == 0
 *     (I_shared likewise).  Inputs must be finite.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t;            /* bfloat16 bit pattern */
typedef struct CUstream_st *moe_stream_t; /* the same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* null pointer, bad size or misalignment */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* sizes outside the limits above */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,
    MOE_ERR_CUDA = 4,               /* a CUDA runtime/launch error */
    MOE_ERR_NO_DEVICE = 5           /* no sm_100-family GPU is current */
} moe_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
    MOE_DEV_BAD_EXPERT_ID = 1,      /* an expert id outside [0, E) */
    MOE_DEV_TIMEOUT = 2,            /* a pipeline wait ran past its limit */
    MOE_DEV_BAD_OFFSETS = 4,        /* group offsets not monotone / out of range */
    MOE_DEV_UNSORTED = 8            /* moe_expert_tokens input not sorted */
};

/* flags */
enum {
    MOE_RENORM = 1u << 0,      /* renormalise the top-k weights to sum 1 */
    MOE_RMSNORM = 1u << 1,     /* RMSNorm before the gate */
    MOE_SHARED = 1u << 2,      /* add the shared expert */
    MOE_OUT_F32 = 1u << 3,     /* layer / finalize output in fp32 (else bf16) */
    MOE_SHARED_F32 = 1u << 4,  /* finalize: `shared` is fp32 (else bf16) */
    MOE_GATE_SEQUENTIAL = 1u << 5, /* layer: the sequential fp32 gate for every T
                                      (see moe_gate_tensor for the default) */
    MOE_Y_F32 = 1u << 6,           /* layer: keep the routed expert outputs y_exp in
                                      fp32, the down matmul's accumulator, instead of
                                      rounding them to bf16 (finalize: y_exp is fp32) */
    MOE_GATHER_A = 1u << 7         /* layer: no permute pass; the routed w13 matmul
                                      reads each expanded row from the (normalised)
                                      input by its source token, and the workspace
                                      holds no expanded_x.  Takes effect only where
                                      that matmul runs as the 256 x 512 pair kernel
                                      (>= 1024 rows per expert on average,
                                      I % 256 == 0); ignored elsewhere.  Same results
                                      bit for bit: the rows are copies either way.
                                      Off by default: the in-kernel row copies make
                                      the matmul slower than the permute pass costs. */
};

typedef struct {
    int32_t T;          /* tokens */
    int32_t H;          /* hidden size */
    int32_t E;          /* routed experts */
    int32_t k;          /* experts per token */
    int32_t I;          /* routed expert intermediate size */
    int32_t I_shared;   /* shared expert intermediate size (MOE_SHARED) */
    float rms_eps;      /* RMSNorm epsilon (MOE_RMSNORM) */
    uint32_t flags;     /* MOE_RENORM | MOE_RMSNORM | MOE_SHARED | MOE_OUT_F32 |
                           MOE_GATE_SEQUENTIAL | MOE_Y_F32 */
} moe_desc_t;

/* Human-readable name of a moe_status_t value. */
const char *moe_status_string(int status);

/*
 * RMSNorm and fp32 gate ("RmsNorm算子优化"; "消除gate计算冗余cast算子":
 * the gate is an fp32 linear layer on the hidden states cast to float).
 *   x      [T, H] bf16
 *   gamma  [H] bf16, or NULL for all ones (used with MOE_RMSNORM only)
 *   wg     [E, H] fp32 gate weight
 *   gate_bias [E] fp32 per-expert logit offset, or NULL
 *   xn     [T, H] bf16 out: bf16((x * r) * gamma), r = 1/sqrt(ss/H + eps)
 *          in fp32, ss the row's sum of squares as moe_rmsnorm_sumsq gives
 *          it.  Required with MOE_RMSNORM, ignored (may be NULL) without it.
 *   logits [T, E] fp32 out: fp32 dot product of the (normalised) row with
 *          wg[e], one fused multiply-add per term in ascending h, plus
 *          gate_bias[e].  These are bit-identical to the same steps done
 *          sequentially on any IEEE fp32 machine.
 * flags: MOE_RMSNORM.  T may be 0.
 * With wg and logits both NULL (and MOE_RMSNORM) only xn is computed, by the
 * RMSNorm pass the layer runs ahead of the tensor-core gate (H % 128 == 0);
 * same bits as above.
 */
moe_status_t moe_rmsnorm_gate(const moe_bf16_t *x, const moe_bf16_t *gamma,
                              const float *wg, const float *gate_bias, int32_t T,
                              int32_t H, int32_t E, float eps, uint32_t flags,
                              moe_bf16_t *xn, float *logits, moe_stream_t stream);

/*
 * The RMSNorm's reduction ("RmsNorm算子优化"): per row, the exact sum of the
 * squares of its bf16 values rounded once to fp32 (nearest, ties to even;
 * fp32 subnormals and overflow to infinity included).  The value does not
 * depend on a summation order; every RMSNorm of this library uses it.
 *   x  [T, H] bf16 (16-byte aligned, H % 8 == 0);  ss [T] fp32 out
 * T may be 0.  A row holding an infinity or a NaN gives inf or NaN.
 */
moe_status_t moe_rmsnorm_sumsq(const moe_bf16_t *x, int32_t T, int32_t H, float *ss,
                               moe_stream_t stream);

/*
 * The same fp32 gate on the tensor cores ("消除gate计算冗余cast算子": an fp32
 * linear layer).  Every fp32 weight is split exactly into three bf16 parts,
 * wg = w1 + w2 + w3 (exact for |wg| >= 2^-110, within 2^-134 below); each
 * product of a bf16 xs value with a part is exact,
 * the grouped GEMM accumulates the three partial dot products in fp32 and a
 * combine kernel adds them, (p1 + p2) + p3, plus gate_bias[e].  The logits
 * are fp32-accurate but summed in another order than moe_rmsnorm_gate's, so
 * they may differ from it in the last bits (and a top-k decision between
 * two logits that close may differ).  moe_layer_forward uses this gate for
 * T > 512 unless MOE_GATE_SEQUENTIAL is set.
 *   xs     [T, H] bf16 in: the (already normalised) hidden states
 *   wg     [E, H] fp32 in;  gate_bias [E] fp32 or NULL
 *   logits [T, E] fp32 out
 * H % 128 == 0, E <= 1024.  T may be 0.  Workspace:
 * moe_gate_tensor_workspace_size() bytes, 256-byte aligned, caller-owned;
 * it starts with the split weight [NW, H] bf16 (NW = 3E rounded up to a
 * multiple of 128; rows [pE, (p+1)E) hold part p+1, the rest are zero),
 * followed (256-byte aligned) by the partial logits [T, NW] fp32.  A
 * device-side wait that runs out sets *dev_status (may be NULL).
 */
moe_status_t moe_gate_tensor_workspace_size(int32_t T, int32_t H, int32_t E, size_t *bytes);
moe_status_t moe_gate_tensor(const moe_bf16_t *xs, const float *wg, const float *gate_bias,
                             int32_t T, int32_t H, int32_t E, float *logits, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, moe_stream_t stream);

/*
 * GatingTopK ("MoE EP优化"): per token, the k largest logits (descending;
 * equal logits, -0 == +0, go to the lower expert index) and their softmax
 * probabilities, renormalised over the k chosen with MOE_RENORM.
 *   logits   [T, E] fp32 in
 *   topk_idx [T, k] int32 out (slot 0 = largest)
 *   topk_w   [T, k] fp32 out
 */
moe_status_t moe_gate_topk(const float *logits, int32_t T, int32_t E, int32_t k,
                           uint32_t flags, int32_t *topk_idx, float *topk_w,
                           moe_stream_t stream);

/*
 * init_routing ("GMM使能&&Routing优化": sort the tokens by expert).
 * Assignment a = t*k + j goes to expert topk_idx[a]; rows are ordered by
 * expert and, within an expert, by a (a stable counting sort):
 *   counts[e] = #assignments to e;  offsets[0..E] = exclusive scan, offsets[E] = T*k
 *   expanded_row_idx[a] = offsets[e] + #{a' < a : topk_idx[a'] == e}
 *   src_token[r]        = token of the assignment placed in row r
 *   sorted_expert_ids[r]= expert of row r (may be NULL)
 *   expanded_x[r]       = x[src_token[r]]  ([T*k, H] bf16; may be NULL
 *                         to build the indices only, then x may be NULL too)
 * Workspace: moe_init_routing_workspace_size() bytes, 256-byte aligned.
 * Bad expert ids set MOE_DEV_BAD_EXPERT_ID; those assignments get no row.
 */
moe_status_t moe_init_routing_workspace_size(int32_t T, int32_t k, int32_t E,
                                             size_t *bytes);
moe_status_t moe_init_routing(const int32_t *topk_idx, const moe_bf16_t *x, int32_t T,
                              int32_t H, int32_t E, int32_t k, moe_bf16_t *expanded_x,
                              int32_t *expanded_row_idx, int32_t *src_token,
                              int32_t *sorted_expert_ids, int32_t *counts,
                              int32_t *offsets, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, moe_stream_t stream);

/*
 * moe_init_routing without a workspace argument, for callers that cannot
 * allocate device memory (for example code that only receives input and
 * output pointers from a host framework that owns all memory, or a context
 * where a cudaMalloc is not allowed or would stall the device).  The page
 * has no counterpart of this entry point; it is a convenience of this
 * library.  Same arguments, results and errors as moe_init_routing.
 *   - The routing histogram lives in a 1 MiB array inside the library
 *     (262144 int32), held on every GPU that loads the library until the
 *     process exits.  A call needs ceil(T/32) * E of its entries; larger
 *     calls are rejected with MOE_ERR_WORKSPACE_TOO_SMALL (e.g. E = 64 allows
 *     T up to 131072).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (every entry a call reads it writes first, so nothing needs clearing).
 *     Calls whose execution overlaps on the GPU (different streams, or
 *     different host threads) race on it and give wrong results: serialise
 *     them.
 * Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 */
moe_status_t moe_init_routing_noalloc(const int32_t *topk_idx, const moe_bf16_t *x, int32_t T,
                                      int32_t H, int32_t E, int32_t k, moe_bf16_t *expanded_x,
                                      int32_t *expanded_row_idx, int32_t *src_token,
                                      int32_t *sorted_expert_ids, int32_t *counts,
                                      int32_t *offsets, int32_t *dev_status,
                                      moe_stream_t stream);

/*
 * compute_expert_tokens ("GMM使能&&Routing优化": how many tokens each expert
 * computes), from the expert ids of the sorted rows:
 *   sorted_expert_ids [n] int32, ascending
 *   counts [E], offsets [E+1] (offsets[e] = first row of expert e)
 * An unsorted input sets MOE_DEV_UNSORTED, an id outside [0,E)
 * MOE_DEV_BAD_EXPERT_ID.  n may be 0.
 */
moe_status_t moe_expert_tokens(const int32_t *sorted_expert_ids, int32_t n, int32_t E,
                               int32_t *counts, int32_t *offsets, int32_t *dev_status,
                               moe_stream_t stream);

/*
 * Grouped expert FFN ("GMM使能&&Routing优化": one grouped matmul for all
 * experts; "MoE TP优化 / 计算分解": x = down(SiLU(gate(x)) * up(x)), gate and
 * up merged into w13, SwiGLU = SiLU(first half) * second half).
 *   expanded_x [n, H] bf16, rows sorted by group
 *   offsets    [G+1] int32 device: group g owns rows [offsets[g], offsets[g+1])
 *   w13        [G, 2I, H] bf16: rows 0..I-1 gate, I..2I-1 up
 *   w2         [G, H, I] bf16
 *   act        [n, I] bf16 out: bf16(SiLU(g) * u), g/u accumulated in fp32
 *   y          [n, H] bf16 out: bf16(act . w2[g]^T), fp32 accumulation
 * Rows past offsets[G] are left untouched.  Both matmuls run on the 5th
 * generation tensor cores (tcgen05, TMEM accumulators, TMA operand loads).
 */
moe_status_t moe_grouped_mlp(const moe_bf16_t *expanded_x, const int32_t *offsets,
                             int32_t G, const moe_bf16_t *w13, const moe_bf16_t *w2,
                             int32_t n, int32_t H, int32_t I, moe_bf16_t *act,
                             moe_bf16_t *y, int32_t *dev_status, moe_stream_t stream);

/*
 * finalize_routing ("GMM使能&&Routing优化": put the expert outputs back in
 * token order and form the weighted sum) plus the shared expert
 * ("MoE多流并行优化"):
 *   out[t, :] = sum_{j=0..k-1} topk_w[t, j] * y_exp[expanded_row_idx[t*k+j], :]
 *               + shared[t, :]
 * summed in fp32 in slot order j = 0..k-1, the shared term last; no atomics,
 * so the result is deterministic.
 *   y_exp [T*k, H] bf16 (fp32 with MOE_Y_F32); expanded_row_idx [T*k];
 *   topk_w [T, k] fp32
 *   shared [T, H] bf16 (fp32 with MOE_SHARED_F32) or NULL
 *   out [T, H] bf16 (fp32 with MOE_OUT_F32)
 */
moe_status_t moe_finalize_routing(const void *y_exp, const int32_t *expanded_row_idx,
                                  const float *topk_w, const void *shared, int32_t T,
                                  int32_t H, int32_t k, uint32_t flags, void *out,
                                  moe_stream_t stream);

/*
 * The whole layer, every step above on `stream` with no host synchronisation:
 *   x [T,H] bf16; gamma [H] bf16 or NULL (MOE_RMSNORM); wg [E,H] fp32;
 *   gate_bias [E] fp32 or NULL; w13 [E,2I,H], w2 [E,H,I] bf16;
 *   w13_s [2I_s,H], w2_s [H,I_s] bf16 (MOE_SHARED, else NULL);
 *   out [T,H] bf16 (fp32 with MOE_OUT_F32).
 * The shared expert runs on the normalised rows with weight 1 and its output
 * enters the final sum in fp32.  The routed expert outputs are rounded to
 * bf16 before the weighted sum (a grouped matmul's output type), or, with
 * MOE_Y_F32, enter it as the down matmul's fp32 accumulator: then nothing
 * between the two matmuls' fp32 sums and the weighted sum is rounded except
 * the SwiGLU output (twice the y_exp bytes: one more write and read of
 * T*k*H*2 bytes per layer).  For T > 512 the gate is moe_gate_tensor's
 * (fp32-accurate, another summation order) unless MOE_GATE_SEQUENTIAL is set;
 * smaller batches always use the sequential gate of moe_rmsnorm_gate.
 * Workspace: moe_layer_workspace_size() bytes,
 * 256-byte aligned; its contents are scratch.
 */
moe_status_t moe_layer_workspace_size(const moe_desc_t *desc, size_t *bytes);
moe_status_t moe_layer_forward(const moe_desc_t *desc, const moe_bf16_t *x,
                               const moe_bf16_t *gamma, const float *wg,
                               const float *gate_bias, const moe_bf16_t *w13,
                               const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                               const moe_bf16_t *w2_s, void *out, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status,
                               moe_stream_t stream);

/*
 * moe_layer_forward with per-stage timing: identical work, plus
 * cudaEventRecord(stage_events[i], stream) before launch stage i and
 * stage_events[MOE_NUM_STAGES] after the last one.  Stages:
 *   0 RMSNorm + gate + top-k (+ routing histogram)
 *   1 routing scan + stable scatter
 *   2 permute (expanded_x rows)
 *   3 grouped w13 matmul + SwiGLU (routed and shared expert)
 *   4 grouped down matmul
 *   5 finalize
 * stage_events: MOE_NUM_STAGES + 1 cudaEvent_t handles owned by the caller
 * (created with timing enabled); NULL behaves as moe_layer_forward.
 */
#define MOE_NUM_STAGES 6
moe_status_t moe_layer_forward_timed(const moe_desc_t *desc, const moe_bf16_t *x,
                                     const moe_bf16_t *gamma, const float *wg,
                                     const float *gate_bias, const moe_bf16_t *w13,
                                     const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                     const moe_bf16_t *w2_s, void *out, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_status,
                                     moe_stream_t stream, void *const *stage_events);

/*
 * moe_layer_forward on two streams ("MoE多流并行优化": the shared expert
 * runs beside the routed path on another stream).  Same results, bit for
 * bit, as moe_layer_forward.  After the routing indices, `fork_event` is
 * recorded on `stream` and awaited by `shared_stream`, which copies the rows
 * into expert order (memory-bound) and records `join_event`; meanwhile
 * `stream` computes the shared expert's w13 matmul (tensor-bound), then
 * awaits `join_event` and runs the routed matmuls and finalize.  (On GB300
 * this beat running the shared expert's matmuls themselves on the second
 * stream: two persistent matmul kernels cannot share the SMs.)
 * The caller owns both streams and both events (cudaEvent_t, any flags) and
 * must not use the events concurrently elsewhere.  Requires MOE_SHARED.
 * stage_events: as in moe_layer_forward_timed (recorded on `stream`), or NULL.
 */
moe_status_t moe_layer_forward_streams(const moe_desc_t *desc, const moe_bf16_t *x,
                                       const moe_bf16_t *gamma, const float *wg,
                                       const float *gate_bias, const moe_bf16_t *w13,
                                       const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                       const moe_bf16_t *w2_s, void *out, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       moe_stream_t stream, moe_stream_t shared_stream,
                                       void *fork_event, void *join_event,
                                       void *const *stage_events);

/*
 * moe_layer_forward over n_batches token batches held in host memory, with
 * the copies overlapped with the compute: while batch i runs on `stream`,
 * batch i+1's tokens are copied in on `copy_in` and batch i-1's output is
 * copied out on `copy_out` (two device staging buffers each way).  The
 * results are those of moe_layer_forward on each batch.
 *   x_host[i]   [T, H] bf16, host memory (pinned, or the copies serialise)
 *   out_host[i] [T, H] host memory, bf16 (fp32 with MOE_OUT_F32)
 *   x_dev       device, 2*T*H bf16 (staging), 16-byte aligned
 *   out_dev     device, 2 * T*H output elements (staging), 16-byte aligned
 *   workspace   as moe_layer_forward (one workspace serves every batch)
 *   stream, copy_in, copy_out: three distinct streams owned by the caller
 *   events      6 cudaEvent_t owned by the caller, used only by this call
 * Returns once everything is enqueued (nothing is synchronised): the last
 * output is in host memory when copy_out has drained.  All arguments are
 * checked before the first copy; a launch or copy error returns MOE_ERR_CUDA
 * with the earlier batches still enqueued.
 */
moe_status_t moe_layer_forward_host(const moe_desc_t *desc, int32_t n_batches,
                                    const moe_bf16_t *const *x_host, void *const *out_host,
                                    const moe_bf16_t *gamma, const float *wg,
                                    const float *gate_bias, const moe_bf16_t *w13,
                                    const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                    const moe_bf16_t *w2_s, moe_bf16_t *x_dev, void *out_dev,
                                    void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                    moe_stream_t stream, moe_stream_t copy_in,
                                    moe_stream_t copy_out, void *const *events);

/*
 * EP DoubleRouting, the steps local to one rank ("MoE EP优化": LocalRerouting
 * orders a rank's received tokens by its local experts; LocalFinalizeRerouting
 * restores the order the second all_to_all expects).  After the token all_to_all a rank holds
 * the received rows grouped by source rank and, within a source rank,
 * ordered by local expert:
 *   recv_counts [ep_size, E_local] int32 device: rows from rank r for local
 *               expert e (ep_size * E_local <= 8192)
 *   recv_x      [R, H] bf16, R = capacity >= sum(recv_counts)
 * moe_local_rerouting reorders them by local expert, then source rank, then
 * arrival order:
 *   local_x[d] = recv_x[local_src[d]] (local_x may be NULL: indices only)
 *   local_src  [R] int32 out (-1 past the received rows)
 *   local_counts [E_local], local_offsets [E_local+1] out (grouped-GEMM input)
 * Negative counts or a total above R set MOE_DEV_BAD_OFFSETS.
 * moe_local_finalize_rerouting moves expert outputs back to the received
 * order: recv_y[local_src[d]] = local_y[d] for every d with local_src[d] >= 0.
 */
moe_status_t moe_local_rerouting(const moe_bf16_t *recv_x, const int32_t *recv_counts,
                                 int32_t ep_size, int32_t E_local, int32_t R, int32_t H,
                                 moe_bf16_t *local_x, int32_t *local_src,
                                 int32_t *local_counts, int32_t *local_offsets,
                                 int32_t *dev_status, moe_stream_t stream);
moe_status_t moe_local_finalize_rerouting(const moe_bf16_t *local_y, const int32_t *local_src,
                                          int32_t R, int32_t H, moe_bf16_t *recv_y,
                                          moe_stream_t stream);

/*
 * Diagnostics (the page has no counterpart): enqueue a kernel that waits,
 * through the same bounded wait every pipeline here uses, on a barrier that
 * nothing completes.  After about one second it ORs MOE_DEV_TIMEOUT into
 * *dev_status (required, device int32) and returns; the context stays usable.
 */
moe_status_t moe_selftest_wait_timeout(int32_t *dev_status, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
