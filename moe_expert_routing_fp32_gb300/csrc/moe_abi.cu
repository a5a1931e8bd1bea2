// moe_abi.cu -- the extern "C" entry points declared in include/moe.h.
//
// Host side only: argument checks, workspace carving and the launch sequence
// of each operation.  Nothing here allocates, frees or synchronises.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

DeviceInfo &device_info(int dev) {
    static DeviceInfo info[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    std::call_once(once[dev], [dev] {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
            info[dev].sms = prop.multiProcessorCount;
            info[dev].ok = prop.major == 10;   // the sm_100 family (sm_103a build)
        } else {
            cudaGetLastError();   // leave no error pending for later launches
        }
    });
    return info[dev];
}

inline bool a16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

#define MOE_TRY(expr)                                   \
    do {                                                \
        cudaError_t err_ = (expr);                      \
        if (err_ != cudaSuccess) return MOE_ERR_CUDA;   \
    } while (0)

// Layout of the layer workspace (offsets in bytes, each 256-aligned).
struct LayerWs {
    size_t xn = 0, logits = 0, wsplit = 0, parts = 0, idx = 0, w = 0, hist = 0, counts = 0,
           offsets = 0, row_idx = 0, src_token = 0, expanded_x = 0, act = 0, y = 0, act_s = 0,
           y_s = 0, total = 0;
};

// The layer's gate runs on the tensor cores for batches above the small
// router's range unless the caller asks for the sequential one.
bool layer_gate_tc(const moe_desc_t &d) {
    return d.T > kGateSmallMaxT && !(d.flags & MOE_GATE_SEQUENTIAL);
}

// Tensor-core gate scratch: the split weight [NW, H] bf16, then the partial
// logits [T, NW] fp32 (NW = gate_tc_cols(E)).
size_t gate_tc_split_bytes(int H, int E) {
    return align256(static_cast<size_t>(gate_tc_cols(E)) * H * 2);
}
size_t gate_tc_parts_bytes(int T, int E) {
    return align256(static_cast<size_t>(T) * gate_tc_cols(E) * 4);
}

// Split, GEMM, combine.  With fuse (E <= kRouterExperts) the combine also
// takes the top-k and the chunk histograms; `logits` may then be NULL.
cudaError_t launch_gate_tc(const uint16_t *xs, const float *wg, const float *gate_bias, int T,
                           int H, int E, uint16_t *wsplit, float *parts, float *logits,
                           bool fuse, int k, bool renorm, int32_t *idx, float *w,
                           int32_t *hist, int32_t *dev_status, cudaStream_t s) {
    const int NW = gate_tc_cols(E);
    cudaError_t e = launch_gate_split(wg, E, H, wsplit, NW, s);
    if (e != cudaSuccess) return e;
    GemmSegment1 g;
    g.A = xs;
    g.B = wsplit;
    g.rows = T;
    g.K1 = H;
    g.N1 = NW;
    g.out = parts;
    g.out_f32 = true;
    // no grouped problem (G = 0): the offsets pointer only has to be readable
    e = launch_gemm_store(nullptr, reinterpret_cast<const int32_t *>(wsplit), 0, 0, H, nullptr,
                          NW, nullptr, g, dev_status, s);
    if (e != cudaSuccess) return e;
    return launch_gate_combine(parts, NW, T, E, gate_bias, logits, fuse, k, renorm, idx, w,
                               hist, s);
}

// MOE_GATHER_A takes effect where the routed w13 matmul runs as the wide pair
// kernel (a shape decision, the same for every call with this descriptor).
bool layer_gathers(const moe_desc_t &d) {
    if (!(d.flags & MOE_GATHER_A)) return false;
    GemmSegment1 sh;
    if (d.flags & MOE_SHARED) {
        sh.rows = d.T;
        sh.K1 = d.H;
        sh.N1 = d.I_shared;
    }
    return gemm_can_gather(d.T * d.k, d.E, d.H, d.I, sh);
}

LayerWs layer_layout(const moe_desc_t &d) {
    LayerWs L;
    const size_t T = d.T, H = d.H, E = d.E, k = d.k, I = d.I, Is = d.I_shared;
    const size_t N = T * k;
    const size_t B = static_cast<size_t>(ceil_div(d.T, kChunkTokens));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += align256(bytes);
        return o;
    };
    if (d.flags & MOE_RMSNORM) L.xn = take(T * H * 2);
    if (d.E > kRouterExperts) L.logits = take(T * E * 4);
    if (layer_gate_tc(d)) {
        L.wsplit = take(gate_tc_split_bytes(d.H, d.E));
        L.parts = take(gate_tc_parts_bytes(d.T, d.E));
    }
    L.idx = take(N * 4);
    L.w = take(N * 4);
    L.hist = take(B * E * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.row_idx = take(N * 4);
    if (layer_gathers(d))
        L.src_token = take(N * 4);      // the w13 matmul reads x's rows through it
    else
        L.expanded_x = take(N * H * 2);
    L.act = take(N * I * 2);
    L.y = take(N * H * ((d.flags & MOE_Y_F32) ? 4 : 2));
    if (d.flags & MOE_SHARED) {
        L.act_s = take(T * Is * 2);
        L.y_s = take(T * H * 4);
    }
    L.total = off;
    return L;
}

moe_status_t check_desc(const moe_desc_t *d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0) return MOE_ERR_INVALID_ARG;
    if (d->E > 1024 || d->k > 32 || d->k > d->E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d->H % 128 != 0 || d->I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(d->T) * d->k >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d->flags & MOE_SHARED) {
        if (d->I_shared <= 0) return MOE_ERR_INVALID_ARG;
        if (d->I_shared % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    }
    if ((d->flags & MOE_RMSNORM) && !(d->rms_eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

bool current_device_ok() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    return device_info(dev).ok;
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    const int s = device_info(dev).sms;
    return s > 0 ? s : 148;
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
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_NO_DEVICE: return "MOE_ERR_NO_DEVICE";
        default: return "MOE_ERR_UNKNOWN";
    }
}

moe_status_t moe_rmsnorm_gate(const moe_bf16_t *x, const moe_bf16_t *gamma, const float *wg,
                              const float *gate_bias, int32_t T, int32_t H, int32_t E, float eps,
                              uint32_t flags, moe_bf16_t *xn, float *logits,
                              moe_stream_t stream) {
    const bool rms = (flags & MOE_RMSNORM) != 0;
    if (T < 0 || H <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 64 != 0 || E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!wg && !logits) {
        // RMSNorm alone (the pass ahead of the tensor-core gate)
        if (!rms || !x || !xn || !a16(x) || !a16(xn) || (gamma && !a16(gamma)) || !(eps >= 0))
            return MOE_ERR_INVALID_ARG;
        if (H % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
        MOE_TRY(launch_rmsnorm(x, gamma, T, H, eps, xn, nullptr,
                               reinterpret_cast<cudaStream_t>(stream)));
        return MOE_OK;
    }
    if (!x || !wg || !logits || (rms && !xn)) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(wg) || (rms && !a16(xn)) || (gamma && !a16(gamma)) || (rms && !(eps >= 0)))
        return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_router(x, rms ? gamma : nullptr, wg, gate_bias, T, H, E, eps, rms,
                          rms ? xn : nullptr, logits, false, 1, false, nullptr, nullptr, nullptr,
                          nullptr, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_rmsnorm_sumsq(const moe_bf16_t *x, int32_t T, int32_t H, float *ss,
                               moe_stream_t stream) {
    if (T < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!x || !ss || !a16(x)) return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_sumsq(x, T, H, ss, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_gate_tensor_workspace_size(int32_t T, int32_t H, int32_t E, size_t *bytes) {
    if (!bytes || T < 0 || H <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 128 != 0 || E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    *bytes = gate_tc_split_bytes(H, E) + gate_tc_parts_bytes(T, E);
    return MOE_OK;
}

moe_status_t moe_gate_tensor(const moe_bf16_t *xs, const float *wg, const float *gate_bias,
                             int32_t T, int32_t H, int32_t E, float *logits, void *workspace,
                             size_t workspace_bytes, int32_t *dev_status, moe_stream_t stream) {
    size_t need = 0;
    const moe_status_t st = moe_gate_tensor_workspace_size(T, H, E, &need);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (!xs || !wg || !logits) return MOE_ERR_INVALID_ARG;
    if (!a16(xs) || !a16(wg)) return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    if (!tensor_maps_available()) return MOE_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    MOE_TRY(launch_gate_tc(xs, wg, gate_bias, T, H, E, reinterpret_cast<uint16_t *>(ws),
                           reinterpret_cast<float *>(ws + gate_tc_split_bytes(H, E)), logits,
                           false, 1, false, nullptr, nullptr, nullptr, dev_status,
                           reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_gate_topk(const float *logits, int32_t T, int32_t E, int32_t k, uint32_t flags,
                           int32_t *topk_idx, float *topk_w, moe_stream_t stream) {
    if (T < 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_topk(logits, T, E, k, (flags & MOE_RENORM) != 0, topk_idx, topk_w,
                        reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_init_routing_workspace_size(int32_t T, int32_t k, int32_t E, size_t *bytes) {
    if (!bytes || T < 0 || k <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    *bytes = align256(static_cast<size_t>(ceil_div(T, kChunkTokens)) * E * 4);
    return MOE_OK;
}

moe_status_t moe_init_routing(const int32_t *topk_idx, const moe_bf16_t *x, int32_t T, int32_t H,
                              int32_t E, int32_t k, moe_bf16_t *expanded_x,
                              int32_t *expanded_row_idx, int32_t *src_token,
                              int32_t *sorted_expert_ids, int32_t *counts, int32_t *offsets,
                              void *workspace, size_t workspace_bytes, int32_t *dev_status,
                              moe_stream_t stream) {
    if (T < 0 || E <= 0 || k <= 0 || H < 0) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<int64_t>(T) * k >= (int64_t{1} << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !expanded_row_idx || !src_token)) return MOE_ERR_INVALID_ARG;
    if (expanded_x) {
        if (!x || H <= 0) return MOE_ERR_INVALID_ARG;
        if (H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (!a16(x) || !a16(expanded_x)) return MOE_ERR_INVALID_ARG;
    }
    size_t need = 0;
    moe_init_routing_workspace_size(T, k, E, &need);
    if (T > 0 && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t *hist = static_cast<int32_t *>(workspace);
    const int B = static_cast<int>(ceil_div(T, kChunkTokens));
    if (T == 0) {
        MOE_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s));
        MOE_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s));
        return MOE_OK;
    }
    if (scan_builds_hist(T, E)) {
        MOE_TRY(launch_route_scan(hist, B, E, counts, offsets, topk_idx, T, k, dev_status, s));
    } else {
        MOE_TRY(launch_route_hist(topk_idx, T, k, E, hist, dev_status, s));
        MOE_TRY(launch_route_scan(hist, B, E, counts, offsets, nullptr, T, k, dev_status, s));
    }
    MOE_TRY(launch_route_scatter(topk_idx, hist, T, k, E, expanded_row_idx, src_token,
                                 sorted_expert_ids, dev_status, s));
    if (expanded_x) MOE_TRY(launch_permute(x, expanded_row_idx, T, H, k, expanded_x, s));
    return MOE_OK;
}

moe_status_t moe_expert_tokens(const int32_t *sorted_expert_ids, int32_t n, int32_t E,
                               int32_t *counts, int32_t *offsets, int32_t *dev_status,
                               moe_stream_t stream) {
    if (n < 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (E > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!counts || !offsets || (n > 0 && !sorted_expert_ids)) return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_expert_tokens(sorted_expert_ids, n, E, counts, offsets, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_grouped_mlp(const moe_bf16_t *expanded_x, const int32_t *offsets, int32_t G,
                             const moe_bf16_t *w13, const moe_bf16_t *w2, int32_t n, int32_t H,
                             int32_t I, moe_bf16_t *act, moe_bf16_t *y, int32_t *dev_status,
                             moe_stream_t stream) {
    if (G <= 0 || n < 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (G > 1024 || H % 128 != 0 || I % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!offsets || !w13 || !w2) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!expanded_x || !act || !y) return MOE_ERR_INVALID_ARG;
    if (!a16(expanded_x) || !a16(w13) || !a16(w2) || !a16(act) || !a16(y))
        return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    if (!tensor_maps_available()) return MOE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    GemmSegment1 none;
    MOE_TRY(launch_gemm_swiglu(expanded_x, offsets, G, n, H, w13, I, act, none, dev_status, s));
    MOE_TRY(launch_gemm_store(act, offsets, G, n, I, w2, H, y, none, dev_status, s));
    return MOE_OK;
}

moe_status_t moe_finalize_routing(const void *y_exp, const int32_t *expanded_row_idx,
                                  const float *topk_w, const void *shared, int32_t T, int32_t H,
                                  int32_t k, uint32_t flags, void *out, moe_stream_t stream) {
    if (T < 0 || H <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0 || k > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!y_exp || !expanded_row_idx || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!a16(y_exp) || !a16(out) || (shared && !a16(shared))) return MOE_ERR_INVALID_ARG;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    MOE_TRY(launch_finalize(y_exp, (flags & MOE_Y_F32) != 0, expanded_row_idx, topk_w, shared,
                            (flags & MOE_SHARED_F32) != 0, T, H, k, out,
                            (flags & MOE_OUT_F32) != 0, reinterpret_cast<cudaStream_t>(stream)));
    return MOE_OK;
}

moe_status_t moe_layer_workspace_size(const moe_desc_t *desc, size_t *bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = check_desc(desc);
    if (st != MOE_OK) return st;
    *bytes = layer_layout(*desc).total;
    return MOE_OK;
}

}  // extern "C"

namespace {

// The layer; `stage_events` as in moe_layer_forward_timed; with
// `shared_stream` the row copies of init_routing run on that stream (between
// `fork_event` and `join_event`) while `stream` computes the shared expert's
// w13, so the memory-bound copies overlap a tensor-bound matmul.
moe_status_t layer_forward_impl(const moe_desc_t *desc, const moe_bf16_t *x,
                                const moe_bf16_t *gamma, const float *wg, const float *gate_bias,
                                const moe_bf16_t *w13, const moe_bf16_t *w2,
                                const moe_bf16_t *w13_s, const moe_bf16_t *w2_s, void *out,
                                void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                moe_stream_t stream, void *const *stage_events,
                                moe_stream_t shared_stream, void *fork_event, void *join_event) {
    moe_status_t st = check_desc(desc);
    if (st != MOE_OK) return st;
    const moe_desc_t d = *desc;
    const bool rms = (d.flags & MOE_RMSNORM) != 0;
    const bool shared = (d.flags & MOE_SHARED) != 0;
    if (!wg || !w13 || !w2 || (shared && (!w13_s || !w2_s))) return MOE_ERR_INVALID_ARG;
    if (d.T == 0) return MOE_OK;
    if (!x || !out) return MOE_ERR_INVALID_ARG;
    if (!a16(x) || !a16(wg) || !a16(w13) || !a16(w2) || !a16(out) || (gamma && !a16(gamma)) ||
        (shared && (!a16(w13_s) || !a16(w2_s))))
        return MOE_ERR_INVALID_ARG;
    const LayerWs L = layer_layout(d);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (!current_device_ok()) return MOE_ERR_NO_DEVICE;
    if (!tensor_maps_available()) return MOE_ERR_CUDA;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto at = [&](size_t off) { return static_cast<void *>(ws + off); };
    uint16_t *xn = rms ? static_cast<uint16_t *>(at(L.xn)) : nullptr;
    float *logits = d.E > kRouterExperts ? static_cast<float *>(at(L.logits)) : nullptr;
    int32_t *idx = static_cast<int32_t *>(at(L.idx));
    float *w = static_cast<float *>(at(L.w));
    int32_t *hist = static_cast<int32_t *>(at(L.hist));
    int32_t *counts = static_cast<int32_t *>(at(L.counts));
    int32_t *offsets = static_cast<int32_t *>(at(L.offsets));
    int32_t *row_idx = static_cast<int32_t *>(at(L.row_idx));
    const bool gather = layer_gathers(d);
    uint16_t *ex = gather ? nullptr : static_cast<uint16_t *>(at(L.expanded_x));
    int32_t *src_token = gather ? static_cast<int32_t *>(at(L.src_token)) : nullptr;
    uint16_t *act = static_cast<uint16_t *>(at(L.act));
    void *y = at(L.y);   // bf16, or fp32 with MOE_Y_F32
    const bool y_f32 = (d.flags & MOE_Y_F32) != 0;
    uint16_t *act_s = shared ? static_cast<uint16_t *>(at(L.act_s)) : nullptr;
    float *y_s = shared ? static_cast<float *>(at(L.y_s)) : nullptr;
    const uint16_t *xs = rms ? xn : x;
    const bool renorm = (d.flags & MOE_RENORM) != 0;
    const int T = d.T, H = d.H, E = d.E, k = d.k, I = d.I;
    const int N = T * k;
    const int B = static_cast<int>(ceil_div(T, kChunkTokens));

    // Each stage is also an NVTX range on the host thread (closed when the
    // next stage starts or the call returns), so a timeline tool shows which
    // launches belong to which step of the layer.
    static const char *const kStageNames[MOE_NUM_STAGES] = {
        "moe/router", "moe/route_scan_scatter", "moe/permute", "moe/gemm_w13_swiglu",
        "moe/gemm_down", "moe/finalize"};
    struct NvtxStage {
        bool open = false;
        void next(int i) {
            if (open) nvtxRangePop();
            open = i < MOE_NUM_STAGES;
            if (open) nvtxRangePushA(kStageNames[i]);
        }
        ~NvtxStage() {
            if (open) nvtxRangePop();
        }
    } nvtx;
    auto mark = [&](int i) -> cudaError_t {
        nvtx.next(i);
        if (!stage_events) return cudaSuccess;
        return cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), s);
    };

    // 1. RMSNorm + gate (+ top-k, and the routing histogram when E <= 64 and
    // the scan does not count it itself)
    MOE_TRY(mark(0));
    const bool fuse = E <= kRouterExperts;
    const bool scan_hist = scan_builds_hist(T, E);
    int32_t *hist_out = fuse && !scan_hist ? hist : nullptr;
    if (layer_gate_tc(d)) {
        // RMSNorm alone, then the gate as a tensor-core GEMM on the normalised rows
        if (rms) MOE_TRY(launch_rmsnorm(x, gamma, T, H, d.rms_eps, xn, dev_status, s));
        MOE_TRY(launch_gate_tc(xs, wg, gate_bias, T, H, E, static_cast<uint16_t *>(at(L.wsplit)),
                               static_cast<float *>(at(L.parts)), logits, fuse, k, renorm, idx, w,
                               hist_out, dev_status, s));
    } else {
        MOE_TRY(launch_router(x, rms ? gamma : nullptr, wg, gate_bias, T, H, E, d.rms_eps, rms,
                              xn, logits, fuse, k, renorm, idx, w, hist_out, dev_status, s));
    }
    if (!fuse) {
        MOE_TRY(launch_topk(logits, T, E, k, renorm, idx, w, s));
        if (!scan_hist) MOE_TRY(launch_route_hist(idx, T, k, E, hist, dev_status, s));
    }
    // 2. init_routing: scan + stable scatter, then the row copies
    MOE_TRY(mark(1));
    MOE_TRY(launch_route_scan(hist, B, E, counts, offsets, scan_hist ? idx : nullptr, T, k,
                              dev_status, s));
    MOE_TRY(launch_route_scatter(idx, hist, T, k, E, row_idx, src_token, nullptr, dev_status, s));
    MOE_TRY(mark(2));
    // with the rows gathered inside the w13 matmul there is no copy to overlap
    const bool two_streams = shared && shared_stream != nullptr && !gather;
    GemmSegment1 sh13;       // the shared expert's w13 + SwiGLU as a dense segment
    if (shared) {
        sh13.A = xs;
        sh13.B = w13_s;
        sh13.rows = T;
        sh13.K1 = H;
        sh13.N1 = d.I_shared;
        sh13.out = act_s;
    }
    if (two_streams) {
        // The row copies (memory-bound) run on the second stream while this
        // stream computes the shared expert's w13 (tensor-bound); the routed
        // w13 waits for both.
        cudaStream_t s2 = reinterpret_cast<cudaStream_t>(shared_stream);
        cudaEvent_t fork = static_cast<cudaEvent_t>(fork_event);
        cudaEvent_t join = static_cast<cudaEvent_t>(join_event);
        MOE_TRY(cudaEventRecord(fork, s));
        MOE_TRY(cudaStreamWaitEvent(s2, fork, 0));
        MOE_TRY(launch_permute(xs, row_idx, T, H, k, ex, s2));
        MOE_TRY(cudaEventRecord(join, s2));
        MOE_TRY(mark(3));
        MOE_TRY(launch_gemm_swiglu(nullptr, offsets, 0, 0, H, nullptr, I, nullptr, sh13,
                                   dev_status, s));
        MOE_TRY(cudaStreamWaitEvent(s, join, 0));
        const GemmSegment1 none{};
        MOE_TRY(launch_gemm_swiglu(ex, offsets, E, N, H, w13, I, act, none, dev_status, s));
    } else if (gather) {
        // 3. grouped w13 + SwiGLU, its A rows read from xs by source token
        MOE_TRY(mark(3));
        MOE_TRY(launch_gemm_swiglu(nullptr, offsets, E, N, H, w13, I, act, sh13, dev_status, s,
                                   xs, src_token, T));
    } else {
        MOE_TRY(launch_permute(xs, row_idx, T, H, k, ex, s));
        // 3. grouped w13 + SwiGLU (the shared expert rides along as a dense segment)
        MOE_TRY(mark(3));
        MOE_TRY(launch_gemm_swiglu(ex, offsets, E, N, H, w13, I, act, sh13, dev_status, s));
    }
    // 4. grouped down projection (the shared expert's as a dense segment, kept in fp32)
    GemmSegment1 s2;
    if (shared) {
        s2.A = act_s;
        s2.B = w2_s;
        s2.rows = T;
        s2.K1 = d.I_shared;
        s2.N1 = H;
        s2.out = y_s;
        s2.out_f32 = true;
    }
    MOE_TRY(mark(4));
    MOE_TRY(launch_gemm_store(act, offsets, E, N, I, w2, H, y, s2, dev_status, s, y_f32));
    // 5. finalize: weighted sum in slot order + shared row
    MOE_TRY(mark(5));
    MOE_TRY(launch_finalize(y, y_f32, row_idx, w, y_s, true, T, H, k, out,
                            (d.flags & MOE_OUT_F32) != 0, s));
    MOE_TRY(mark(6));
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_layer_forward(const moe_desc_t *desc, const moe_bf16_t *x,
                               const moe_bf16_t *gamma, const float *wg, const float *gate_bias,
                               const moe_bf16_t *w13, const moe_bf16_t *w2,
                               const moe_bf16_t *w13_s, const moe_bf16_t *w2_s, void *out,
                               void *workspace, size_t workspace_bytes, int32_t *dev_status,
                               moe_stream_t stream) {
    return layer_forward_impl(desc, x, gamma, wg, gate_bias, w13, w2, w13_s, w2_s, out,
                              workspace, workspace_bytes, dev_status, stream, nullptr, nullptr,
                              nullptr, nullptr);
}

moe_status_t moe_layer_forward_timed(const moe_desc_t *desc, const moe_bf16_t *x,
                                     const moe_bf16_t *gamma, const float *wg,
                                     const float *gate_bias, const moe_bf16_t *w13,
                                     const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                     const moe_bf16_t *w2_s, void *out, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_status,
                                     moe_stream_t stream, void *const *stage_events) {
    return layer_forward_impl(desc, x, gamma, wg, gate_bias, w13, w2, w13_s, w2_s, out,
                              workspace, workspace_bytes, dev_status, stream, stage_events,
                              nullptr, nullptr, nullptr);
}

moe_status_t moe_layer_forward_streams(const moe_desc_t *desc, const moe_bf16_t *x,
                                       const moe_bf16_t *gamma, const float *wg,
                                       const float *gate_bias, const moe_bf16_t *w13,
                                       const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                       const moe_bf16_t *w2_s, void *out, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status,
                                       moe_stream_t stream, moe_stream_t shared_stream,
                                       void *fork_event, void *join_event,
                                       void *const *stage_events) {
    if (!shared_stream || !fork_event || !join_event || shared_stream == stream)
        return MOE_ERR_INVALID_ARG;
    return layer_forward_impl(desc, x, gamma, wg, gate_bias, w13, w2, w13_s, w2_s, out,
                              workspace, workspace_bytes, dev_status, stream, stage_events,
                              shared_stream, fork_event, join_event);
}

moe_status_t moe_layer_forward_host(const moe_desc_t *desc, int32_t n_batches,
                                    const moe_bf16_t *const *x_host, void *const *out_host,
                                    const moe_bf16_t *gamma, const float *wg,
                                    const float *gate_bias, const moe_bf16_t *w13,
                                    const moe_bf16_t *w2, const moe_bf16_t *w13_s,
                                    const moe_bf16_t *w2_s, moe_bf16_t *x_dev, void *out_dev,
                                    void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                    moe_stream_t stream, moe_stream_t copy_in,
                                    moe_stream_t copy_out, void *const *events) {
    moe_status_t st = check_desc(desc);
    if (st != MOE_OK) return st;
    if (n_batches < 0) return MOE_ERR_INVALID_ARG;
    if (n_batches == 0 || desc->T == 0) return MOE_OK;
    if (!x_host || !out_host || !x_dev || !out_dev || !events || !copy_in || !copy_out ||
        copy_in == stream || copy_out == stream || copy_in == copy_out)
        return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_batches; ++i)
        if (!x_host[i] || !out_host[i]) return MOE_ERR_INVALID_ARG;
    // the per-batch layer checks, once, before anything is enqueued
    const bool shared = (desc->flags & MOE_SHARED) != 0;
    if (!wg || !w13 || !w2 || (shared && (!w13_s || !w2_s))) return MOE_ERR_INVALID_ARG;
    if (!a16(x_dev) || !a16(out_dev) || !a16(wg) || !a16(w13) || !a16(w2) ||
        (gamma && !a16(gamma)) || (shared && (!a16(w13_s) || !a16(w2_s))))
        return MOE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < layer_layout(*desc).total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    const size_t rows = static_cast<size_t>(desc->T) * desc->H;
    const size_t x_bytes = rows * 2;
    const size_t o_bytes = rows * ((desc->flags & MOE_OUT_F32) ? 4 : 2);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t cin = reinterpret_cast<cudaStream_t>(copy_in);
    cudaStream_t cout = reinterpret_cast<cudaStream_t>(copy_out);
    cudaEvent_t in_ready[2] = {static_cast<cudaEvent_t>(events[0]),
                               static_cast<cudaEvent_t>(events[1])};
    cudaEvent_t computed[2] = {static_cast<cudaEvent_t>(events[2]),
                               static_cast<cudaEvent_t>(events[3])};
    cudaEvent_t copied_out[2] = {static_cast<cudaEvent_t>(events[4]),
                                 static_cast<cudaEvent_t>(events[5])};
    auto cuda = [](cudaError_t e) { return e == cudaSuccess; };
    for (int32_t i = 0; i < n_batches; ++i) {
        const int b = i & 1;
        uint16_t *xb = reinterpret_cast<uint16_t *>(x_dev) + b * rows;
        uint8_t *ob = static_cast<uint8_t *>(out_dev) + b * o_bytes;
        // tokens in: staging buffer b was last read by batch i-2's layer
        if (i >= 2 && !cuda(cudaStreamWaitEvent(cin, computed[b], 0))) return MOE_ERR_CUDA;
        if (!cuda(cudaMemcpyAsync(xb, x_host[i], x_bytes, cudaMemcpyHostToDevice, cin)) ||
            !cuda(cudaEventRecord(in_ready[b], cin)))
            return MOE_ERR_CUDA;
        // the layer: after its tokens landed and batch i-2's output left buffer b
        if (!cuda(cudaStreamWaitEvent(s, in_ready[b], 0))) return MOE_ERR_CUDA;
        if (i >= 2 && !cuda(cudaStreamWaitEvent(s, copied_out[b], 0))) return MOE_ERR_CUDA;
        st = layer_forward_impl(desc, reinterpret_cast<const moe_bf16_t *>(xb), gamma, wg,
                                gate_bias, w13, w2, w13_s, w2_s, ob, workspace, workspace_bytes,
                                dev_status, stream, nullptr, nullptr, nullptr, nullptr);
        if (st != MOE_OK) return st;
        if (!cuda(cudaEventRecord(computed[b], s))) return MOE_ERR_CUDA;
        // output out
        if (!cuda(cudaStreamWaitEvent(cout, computed[b], 0)) ||
            !cuda(cudaMemcpyAsync(out_host[i], ob, o_bytes, cudaMemcpyDeviceToHost, cout)) ||
            !cuda(cudaEventRecord(copied_out[b], cout)))
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

}  // extern "C"
