"""Python binding of libmoe, a GB300 (sm_103a) MoE feed-forward layer.

Argument marshalling only: every function below checks dtypes/devices,
allocates its outputs with torch on the input's device and calls the
same-named C entry point of ``libmoe.so`` on torch's current stream.  All
arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or no suitable GPU is present the call raises.

The layer follows "NPU HunyuanImage-3.0模型推理优化实践" (HunyuanImage-3.0 MoE
block: RMSNorm, fp32 gate, GatingTopK, init_routing, compute_expert_tokens,
grouped matmul with SwiGLU on the merged w13 weight, down projection,
finalize_routing, shared expert).  See include/moe.h for the contracts.

Two fp32 gates: ``rmsnorm_gate`` sums each logit sequentially (the oracle's
order, bit for bit); ``gate_tensor`` sums the same exact products on the
tensor cores (the weight split exactly into three bf16 parts), which the
layer uses above 512 tokens unless ``make_desc(..., gate_sequential=True)``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
                3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_NO_DEVICE"}
DEV_BAD_EXPERT_ID, DEV_TIMEOUT, DEV_BAD_OFFSETS, DEV_UNSORTED = 1, 2, 4, 8
RENORM, RMSNORM, SHARED, OUT_F32, SHARED_F32, GATE_SEQUENTIAL, Y_F32 = 1, 2, 4, 8, 16, 32, 64
GATHER_A = 128

# every symbol include/moe.h declares
EXPORTS = ("moe_status_string", "moe_rmsnorm_gate", "moe_rmsnorm_sumsq",
           "moe_gate_tensor_workspace_size",
           "moe_gate_tensor", "moe_gate_topk",
           "moe_init_routing_workspace_size", "moe_init_routing", "moe_init_routing_noalloc",
           "moe_expert_tokens",
           "moe_grouped_mlp", "moe_finalize_routing", "moe_layer_workspace_size",
           "moe_layer_forward", "moe_layer_forward_timed", "moe_layer_forward_streams",
           "moe_layer_forward_host", "moe_local_rerouting",
           "moe_local_finalize_rerouting", "moe_selftest_wait_timeout")
NUM_STAGES = 6
STAGE_NAMES = ("router", "route_scan_scatter", "permute", "gemm_w13_swiglu", "gemm_down",
               "finalize")


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


class MoeDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("rms_eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    from . import native_build
    return native_build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libmoe.so not found at {LIB_PATH}: build it with "
                    "`python -m moe_expert_routing_fp32_gb300.native_build` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, U32, F, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32,
                                  ctypes.c_float, ctypes.c_size_t)
            PSZ = ctypes.POINTER(ctypes.c_size_t)
            sigs = {
                "moe_rmsnorm_gate": [P, P, P, P, I32, I32, I32, F, U32, P, P, P],
                "moe_rmsnorm_sumsq": [P, I32, I32, P, P],
                "moe_gate_tensor_workspace_size": [I32, I32, I32, PSZ],
                "moe_gate_tensor": [P, P, P, I32, I32, I32, P, P, SZ, P, P],
                "moe_gate_topk": [P, I32, I32, I32, U32, P, P, P],
                "moe_init_routing_workspace_size": [I32, I32, I32, PSZ],
                "moe_init_routing": [P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, SZ, P, P],
                "moe_init_routing_noalloc": [P, P, I32, I32, I32, I32, P, P, P, P, P, P, P, P],
                "moe_expert_tokens": [P, I32, I32, P, P, P, P],
                "moe_grouped_mlp": [P, P, I32, P, P, I32, I32, I32, P, P, P, P],
                "moe_finalize_routing": [P, P, P, P, I32, I32, I32, U32, P, P],
                "moe_layer_workspace_size": [ctypes.POINTER(MoeDesc), PSZ],
                "moe_layer_forward": [ctypes.POINTER(MoeDesc), P, P, P, P, P, P, P, P, P, P,
                                      SZ, P, P],
                "moe_layer_forward_timed": [ctypes.POINTER(MoeDesc), P, P, P, P, P, P, P, P, P,
                                            P, SZ, P, P, P],
                "moe_layer_forward_streams": [ctypes.POINTER(MoeDesc), P, P, P, P, P, P, P, P, P,
                                              P, SZ, P, P, P, P, P, P],
                "moe_layer_forward_host": [ctypes.POINTER(MoeDesc), I32, P, P, P, P, P, P, P, P,
                                           P, P, P, P, SZ, P, P, P, P, P],
            }
            for name, args in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            L.moe_local_rerouting.argtypes = [P, P, I32, I32, I32, I32, P, P, P, P, P, P]
            L.moe_local_rerouting.restype = ctypes.c_int
            L.moe_local_finalize_rerouting.argtypes = [P, P, I32, I32, P, P]
            L.moe_local_finalize_rerouting.restype = ctypes.c_int
            L.moe_selftest_wait_timeout.argtypes = [P, P]
            L.moe_selftest_wait_timeout.restype = ctypes.c_int
            L.moe_status_string.argtypes = [ctypes.c_int]
            L.moe_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _call(name: str, *args):
    st = getattr(lib(), name)(*args)
    if st != MOE_OK:
        raise MoeError(name, st)


def _check(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def local_rerouting(recv_x, recv_counts, with_rows=True, status=None):
    """EP local step: -> dict(local_x, local_src, local_counts, local_offsets)."""
    _check(recv_x, torch.bfloat16, "recv_x")
    _check(recv_counts, torch.int32, "recv_counts")
    R, H = recv_x.shape
    ep, El = recv_counts.shape
    dev = recv_x.device
    lx = torch.empty_like(recv_x) if with_rows else None
    src = torch.empty(R, dtype=torch.int32, device=dev)
    lc = torch.empty(El, dtype=torch.int32, device=dev)
    lo = torch.empty(El + 1, dtype=torch.int32, device=dev)
    _call("moe_local_rerouting", _ptr(recv_x), _ptr(recv_counts), ep, El, R, H, _ptr(lx),
          _ptr(src), _ptr(lc), _ptr(lo), _ptr(status), _stream(dev))
    return dict(local_x=lx, local_src=src, local_counts=lc, local_offsets=lo)


def local_finalize_rerouting(local_y, local_src, recv_y=None):
    """EP local step: recv_y[local_src[d]] = local_y[d]."""
    _check(local_y, torch.bfloat16, "local_y")
    R, H = local_y.shape
    if recv_y is None:
        recv_y = torch.zeros_like(local_y)
    _call("moe_local_finalize_rerouting", _ptr(local_y), _ptr(local_src), R, H, _ptr(recv_y),
          _stream(local_y.device))
    return recv_y


def selftest_wait_timeout(status):
    """Enqueue the bounded-wait check (see include/moe.h); sets DEV_TIMEOUT."""
    _call("moe_selftest_wait_timeout", _ptr(status), _stream(status.device))


def new_status(device) -> torch.Tensor:
    """A zeroed device int32 for the MOE_DEV_* bits."""
    return torch.zeros(1, dtype=torch.int32, device=device)


# ----------------------------------------------------------------- operations
def rmsnorm_gate(x, wg, gamma=None, gate_bias=None, eps=1e-6, rmsnorm=True):
    """-> (xn or None, logits fp32 [T, E]); with wg None: (xn, None) from the
    RMSNorm-only pass."""
    _check(x, torch.bfloat16, "x")
    _check(wg, torch.float32, "wg")
    _check(gamma, torch.bfloat16, "gamma")
    _check(gate_bias, torch.float32, "gate_bias")
    T, H = x.shape
    if wg is None:
        xn = torch.empty_like(x)
        _call("moe_rmsnorm_gate", _ptr(x), _ptr(gamma), None, None, T, H, 1, float(eps),
              RMSNORM, _ptr(xn), None, _stream(x.device))
        return xn, None
    E = wg.shape[0]
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    xn = torch.empty_like(x) if rmsnorm else None
    _call("moe_rmsnorm_gate", _ptr(x), _ptr(gamma), _ptr(wg), _ptr(gate_bias), T, H, E,
          float(eps), RMSNORM if rmsnorm else 0, _ptr(xn), _ptr(logits), _stream(x.device))
    return xn, logits


def rmsnorm_sumsq(x):
    """-> float32 [T]: each row's sum of squares as the RMSNorm takes it (the
    exact sum of the bf16 squares rounded once to fp32)."""
    _check(x, torch.bfloat16, "x")
    T, H = x.shape
    ss = torch.empty(T, dtype=torch.float32, device=x.device)
    _call("moe_rmsnorm_sumsq", _ptr(x), T, H, _ptr(ss), _stream(x.device))
    return ss


def gate_tensor_workspace_size(T, H, E) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_gate_tensor_workspace_size", T, H, E, ctypes.byref(n))
    return n.value


def gate_tensor(xs, wg, gate_bias=None, workspace=None, status=None):
    """The tensor-core fp32 gate on already-normalised rows -> logits fp32 [T, E]."""
    _check(xs, torch.bfloat16, "xs")
    _check(wg, torch.float32, "wg")
    _check(gate_bias, torch.float32, "gate_bias")
    T, H = xs.shape
    E = wg.shape[0]
    logits = torch.empty((T, E), dtype=torch.float32, device=xs.device)
    need = gate_tensor_workspace_size(T, H, E)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=xs.device)
    _call("moe_gate_tensor", _ptr(xs), _ptr(wg), _ptr(gate_bias), T, H, E, _ptr(logits),
          _ptr(workspace), workspace.numel(), _ptr(status), _stream(xs.device))
    return logits


def gate_topk(logits, k, renorm=True):
    """-> (topk_idx int32 [T, k], topk_w fp32 [T, k])."""
    _check(logits, torch.float32, "logits")
    T, E = logits.shape
    idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _call("moe_gate_topk", _ptr(logits), T, E, k, RENORM if renorm else 0, _ptr(idx), _ptr(w),
          _stream(logits.device))
    return idx, w


def init_routing(topk_idx, x, E, with_rows=True, status=None):
    """-> dict(expanded_x, row_idx, src_token, sorted_ids, counts, offsets)."""
    _check(topk_idx, torch.int32, "topk_idx")
    _check(x, torch.bfloat16, "x")
    T, k = topk_idx.shape
    dev = topk_idx.device
    H = x.shape[1] if x is not None else 0
    N = T * k
    ex = torch.empty((N, H), dtype=torch.bfloat16, device=dev) if (with_rows and x is not None) \
        else None
    row_idx = torch.empty(N, dtype=torch.int32, device=dev)
    src = torch.empty(N, dtype=torch.int32, device=dev)
    sorted_ids = torch.empty(N, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    nbytes = ctypes.c_size_t(0)
    _call("moe_init_routing_workspace_size", T, k, E, ctypes.byref(nbytes))
    ws = torch.empty(max(nbytes.value, 256), dtype=torch.uint8, device=dev)
    _call("moe_init_routing", _ptr(topk_idx), _ptr(x if ex is not None else None), T, H, E, k,
          _ptr(ex), _ptr(row_idx), _ptr(src), _ptr(sorted_ids), _ptr(counts), _ptr(offsets),
          _ptr(ws), nbytes.value, _ptr(status), _stream(dev))
    return dict(expanded_x=ex, row_idx=row_idx, src_token=src, sorted_ids=sorted_ids,
                counts=counts, offsets=offsets)


def expert_tokens(sorted_ids, E, status=None):
    """-> (counts int32 [E], offsets int32 [E+1])."""
    _check(sorted_ids, torch.int32, "sorted_ids")
    dev = sorted_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    _call("moe_expert_tokens", _ptr(sorted_ids), sorted_ids.numel(), E, _ptr(counts),
          _ptr(offsets), _ptr(status), _stream(dev))
    return counts, offsets


def grouped_mlp(expanded_x, offsets, w13, w2, status=None):
    """-> (act bf16 [n, I], y bf16 [n, H])."""
    _check(expanded_x, torch.bfloat16, "expanded_x")
    _check(offsets, torch.int32, "offsets")
    _check(w13, torch.bfloat16, "w13")
    _check(w2, torch.bfloat16, "w2")
    n, H = expanded_x.shape
    G, I2, _ = w13.shape
    I = I2 // 2
    act = torch.zeros((n, I), dtype=torch.bfloat16, device=expanded_x.device)
    y = torch.zeros((n, H), dtype=torch.bfloat16, device=expanded_x.device)
    _call("moe_grouped_mlp", _ptr(expanded_x), _ptr(offsets), G, _ptr(w13), _ptr(w2), n, H, I,
          _ptr(act), _ptr(y), _ptr(status), _stream(expanded_x.device))
    return act, y


def finalize_routing(y_exp, row_idx, topk_w, shared=None, out_f32=False):
    """-> out [T, H] (bf16, or fp32 with out_f32).  y_exp bf16 or fp32."""
    if y_exp.dtype != torch.float32:
        _check(y_exp, torch.bfloat16, "y_exp")
    _check(row_idx, torch.int32, "row_idx")
    _check(topk_w, torch.float32, "topk_w")
    T, k = topk_w.shape
    H = y_exp.shape[1]
    flags = (OUT_F32 if out_f32 else 0) | (Y_F32 if y_exp.dtype == torch.float32 else 0)
    if shared is not None:
        if shared.dtype == torch.float32:
            flags |= SHARED_F32
        else:
            _check(shared, torch.bfloat16, "shared")
    out = torch.empty((T, H), dtype=torch.float32 if out_f32 else torch.bfloat16,
                      device=y_exp.device)
    _call("moe_finalize_routing", _ptr(y_exp), _ptr(row_idx), _ptr(topk_w), _ptr(shared), T, H,
          k, flags, _ptr(out), _stream(y_exp.device))
    return out


def make_desc(T, H, E, k, I, I_shared=0, rmsnorm=False, eps=1e-6, renorm=True,
              out_f32=False, gate_sequential=False, y_f32=False, gather_a=False) -> MoeDesc:
    """``gate_sequential``: the sequential fp32 gate (moe_rmsnorm_gate's
    logits, bit for bit) instead of the tensor-core gate for T > 512.
    ``y_f32``: the routed expert outputs enter the weighted sum as the down
    matmul's fp32 accumulator instead of rounded to bf16 (MOE_Y_F32).
    ``gather_a``: the routed w13 matmul reads its rows by source token, with
    no permute pass, where it runs as the wide pair kernel (MOE_GATHER_A)."""
    flags = (RENORM if renorm else 0) | (RMSNORM if rmsnorm else 0) | \
        (SHARED if I_shared > 0 else 0) | (OUT_F32 if out_f32 else 0) | \
        (GATE_SEQUENTIAL if gate_sequential else 0) | (Y_F32 if y_f32 else 0) | \
        (GATHER_A if gather_a else 0)
    return MoeDesc(T, H, E, k, I, I_shared, eps, flags)


def layer_workspace_size(desc: MoeDesc) -> int:
    n = ctypes.c_size_t(0)
    _call("moe_layer_workspace_size", ctypes.byref(desc), ctypes.byref(n))
    return n.value


@dataclasses.dataclass
class LayerWeights:
    wg: torch.Tensor
    w13: torch.Tensor
    w2: torch.Tensor
    gamma: Optional[torch.Tensor] = None
    gate_bias: Optional[torch.Tensor] = None
    w13_s: Optional[torch.Tensor] = None
    w2_s: Optional[torch.Tensor] = None


def layer_forward(desc: MoeDesc, x, weights: LayerWeights, out=None, workspace=None,
                  status=None, stage_events=None, shared_stream=None, events=None):
    """The whole MoE layer.  ``workspace`` (uint8, >= layer_workspace_size)
    and ``out`` are allocated when not given.  ``stage_events``: a list of
    NUM_STAGES + 1 recorded-once torch.cuda.Event (timing enabled) to time
    the internal stages.  ``shared_stream`` (a torch.cuda.Stream) with
    ``events`` (two recorded-once torch.cuda.Event) runs the shared expert on
    that stream.  Returns ``out``."""
    _check(x, torch.bfloat16, "x")
    dev = x.device
    if out is None:
        out = torch.empty((desc.T, desc.H),
                          dtype=torch.float32 if desc.flags & OUT_F32 else torch.bfloat16,
                          device=dev)
    nbytes = layer_workspace_size(desc)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    w = weights
    args = [ctypes.byref(desc), _ptr(x), _ptr(w.gamma), _ptr(w.wg), _ptr(w.gate_bias),
            _ptr(w.w13), _ptr(w.w2), _ptr(w.w13_s), _ptr(w.w2_s), _ptr(out), _ptr(workspace),
            workspace.numel(), _ptr(status), _stream(dev)]
    arr = None
    if stage_events is not None:
        assert len(stage_events) == NUM_STAGES + 1
        arr = (ctypes.c_void_p * (NUM_STAGES + 1))(*[e.cuda_event for e in stage_events])
    if shared_stream is not None:
        fork, join = events
        _call("moe_layer_forward_streams", *args, ctypes.c_void_p(shared_stream.cuda_stream),
              ctypes.c_void_p(fork.cuda_event), ctypes.c_void_p(join.cuda_event), arr)
    elif arr is None:
        _call("moe_layer_forward", *args)
    else:
        _call("moe_layer_forward_timed", *args, arr)
    return out


_host_pipes = {}


def _host_pipe(dev):
    """Per device: the two copy streams and six events of the host pipeline
    (created once; a torch event gets its CUDA handle on its first record)."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    pipe = _host_pipes.get(key)
    if pipe is None:
        with torch.cuda.device(key):
            cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
            evs = [torch.cuda.Event() for _ in range(6)]
            for e in evs:
                e.record(cin)
            cin.synchronize()
        pipe = _host_pipes[key] = (cin, cout, evs)
    return pipe


def layer_forward_host(desc: MoeDesc, x_host, weights: LayerWeights, out_host=None,
                       staging=None, workspace=None, status=None):
    """The layer on token batches in host memory (moe_layer_forward_host).
    ``x_host``: one [T, H] bf16 CPU tensor (pinned) or a list of them, one
    per batch; the outputs land in ``out_host`` (the same form; pinned CPU
    tensors are allocated when None).  Batch i+1's tokens are copied in and
    batch i-1's output copied out while batch i runs on the current stream.
    ``staging`` = (x_dev, out_dev): device tensors of 2*T*H elements
    (allocated when None).  Returns once the last output has arrived."""
    single = isinstance(x_host, torch.Tensor)
    xs = [x_host] if single else list(x_host)
    T, H = desc.T, desc.H
    odt = torch.float32 if desc.flags & OUT_F32 else torch.bfloat16
    for t in xs:
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or \
                tuple(t.shape) != (T, H):
            raise ValueError("x_host: contiguous [T, H] bf16 CPU tensors")
    if out_host is None:
        outs = [torch.empty((T, H), dtype=odt, pin_memory=True) for _ in xs]
    else:
        outs = [out_host] if single else list(out_host)
    if len(outs) != len(xs):
        raise ValueError("one output per batch")
    for t in outs:
        if t.is_cuda or t.dtype != odt or not t.is_contiguous() or tuple(t.shape) != (T, H):
            raise ValueError(f"out_host: contiguous [T, H] {odt} CPU tensors")
    dev = weights.w13.device
    if staging is None:
        staging = (torch.empty((2, T, H), dtype=torch.bfloat16, device=dev),
                   torch.empty((2, T, H), dtype=odt, device=dev))
    x_dev, out_dev = staging
    if x_dev.numel() < 2 * T * H or out_dev.numel() < 2 * T * H or out_dev.dtype != odt:
        raise ValueError("staging: (x_dev, out_dev) with 2*T*H elements each")
    if workspace is None:
        workspace = torch.empty(max(layer_workspace_size(desc), 256), dtype=torch.uint8,
                                device=dev)
    cin, cout, evs = _host_pipe(dev)
    cur = torch.cuda.current_stream(dev)
    cin.wait_stream(cur)          # staging buffers and workspace as the caller left them
    cout.wait_stream(cur)
    n = len(xs)
    xa = (ctypes.c_void_p * n)(*[t.data_ptr() for t in xs])
    oa = (ctypes.c_void_p * n)(*[t.data_ptr() for t in outs])
    ea = (ctypes.c_void_p * 6)(*[e.cuda_event for e in evs])
    w = weights
    _call("moe_layer_forward_host", ctypes.byref(desc), n, xa, oa, _ptr(w.gamma), _ptr(w.wg),
          _ptr(w.gate_bias), _ptr(w.w13), _ptr(w.w2), _ptr(w.w13_s), _ptr(w.w2_s),
          _ptr(x_dev), _ptr(out_dev), _ptr(workspace), workspace.numel(), _ptr(status),
          _stream(dev), ctypes.c_void_p(cin.cuda_stream), ctypes.c_void_p(cout.cuda_stream), ea)
    cout.synchronize()
    return outs[0] if single else outs
