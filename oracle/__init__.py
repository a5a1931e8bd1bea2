"""CPU oracle of the MoE feed-forward layer (ctypes binding of moe_oracle.c).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA library and never imports it.

Every function takes and returns numpy arrays; bf16 tensors travel as uint16
bit patterns (``bf16_bits`` / ``bits_to_float`` convert).  See moe_oracle.c
for the definitions each function follows and the page sections they cite.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, BAD_ARG, BAD_EXPERT, NOMEM = 0, 1, 2, 3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile moe_oracle.c with gcc (OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    INT = ctypes.c_int
    F = ctypes.c_float
    sigs = {
        "oracle_rmsnorm": [P, P, I64, I64, F, P],
        "oracle_sumsq": [P, I64, I64, P],
        "oracle_gate_logits": [P, P, P, I64, I64, I64, P],
        "oracle_topk_softmax": [P, I64, I64, I64, INT, P, P],
        "oracle_init_routing": [P, I64, I64, I64, P, P, P, P, P],
        "oracle_expert_tokens": [P, I64, I64, P, P],
        "oracle_permute": [P, P, I64, I64, P],
        "oracle_expert_mlp": [P, I64, P, P, I64, I64, P, P, P],
        "oracle_grouped_mlp": [P, P, I64, P, P, I64, I64, P, P],
        "oracle_finalize": [P, P, P, P, I64, I64, I64, P],
        "oracle_finalize_f64": [P, P, P, P, I64, I64, I64, P],
        "oracle_layer_tokens": [P, I64, I64, I64, I64, I64, I64, INT, F, INT,
                                P, P, P, P, P, P, P, P, I64, P, P, P, P, P],
        "oracle_local_rerouting": [P, P, I64, I64, I64, I64, P, P, P, P],
        "oracle_local_finalize_rerouting": [P, P, I64, I64, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    for name in ("oracle_bf16_round", "oracle_bf16_to_float"):
        fn = getattr(lib, name)
        fn.argtypes = [P, I64, P]
        fn.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this module to another build of the oracle source
    (the mutation tests plant a mistake in a copy and load it here)."""
    global _lib
    _load()
    with _lock:
        old = _lib
        _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = old


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != OK:
        raise OracleError(f"{name} returned {rc}")


def _u16(a):
    """Accept a torch bf16 tensor or a uint16 array; return a uint16 array."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16
            return np.ascontiguousarray(
                a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def _arr(a, dtype):
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- bf16 helpers
def bf16_bits(values) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even); uint16 bits."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_round(_p(v), v.size, _p(out))
    return out


def bits_to_float(bits) -> np.ndarray:
    b = _u16(bits)
    out = np.empty(b.shape, dtype=np.float32)
    _load().oracle_bf16_to_float(_p(b), b.size, _p(out))
    return out


# ---------------------------------------------------------------- layer steps
def rmsnorm(x, gamma, eps):
    x = _u16(x)
    T, H = x.shape
    g = _u16(gamma)
    out = np.empty_like(x)
    _check(_load().oracle_rmsnorm(_p(x), _p(g), T, H, ctypes.c_float(eps), _p(out)),
           "oracle_rmsnorm")
    return out


def sumsq(x):
    """The RMSNorm's row sums of squares: the exact sum of the bf16 squares
    of each row, rounded once to fp32 -> float32 [T]."""
    x = _u16(x)
    T, H = x.shape
    out = np.empty(T, dtype=np.float32)
    _check(_load().oracle_sumsq(_p(x), T, H, _p(out)), "oracle_sumsq")
    return out


def gate_logits(xs, wg, bias=None):
    xs = _u16(xs)
    T, H = xs.shape
    wg = _arr(wg, np.float32)
    E = wg.shape[0]
    b = _arr(bias, np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _check(_load().oracle_gate_logits(_p(xs), _p(wg), _p(b), T, H, E, _p(out)),
           "oracle_gate_logits")
    return out


def topk_softmax(logits, k, renorm=True):
    lg = _arr(logits, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    _check(_load().oracle_topk_softmax(_p(lg), T, E, k, int(bool(renorm)), _p(idx), _p(w)),
           "oracle_topk_softmax")
    return idx, w


def init_routing(topk_idx, E):
    ti = _arr(topk_idx, np.int32)
    T, k = ti.shape
    N = T * k
    row_idx = np.empty(N, dtype=np.int32)
    src = np.empty(N, dtype=np.int32)
    sorted_ids = np.empty(N, dtype=np.int32)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    _check(_load().oracle_init_routing(_p(ti), T, k, E, _p(row_idx), _p(src),
                                       _p(sorted_ids), _p(counts), _p(offsets)),
           "oracle_init_routing")
    return dict(row_idx=row_idx, src_token=src, sorted_ids=sorted_ids,
                counts=counts, offsets=offsets)


def expert_tokens(sorted_ids, E):
    ids = _arr(sorted_ids, np.int32).reshape(-1)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    _check(_load().oracle_expert_tokens(_p(ids), ids.size, E, _p(counts), _p(offsets)),
           "oracle_expert_tokens")
    return counts, offsets


def permute(xs, src_token):
    xs = _u16(xs)
    H = xs.shape[1]
    src = _arr(src_token, np.int32).reshape(-1)
    out = np.empty((src.size, H), dtype=np.uint16)
    _check(_load().oracle_permute(_p(xs), _p(src), src.size, H, _p(out)),
           "oracle_permute")
    return out


def expert_mlp(xe, w13, w2, want_f64=False):
    xe = _u16(xe)
    n, H = xe.shape
    w13 = _u16(w13)
    w2 = _u16(w2)
    I = w13.shape[0] // 2
    act = np.empty((n, I), dtype=np.uint16)
    yb = np.empty((n, H), dtype=np.uint16)
    yf = np.empty((n, H), dtype=np.float64) if want_f64 else None
    _check(_load().oracle_expert_mlp(_p(xe), n, _p(w13), _p(w2), H, I, _p(act), _p(yb),
                                     _p(yf)), "oracle_expert_mlp")
    return (act, yb, yf) if want_f64 else (act, yb)


def grouped_mlp(expanded_x, offsets, w13, w2):
    ex = _u16(expanded_x)
    n, H = ex.shape
    off = _arr(offsets, np.int32)
    G = off.size - 1
    w13 = _u16(w13)
    w2 = _u16(w2)
    I = w13.shape[1] // 2
    act = np.zeros((n, I), dtype=np.uint16)
    y = np.zeros((n, H), dtype=np.uint16)
    _check(_load().oracle_grouped_mlp(_p(ex), _p(off), G, _p(w13), _p(w2), H, I,
                                      _p(act), _p(y)), "oracle_grouped_mlp")
    return act, y


def finalize(y_exp, row_idx, topk_w, shared=None):
    """Weighted sum of the routed rows: bf16 rows (uint16 bits or a torch bf16
    tensor), or unrounded rows as a float64 array (the fp32-y reading)."""
    w = _arr(topk_w, np.float32)
    T, k = w.shape
    ri = _arr(row_idx, np.int32).reshape(-1)
    sh = _arr(shared, np.float64)
    if isinstance(y_exp, np.ndarray) and y_exp.dtype == np.float64:
        y = np.ascontiguousarray(y_exp)
        H = y.shape[1]
        out = np.empty((T, H), dtype=np.float64)
        _check(_load().oracle_finalize_f64(_p(y), _p(ri), _p(w), _p(sh), T, H, k, _p(out)),
               "oracle_finalize_f64")
        return out
    y = _u16(y_exp)
    H = y.shape[1]
    out = np.empty((T, H), dtype=np.float64)
    _check(_load().oracle_finalize(_p(y), _p(ri), _p(w), _p(sh), T, H, k, _p(out)),
           "oracle_finalize")
    return out


def layer_tokens(inputs: dict, wl, tokens=None, routed_rows=False, y_f32=False):
    """Whole layer for ``tokens`` (default: all).  ``inputs`` is the dict made
    by moe_inputs.make_inputs; ``wl`` the Workload.  Returns (out f64 [n,H],
    topk_idx [n,k], topk_w [n,k]), and with ``routed_rows`` also each slot's
    routed expert output as bf16 bits [n,k,H].  ``y_f32``: ``out`` is the
    fp32-y reading (routed expert outputs enter the weighted sum unrounded)."""
    out, out_yf, idx, w, y = _layer(inputs, wl, tokens, routed_rows, y_f32)
    o = out_yf if y_f32 else out
    return (o, idx, w, y) if routed_rows else (o, idx, w)


def layer_tokens_both(inputs: dict, wl, tokens=None):
    """One pass of the layer giving both readings: (out with bf16 routed
    outputs, out with unrounded routed outputs, topk_idx, topk_w, routed
    rows as bf16 bits [n,k,H])."""
    return _layer(inputs, wl, tokens, True, True)


def _layer(inputs, wl, tokens, routed_rows, want_yf):
    x = _u16(inputs["x"])
    T, H = x.shape
    E, k, I, I_s = wl.E, wl.k, wl.I, wl.I_s
    tok = None if tokens is None else _arr(tokens, np.int32).reshape(-1)
    n = T if tok is None else tok.size
    out = np.empty((n, H), dtype=np.float64)
    out_yf = np.empty((n, H), dtype=np.float64) if want_yf else None
    idx = np.empty((n, k), dtype=np.int32)
    w = np.empty((n, k), dtype=np.float32)
    y = np.empty((n, k, H), dtype=np.uint16) if routed_rows else None
    gamma = _u16(inputs.get("gamma"))
    wg = _arr(inputs["wg"], np.float32)
    bias = _arr(inputs.get("gate_bias"), np.float32)
    w13 = _u16(inputs["w13"])
    w2 = _u16(inputs["w2"])
    w13_s = _u16(inputs.get("w13_s")) if I_s > 0 else None
    w2_s = _u16(inputs.get("w2_s")) if I_s > 0 else None
    rc = _load().oracle_layer_tokens(
        _p(x), T, H, E, k, I, I_s, int(wl.rmsnorm), ctypes.c_float(wl.eps),
        int(wl.renorm), _p(gamma), _p(wg), _p(bias), _p(w13), _p(w2), _p(w13_s),
        _p(w2_s), _p(tok), 0 if tok is None else tok.size, _p(out), _p(idx), _p(w), _p(y),
        _p(out_yf))
    _check(rc, "oracle_layer_tokens")
    return out, out_yf, idx, w, y


# ------------------------------------------------------------ EP local steps
def local_rerouting(recv_x, counts):
    """counts [ep, E_local] (rows per source rank and local expert), recv_x
    [R, H] in arrival order.  Returns (local_x, local_src, local_counts,
    local_offsets)."""
    x = _u16(recv_x)
    R, H = x.shape
    c = _arr(counts, np.int32)
    ep, El = c.shape
    lx = np.zeros_like(x)
    src = np.full(R, -1, dtype=np.int32)
    lc = np.empty(El, dtype=np.int32)
    lo = np.empty(El + 1, dtype=np.int32)
    _check(_load().oracle_local_rerouting(_p(x), _p(c), ep, El, R, H, _p(lx), _p(src), _p(lc),
                                          _p(lo)), "oracle_local_rerouting")
    return lx, src, lc, lo


def local_finalize_rerouting(local_y, local_src, n, R):
    """recv_y[local_src[d]] = local_y[d] for d < n; returns recv_y [R, H]."""
    y = _u16(local_y)
    H = y.shape[1]
    src = _arr(local_src, np.int32)
    out = np.zeros((R, H), dtype=np.uint16)
    _check(_load().oracle_local_finalize_rerouting(_p(y), _p(src), n, H, _p(out)),
           "oracle_local_finalize_rerouting")
    return out
