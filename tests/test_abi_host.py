"""Host-side checks of the C ABI that need no GPU: the library loads, it
exports every entry point include/moe.h declares, and argument errors are
reported as status codes before any CUDA work is attempted.

(The failure-detection pattern: the fault is made on the host, here an
invalid argument, and the test checks the reported status.)
"""
import ctypes
import os
import re

import pytest

import moe_expert_routing_fp32_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    moe.build()
    return moe.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert set(names) == set(moe.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in moe.STATUS_NAMES.items():
        assert L.moe_status_string(code).decode() == name
    assert L.moe_status_string(99).decode() == "MOE_ERR_UNKNOWN"


def test_invalid_arguments_rejected_on_host(L):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # k > E, E > 1024, negative sizes
    assert L.moe_gate_topk(fake, 4, 4, 5, 0, fake, fake, None) == 2
    assert L.moe_gate_topk(fake, 4, 2000, 2, 0, fake, fake, None) == 2
    assert L.moe_gate_topk(fake, -1, 8, 2, 0, fake, fake, None) == 1
    # null outputs
    assert L.moe_gate_topk(fake, 4, 8, 2, 0, None, fake, None) == 1
    # H not a multiple of 64 / misaligned x
    assert L.moe_rmsnorm_gate(fake, None, fake, None, 4, 100, 8, 1e-6, 0, None, fake, None) == 2
    assert L.moe_rmsnorm_gate(P(0x1002), None, fake, None, 4, 128, 8, 1e-6, 0, None, fake,
                              None) == 1
    # RMSNorm without xn
    assert L.moe_rmsnorm_gate(fake, None, fake, None, 4, 128, 8, 1e-6, moe.RMSNORM, None, fake,
                              None) == 1
    # grouped mlp: I not a multiple of 128, too many groups
    assert L.moe_grouped_mlp(fake, fake, 4, fake, fake, 10, 128, 96, fake, fake, None, None) == 2
    assert L.moe_grouped_mlp(fake, fake, 2000, fake, fake, 10, 128, 128, fake, fake, None,
                             None) == 2
    # init_routing: workspace too small
    n = ctypes.c_size_t()
    assert L.moe_init_routing_workspace_size(100, 2, 8, ctypes.byref(n)) == 0
    assert n.value >= 4 * 8 * 4
    assert L.moe_init_routing(fake, None, 100, 0, 8, 2, None, fake, fake, None, fake, fake,
                              fake, n.value - 1, None, None) == 3
    # finalize: H % 8
    assert L.moe_finalize_routing(fake, fake, fake, None, 4, 12, 2, 0, fake, None) == 2
    # tensor-core gate: H % 128, E <= 1024, workspace size, alignment
    assert L.moe_gate_tensor_workspace_size(4, 192, 8, ctypes.byref(n)) == 2
    assert L.moe_gate_tensor_workspace_size(4, 128, 2000, ctypes.byref(n)) == 2
    assert L.moe_gate_tensor_workspace_size(600, 256, 16, ctypes.byref(n)) == 0
    # the split weight [128, 256] bf16, then the partial logits [600, 128] fp32
    assert n.value == 128 * 256 * 2 + 600 * 128 * 4
    assert L.moe_gate_tensor(fake, fake, None, 600, 256, 16, fake, fake, n.value - 1, None,
                             None) == 3
    assert L.moe_gate_tensor(P(0x1002), fake, None, 600, 256, 16, fake, fake, n.value, None,
                             None) == 1
    assert L.moe_gate_tensor(fake, fake, None, 600, 256, 16, None, fake, n.value, None,
                             None) == 1
    # the RMSNorm-only form of moe_rmsnorm_gate: H % 128, xn and the flag required
    assert L.moe_rmsnorm_gate(fake, None, None, None, 4, 192, 1, 1e-6, moe.RMSNORM, fake, None,
                              None) == 2
    assert L.moe_rmsnorm_gate(fake, None, None, None, 4, 256, 1, 1e-6, moe.RMSNORM, None, None,
                              None) == 1
    assert L.moe_rmsnorm_gate(fake, None, None, None, 4, 256, 1, 1e-6, 0, fake, None,
                              None) == 1


def test_layer_desc_checks(L):
    d = moe.make_desc(T=16, H=100, E=8, k=2, I=128)
    n = ctypes.c_size_t()
    assert L.moe_layer_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 2
    d = moe.make_desc(T=16, H=128, E=8, k=9, I=128)
    assert L.moe_layer_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 2
    d = moe.make_desc(T=16, H=128, E=8, k=2, I=128, I_shared=128, rmsnorm=True)
    assert L.moe_layer_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 0
    # xn + idx + w + row_idx + act + y + act_s + y_s (+ hist, counts, offsets and
    # expanded_x)
    assert n.value >= 16 * 128 * 2 + 3 * 32 * 4 + 32 * 128 * 2 * 2 + 16 * 128 * 6
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert L.moe_layer_forward(ctypes.byref(d), fake, None, fake, None, fake, fake, fake, fake,
                               fake, fake, n.value - 256, None, None) == 3
    assert L.moe_layer_forward(ctypes.byref(d), fake, None, fake, None, fake, fake, None, None,
                               fake, fake, n.value, None, None) == 1   # shared weights missing


def test_no_device_is_an_error_not_a_fallback(L):
    """Valid arguments on a machine without a usable GPU fail loudly."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert L.moe_gate_topk(fake, 4, 8, 2, 0, fake, fake, None) == 5


def _ws(L, desc):
    n = ctypes.c_size_t(0)
    assert L.moe_layer_workspace_size(ctypes.byref(desc), ctypes.byref(n)) == 0
    return n.value


def test_gathered_rows_change_the_workspace_only_where_they_apply(L):
    """MOE_GATHER_A drops expanded_x from the layer workspace (its N x H
    bf16 rows) and adds the source-token array (N int32), but only where the
    w13 matmul runs on the wide pair kernel (>= 1024 rows per expert on
    average, I a multiple of 256); elsewhere the flag is ignored."""
    if os.environ.get("MOE_GEMM_KERNEL"):
        pytest.skip("kernel choice forced in the environment")
    T, H, E, k, I = 16384, 4096, 64, 8, 3072                 # 2048 rows per expert
    N = T * k
    plain = _ws(L, moe.make_desc(T, H, E, k, I, I, rmsnorm=True))
    gath = _ws(L, moe.make_desc(T, H, E, k, I, I, rmsnorm=True, gather_a=True))
    assert plain - gath >= N * H * 2 - N * 4 - 512            # alignment slack
    T, H, I = 4096, 2048, 1024                                # 512 rows per expert
    plain = _ws(L, moe.make_desc(T, H, E, k, I))
    gath = _ws(L, moe.make_desc(T, H, E, k, I, gather_a=True))
    assert plain == gath
