"""GPU tests of the tensor-core gate (moe_gate_tensor; the layer's gate for
T > 512) against the oracle.

The gate of "NPU HunyuanImage-3.0模型推理优化实践" (section
"消除gate计算冗余cast算子") is an fp32 linear layer.  The tensor-core gate
splits every fp32 weight exactly into three bf16 parts and accumulates the
partial dot products in fp32, so its logits carry the same products as the
oracle's sequential fp32 sum, added in another order.  Checked here:
  - the split is exact: w1 + w2 + w3 == wg for every weight (read from the
    documented head of the workspace), padding rows zero;
  - logits within the fp32 rounding bound of the oracle's per element and
    far inside it in RMS (the bound is derived in tests/_helpers.py);
  - top-k on these logits equals the oracle's routing except at tokens where
    the oracle's own choice lies within that bound of a tie, and is a valid
    top-k there.
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe
import oracle
from moe_inputs import WORKLOADS, Workload, make_inputs
from tests._helpers import (bf16_to_f64, check_gate_tc_logits, gate_tc_bound, routing_flips,
                            u16)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # NW = 128: the one-CTA GEMM (fewer than 1024 rows)
    Workload("gt-e16", T=600, H=256, E=16, k=4, I=128, rmsnorm=True, gamma_std=0.1),
    # NW = 256 with a ragged row tail; gate offsets
    Workload("gt-e80-bias", T=777, H=384, E=80, k=5, I=128, skew_s=1.2, skew_beta=1.0),
    # NW = 256, >= 1024 rows: the CTA-pair GEMM, half tile at the end
    Workload("gt-e64-pair", T=2100, H=1024, E=64, k=8, I=128, rmsnorm=True, gamma_std=0.1),
    # the limits: 1024 experts (NW = 3072), 32 slots
    Workload("gt-e1024", T=530, H=128, E=1024, k=32, I=128),
    # a single token and few experts
    Workload("gt-one", T=1, H=128, E=4, k=1, I=128),
    # deep K: H = 8192
    Workload("gt-deep", T=1100, H=8192, E=24, k=4, I=128, x_std=1.0),
]


def _xs(d, wl):
    return oracle.rmsnorm(d["x"], d["gamma"], wl.eps) if wl.rmsnorm else u16(d["x"])


def _nw(E):
    return -(-3 * E // 128) * 128


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_gate_tensor_logits_and_routing(wl):
    d = make_inputs(wl, 5)
    xs_ref = _xs(d, wl)
    wg = d["wg"].to(DEV)
    bias = d["gate_bias"].to(DEV) if d["gate_bias"] is not None else None
    xs = d["x"].to(DEV)
    if wl.rmsnorm:
        xs, _ = moe.rmsnorm_gate(xs, wg, d["gamma"].to(DEV), bias, wl.eps)
    st = moe.new_status(DEV)
    ws = torch.full((moe.gate_tensor_workspace_size(wl.T, wl.H, wl.E),), 0x5A,
                    dtype=torch.uint8, device=DEV)
    lg = moe.gate_tensor(xs, wg, bias, workspace=ws, status=st)
    idx, w = moe.gate_topk(lg, wl.k, wl.renorm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(u16(xs), xs_ref)

    # the split weight heads the workspace: [NW, H] bf16, part p in rows [pE, (p+1)E)
    NW = _nw(wl.E)
    split = bf16_to_f64(u16(ws[:NW * wl.H * 2].view(torch.bfloat16).view(NW, wl.H)))
    wg64 = d["wg"].numpy().astype(np.float64)
    E = wl.E
    assert np.array_equal(split[:E] + split[E:2 * E] + split[2 * E:3 * E], wg64)
    assert not split[3 * E:].any()

    lg_ref = oracle.gate_logits(xs_ref, d["wg"], d["gate_bias"])
    per, rms_b = gate_tc_bound(xs_ref, d["wg"], lg_ref)
    mx, rms = check_gate_tc_logits(lg.cpu().numpy(), lg_ref, per, rms_b, wl.name)
    ridx, rw = oracle.topk_softmax(lg_ref, wl.k, wl.renorm)
    flips = routing_flips(idx.cpu().numpy(), ridx, lg_ref, per)
    keep = np.setdiff1d(np.arange(wl.T), flips)
    # weights: softmax of logits within `per` of the oracle's moves by at most
    # 2 max|dl| relatively (plus the top-k kernel's own rounding)
    tol = 2 * per.max(axis=1, keepdims=True) + 2e-6
    got_w = w.cpu().numpy()[keep]
    same = (idx.cpu().numpy()[keep] == ridx[keep]).all(axis=1)
    assert (np.abs(got_w[same] - rw[keep][same]) <= tol[keep][same] * np.abs(rw[keep][same])
            + 2e-7).all()
    print(f"{wl.name}: max |dlogit| {mx:.3g}, rms {rms:.3g} (bound {rms_b:.3g}), "
          f"{len(flips)} ambiguous tokens")


def test_gate_tensor_empty_and_errors():
    wl = CASES[0]
    d = make_inputs(wl, 1, T=0)
    xs = d["x"].to(DEV)
    lg = moe.gate_tensor(xs, d["wg"].to(DEV))
    assert lg.shape == (0, wl.E)
    # H not a multiple of 128: refused before any launch
    with pytest.raises(moe.MoeError):
        moe.gate_tensor_workspace_size(4, 192, 8)
    # a workspace one byte short
    d = make_inputs(wl, 1, T=8)
    need = moe.gate_tensor_workspace_size(8, wl.H, wl.E)
    ws = torch.empty(need - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoeError):
        moe.gate_tensor(d["x"].to(DEV), d["wg"].to(DEV), workspace=ws)


@pytest.mark.parametrize("name,seed", [("imagegen-16k", 0), ("skewed-32k", 0),
                                       ("skewed-32k", 1)])
def test_gate_tensor_full_size(name, seed):
    """The gate at the benchmark's sizes, every logit checked.  (Seed 1 of the
    skewed load has a token whose top-8 boundary is within rounding of a tie:
    its other valid choice is checked for validity.)"""
    wl = WORKLOADS[name]
    g = make_inputs(wl, seed, device=DEV, only=("x", "gamma", "wg", "gate_bias"))
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}
    if wl.rmsnorm:
        xn, _ = moe.rmsnorm_gate(g["x"], g["wg"], g["gamma"], g["gate_bias"], wl.eps)
        xs = xn
    else:
        xs = g["x"]
    lg = moe.gate_tensor(xs, g["wg"], g["gate_bias"])
    idx, _ = moe.gate_topk(lg, wl.k, wl.renorm)
    torch.cuda.synchronize()
    xs_ref = oracle.rmsnorm(cpu["x"], cpu["gamma"], wl.eps) if wl.rmsnorm else u16(cpu["x"])
    assert np.array_equal(u16(xs), xs_ref)
    lg_ref = oracle.gate_logits(xs_ref, cpu["wg"], cpu["gate_bias"])
    per, rms_b = gate_tc_bound(xs_ref, cpu["wg"], lg_ref)
    mx, rms = check_gate_tc_logits(lg.cpu().numpy(), lg_ref, per, rms_b, name)
    ridx, _ = oracle.topk_softmax(lg_ref, wl.k, wl.renorm)
    flips = routing_flips(idx.cpu().numpy(), ridx, lg_ref, per)
    print(f"{name}: max |dlogit| {mx:.3g}, rms {rms:.3g} (bound {rms_b:.3g}), "
          f"{len(flips)} of {wl.T} tokens chose another valid set")
