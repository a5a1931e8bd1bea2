"""MoE tensor parallelism ("MoE TP优化 / 切分策略": gate_proj and up_proj split
by columns and merged per rank into that rank's w13, down_proj split by
rows) as a single-GPU workload: each TP shard runs the layer on its I/tp
slice of every expert (and of the shared expert) and yields a partial
output; the TP all-reduce is the sum of the shards' fp32 outputs.  Routing
(gate, top-k, init/finalize) is replicated on every shard, as on the page.
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe
import oracle
from moe_inputs import Workload, make_inputs
from tests._helpers import check_out, t2f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def tp_shard(g, wl, tp, rank):
    """Rank `rank`'s weights: its I/tp columns of gate and of up, merged into
    one w13 [E, 2I/tp, H]; its I/tp input columns of down [E, H, I/tp]."""
    I, Is = wl.I, wl.I_s
    i0, i1 = rank * I // tp, (rank + 1) * I // tp
    w13 = torch.cat([g["w13"][:, i0:i1], g["w13"][:, I + i0:I + i1]], dim=1).contiguous()
    w2 = g["w2"][:, :, i0:i1].contiguous()
    w13_s = w2_s = None
    if Is:
        s0, s1 = rank * Is // tp, (rank + 1) * Is // tp
        w13_s = torch.cat([g["w13_s"][s0:s1], g["w13_s"][Is + s0:Is + s1]]).contiguous()
        w2_s = g["w2_s"][:, s0:s1].contiguous()
    return w13, w2, w13_s, w2_s


@pytest.mark.parametrize("tp", [2, 4])
def test_tp_shards_sum_to_full_layer(tp):
    wl = Workload("tp", T=300, H=256, E=16, k=4, I=512, I_s=512, rmsnorm=True, gamma_std=0.1)
    d = make_inputs(wl, 9)
    g = {kk: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for kk, v in d.items()}
    ref, _, _ = oracle.layer_tokens(d, wl)
    total = torch.zeros((wl.T, wl.H), dtype=torch.float32, device=DEV)
    for rank in range(tp):
        w13, w2, w13_s, w2_s = tp_shard(g, wl, tp, rank)
        desc = moe.make_desc(wl.T, wl.H, wl.E, wl.k, wl.I // tp, wl.I_s // tp, rmsnorm=True,
                             eps=wl.eps, out_f32=True)
        w = moe.LayerWeights(wg=g["wg"], w13=w13, w2=w2, gamma=g["gamma"], w13_s=w13_s,
                             w2_s=w2_s)
        st = moe.new_status(DEV)
        total += moe.layer_forward(desc, g["x"], w, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
    check_out(t2f64(total), ref, bf16_out=False, what=f"tp={tp}")
    # each shard's act equals the matching slice of the full act exactly
    full_act, _ = moe.grouped_mlp(*_routed(g, wl), g["w13"], g["w2"])
    for rank in range(tp):
        w13, w2, _, _ = tp_shard(g, wl, tp, rank)
        act, _ = moe.grouped_mlp(*_routed(g, wl), w13, w2)
        i0, i1 = rank * wl.I // tp, (rank + 1) * wl.I // tp
        assert torch.equal(act, full_act[:, i0:i1])


def _routed(g, wl):
    xn, lg = moe.rmsnorm_gate(g["x"], g["wg"], g["gamma"], None, wl.eps, rmsnorm=True)
    idx, _ = moe.gate_topk(lg, wl.k)
    r = moe.init_routing(idx, xn, wl.E)
    return r["expanded_x"], r["offsets"]
