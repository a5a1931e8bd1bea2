"""EP DoubleRouting local steps ("MoE EP优化": LocalRerouting and
LocalFinalizeRerouting) on the GPU: parity with the oracle on synthetic
received buffers, and a two-rank expert-parallel pass emulated on one GPU
(the all_to_all exchanges are done with torch indexing, as test plumbing)
that must reproduce the single-rank layer bit for bit.
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe
import oracle
from moe_inputs import Workload, make_inputs
from tests._helpers import u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("ep,El,H,slack", [(4, 6, 64, 5), (8, 16, 256, 0), (1, 3, 128, 2),
                                           (16, 64, 128, 33)])
def test_local_rerouting_parity(ep, El, H, slack):
    rng = np.random.default_rng(ep * 100 + El)
    counts = rng.integers(0, 9, (ep, El)).astype(np.int32)
    counts[rng.integers(0, ep)] = 0              # a rank that sent nothing
    total = int(counts.sum())
    R = total + slack
    x = torch.randn((R, H)).to(torch.bfloat16)
    st = moe.new_status(DEV)
    r = moe.local_rerouting(x.to(DEV), torch.from_numpy(counts).to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    lx, src, lc, lo = oracle.local_rerouting(x, counts)
    assert np.array_equal(r["local_src"].cpu().numpy(), src)
    assert np.array_equal(u16(r["local_x"])[:total], lx[:total])
    assert np.array_equal(r["local_counts"].cpu().numpy(), lc)
    assert np.array_equal(r["local_offsets"].cpu().numpy(), lo)
    # back to the received order
    back = moe.local_finalize_rerouting(r["local_x"], r["local_src"])
    assert torch.equal(back[:total].view(torch.int16), x[:total].to(DEV).view(torch.int16))


def test_local_rerouting_bad_counts_reported():
    counts = torch.tensor([[3, 2], [4, 1]], dtype=torch.int32, device=DEV)   # 10 rows
    x = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)               # capacity 8
    st = moe.new_status(DEV)
    moe.local_rerouting(x, counts, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_OFFSETS


def test_two_rank_expert_parallel_matches_single_rank():
    wl = Workload("ep2", T=512, H=256, E=16, k=4, I=256, rmsnorm=True, gamma_std=0.1)
    d = make_inputs(wl, 5)
    g = {kk: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for kk, v in d.items()}
    ep, El = 2, wl.E // 2
    # reference: the whole layer on one rank
    desc = moe.make_desc(wl.T, wl.H, wl.E, wl.k, wl.I, rmsnorm=True, eps=wl.eps, out_f32=True)
    w = moe.LayerWeights(wg=g["wg"], w13=g["w13"], w2=g["w2"], gamma=g["gamma"])
    ref = moe.layer_forward(desc, g["x"], w)

    Tr = wl.T // ep
    ranks = []
    for r in range(ep):                          # per-rank gate, top-k, init_routing
        xr = g["x"][r * Tr:(r + 1) * Tr].contiguous()
        xn, lg = moe.rmsnorm_gate(xr, g["wg"], g["gamma"], None, wl.eps, rmsnorm=True)
        idx, wt = moe.gate_topk(lg, wl.k)
        rt = moe.init_routing(idx, xn, wl.E)
        ranks.append(dict(idx=idx, w=wt, **rt))
    # token all_to_all: rank r sends its rows of experts [d*El, (d+1)*El) to rank d
    outs_recv = []
    for dst in range(ep):
        parts, cnts = [], []
        for r in range(ep):
            off = ranks[r]["offsets"].cpu()
            a, b = int(off[dst * El]), int(off[(dst + 1) * El])
            parts.append(ranks[r]["expanded_x"][a:b])
            cnts.append(ranks[r]["counts"][dst * El:(dst + 1) * El])
        recv_x = torch.cat(parts).contiguous()
        recv_counts = torch.stack(cnts).contiguous()
        st = moe.new_status(DEV)
        lr = moe.local_rerouting(recv_x, recv_counts, status=st)
        _, y_local = moe.grouped_mlp(lr["local_x"], lr["local_offsets"],
                                     g["w13"][dst * El:(dst + 1) * El].contiguous(),
                                     g["w2"][dst * El:(dst + 1) * El].contiguous(), status=st)
        y_recv = moe.local_finalize_rerouting(y_local, lr["local_src"])
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs_recv.append((y_recv, [p.shape[0] for p in parts]))
    # return all_to_all, then FinalizeRouting on each rank
    outs = []
    for r in range(ep):
        back = []
        for dst in range(ep):
            y_recv, sizes = outs_recv[dst]
            a = sum(sizes[:r])
            back.append(y_recv[a:a + sizes[r]])
        y_exp = torch.cat(back).contiguous()           # rank r's rows in its sorted order
        outs.append(moe.finalize_routing(y_exp, ranks[r]["row_idx"], ranks[r]["w"],
                                         out_f32=True))
    got = torch.cat(outs)
    assert torch.equal(got, ref)
