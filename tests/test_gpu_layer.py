"""GPU parity of the whole layer (moe_layer_forward through the C ABI)
against the CPU oracle.

Small workloads are compared on every token.  The full-size workloads
(T=4096 balanced, T=16384 image-gen block, T=32768 skewed, small batches)
are run exactly as the benchmark runs them; the oracle recomputes the gate,
top-k and routing for every token (bit-exact comparison of the step entry
points on the same inputs) and the layer output for every token of the
balanced and small-batch loads and 2048 tokens of the two large ones.

Two readings of the routed expert outputs are checked.  With MOE_Y_F32 the
down matmul's fp32 accumulator enters the weighted sum (the oracle keeps it
unrounded): the output must meet max-abs 2e-2 and rel-L2 5e-3 with no other
allowance.  Without it both sides round each routed output to bf16 first;
where the two fp32/exact sums straddle a bf16 rounding boundary they land one
ulp apart, so that check admits, on rare elements, one bf16 ulp of each
routed term (routed_flip_allowance).
Inputs of the full-size workloads are drawn on the GPU by the seeded
generator and copied to the host for the oracle.

Above 512 tokens the layer's gate is the tensor-core one (moe_gate_tensor):
fp32-accurate logits in another summation order than the oracle's.  Its
routing is compared with the oracle's through the step entry points; a
token whose oracle choice lies within the fp32 rounding bound of a tie may
take another valid set of experts (checked for validity) and is then left
out of the output comparison.  The same layer with MOE_GATE_SEQUENTIAL
(the oracle's summation order) is compared on every token.
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe
import oracle
from moe_inputs import WORKLOADS, Workload, make_inputs
from tests._helpers import (check_gate_tc_logits, check_out, gate_tc_bound, routed_flip_allowance,
                            routing_flips, t2f64, u16)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _weights(g):
    return moe.LayerWeights(wg=g["wg"], w13=g["w13"], w2=g["w2"], gamma=g["gamma"],
                            gate_bias=g["gate_bias"], w13_s=g["w13_s"], w2_s=g["w2_s"])


def _desc(wl, T=None, out_f32=True, seq=False, y_f32=False, gather_a=False):
    return moe.make_desc(wl.T if T is None else T, wl.H, wl.E, wl.k, wl.I, wl.I_s,
                         rmsnorm=wl.rmsnorm, eps=wl.eps, renorm=wl.renorm, out_f32=out_f32,
                         gate_sequential=seq, y_f32=y_f32, gather_a=gather_a)


def _run_layer(wl, g, out_f32, T=None, seq=False, y_f32=False, gather_a=False):
    st = moe.new_status(DEV)
    out = moe.layer_forward(_desc(wl, T, out_f32, seq, y_f32, gather_a), g["x"], _weights(g),
                            status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return out


def _tc_flips(wl, g, cpu, xs_ref=None, lg_ref=None, ridx=None):
    """Tokens for which the tensor-core gate (the layer's gate for T > 512)
    picks another valid set of experts than the oracle; empty for T <= 512.
    Also checks its logits against the oracle's within the rounding bound."""
    if wl.T <= 512:
        return np.zeros(0, dtype=np.int64)
    if xs_ref is None:
        xs_ref = oracle.rmsnorm(cpu["x"], cpu["gamma"], wl.eps) if wl.rmsnorm else u16(cpu["x"])
    if lg_ref is None:
        lg_ref = oracle.gate_logits(xs_ref, cpu["wg"], cpu["gate_bias"])
    if ridx is None:
        ridx, _ = oracle.topk_softmax(lg_ref, wl.k, wl.renorm)
    xs = g["x"]
    if wl.rmsnorm:
        xs, _ = moe.rmsnorm_gate(g["x"], g["wg"], g["gamma"], g["gate_bias"], wl.eps)
    lg = moe.gate_tensor(xs, g["wg"], g["gate_bias"])
    idx, _ = moe.gate_topk(lg, wl.k, wl.renorm)
    torch.cuda.synchronize()
    assert np.array_equal(u16(xs), xs_ref)
    per, rms_b = gate_tc_bound(xs_ref, cpu["wg"], lg_ref)
    check_gate_tc_logits(lg.cpu().numpy(), lg_ref, per, rms_b, wl.name)
    flips = routing_flips(idx.cpu().numpy(), ridx, lg_ref, per)
    if len(flips):
        print(f"{wl.name}: {len(flips)} tokens take another valid expert set")
    return flips


SMALL = [
    WORKLOADS["tiny"],
    Workload("small-shared", T=300, H=256, E=16, k=4, I=256, I_s=384, rmsnorm=True,
             gamma_std=0.1, x_std=1.0),
    Workload("small-skew", T=257, H=384, E=64, k=8, I=128, x_std=1.0, skew_s=1.2,
             skew_beta=1.5),
    Workload("small-wideE", T=129, H=256, E=96, k=6, I=128, I_s=128, rmsnorm=True),
    Workload("small-one", T=1, H=128, E=4, k=1, I=128),
    # > 512 tokens: tiled router with the routing histogram fused in
    Workload("mid-tiled", T=700, H=256, E=32, k=4, I=128, I_s=128, rmsnorm=True,
             gamma_std=0.1),
    # E > 64: separate top-k and histogram launches
    Workload("mid-wideE", T=640, H=128, E=80, k=5, I=128),
    # the fused top-k of the tensor-core gate with more than 8 slots, softmax
    # over all experts (no renorm), and gate offsets
    Workload("mid-k12", T=600, H=256, E=48, k=12, I=128, renorm=False, skew_s=1.2,
             skew_beta=0.5),
    # the limits: 1024 experts (most of them empty), 32 slots per token
    Workload("max-Ek", T=200, H=128, E=1024, k=32, I=128, I_s=128, rmsnorm=True),
    # either side of the gate switch (512 tokens: sequential; 513: tensor cores, with
    # 65 experts the combine writes logits for the separate top-k)
    Workload("edge-512", T=512, H=128, E=65, k=3, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("edge-513", T=513, H=128, E=65, k=3, I=128, rmsnorm=True, gamma_std=0.1),
    # shapes the wide pair kernel takes (I, I_s % 256 == 0, H % 512 == 0)
    Workload("mid-wide", T=900, H=512, E=8, k=2, I=256, I_s=256, rmsnorm=True,
             gamma_std=0.1, x_std=1.0),
    # 1100 rows per expert and in the shared segment: the wide pair kernel by
    # default, each group ending in a 76-row block
    Workload("mid-wide-tails", T=1100, H=512, E=2, k=2, I=256, I_s=256, rmsnorm=True,
             gamma_std=0.1, x_std=1.0),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("out_f32", [True, False], ids=["f32", "bf16"])
def test_layer_small_all_tokens(wl, out_f32):
    d = make_inputs(wl, 2)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    ref, ref_yf, ridx, rw, ys = oracle.layer_tokens_both(d, wl)
    allow = routed_flip_allowance(ys, rw)
    keep = np.setdiff1d(np.arange(wl.T), _tc_flips(wl, g, d, ridx=ridx))
    for seq in ((False, True) if wl.T > 512 else (False,)):
        sel = np.arange(wl.T) if seq else keep
        what = f"{wl.name}{' sequential gate' if seq else ''}"
        out = _run_layer(wl, g, out_f32, seq=seq)
        check_out(t2f64(out)[sel], ref[sel], bf16_out=not out_f32, what=what,
                  flip_allowance=allow[sel])
        # fp32 routed outputs: the strict bar, no allowance
        out = _run_layer(wl, g, out_f32, seq=seq, y_f32=True)
        check_out(t2f64(out)[sel], ref_yf[sel], bf16_out=not out_f32, what=what + " y_f32")
        # rows gathered inside the w13 matmul (where it runs as the wide pair
        # kernel; elsewhere the flag is ignored): the same bytes
        gat = _run_layer(wl, g, out_f32, seq=seq, y_f32=True, gather_a=True)
        assert torch.equal(gat, out), what + " gather_a"


def test_layer_deterministic_and_workspace_reuse():
    wl = SMALL[1]
    d = make_inputs(wl, 4)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    desc = _desc(wl)
    ws = torch.full((moe.layer_workspace_size(desc),), 0x7F, dtype=torch.uint8, device=DEV)
    a = moe.layer_forward(desc, g["x"], _weights(g), workspace=ws)
    ws.fill_(0xFF)
    b = moe.layer_forward(desc, g["x"], _weights(g), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_layer_empty_tokens():
    wl = WORKLOADS["tiny"]
    d = make_inputs(wl, 0)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    x0 = g["x"][:0]
    out = moe.layer_forward(_desc(wl, T=0), x0, _weights(g))
    assert out.shape == (0, wl.H)


# ------------------------------------------------------------ full sizes
FULL = ["balanced-4k", "imagegen-16k", "skewed-32k", "smallbatch-8", "smallbatch-64",
        "smallbatch-256"]


def _sample_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(T, n), replace=False).tolist())
    pick.update({0, T - 1})
    return np.array(sorted(pick), dtype=np.int32)


# seed 0 on every full-size workload; seeds 1 and 2 on the three large ones
FULL_SEEDS = [(n, 0) for n in FULL] + [(n, sd) for sd in (1, 2)
                                        for n in ("balanced-4k", "imagegen-16k", "skewed-32k")]


@pytest.mark.parametrize("name,seed", FULL_SEEDS, ids=lambda v: str(v))
def test_layer_full_size(name, seed):
    wl = WORKLOADS[name]
    g = make_inputs(wl, seed, device=DEV)
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in g.items()}

    # routing over every token, bit-exact given the same inputs
    xn, logits = moe.rmsnorm_gate(g["x"], g["wg"], g["gamma"], g["gate_bias"], wl.eps,
                                  rmsnorm=wl.rmsnorm)
    idx, w = moe.gate_topk(logits, wl.k, wl.renorm)
    r = moe.init_routing(idx, None, wl.E, with_rows=False)
    torch.cuda.synchronize()
    xs_ref = oracle.rmsnorm(cpu["x"], cpu["gamma"], wl.eps) if wl.rmsnorm else u16(cpu["x"])
    if wl.rmsnorm:
        assert np.array_equal(u16(xn), xs_ref)
    lg_ref = oracle.gate_logits(xs_ref, cpu["wg"], cpu["gate_bias"])
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), lg_ref.view(np.uint32))
    ridx, rw = oracle.topk_softmax(lg_ref, wl.k, wl.renorm)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=2e-7)
    rr = oracle.init_routing(ridx, wl.E)
    for key in ("row_idx", "src_token", "counts", "offsets"):
        assert np.array_equal(r[key].cpu().numpy(), rr[key]), key
    counts = rr["counts"]
    if name.startswith("skewed"):
        print(f"{name}: {int((counts == 0).sum())} idle experts, top share "
              f"{counts.max() / counts.sum():.4f}")

    # the tensor-core gate's routing (the layer's for T > 512)
    flips = _tc_flips(wl, g, cpu, xs_ref, lg_ref, ridx)

    # layer output on every token of the smaller loads and 2048 tokens of the
    # large ones (fp32 output strict, bf16 output + half an ulp), with the
    # layer's own gate and with the sequential one, in both y readings
    if wl.T <= 4096:
        tok = np.arange(wl.T, dtype=np.int32)
    else:
        tok = _sample_tokens(wl.T, 2040, 7 + seed)
        # include tokens routed to the busiest expert
        busiest = int(np.argmax(counts))
        hot = np.nonzero((ridx == busiest).any(axis=1))[0][:8]
        tok = np.unique(np.concatenate([tok, hot]).astype(np.int32))
    ref, ref_yf, _, rw_s, ys = oracle.layer_tokens_both(cpu, wl, tok)
    allow = routed_flip_allowance(ys, rw_s)
    keep = ~np.isin(tok, flips)
    tok_dev = torch.from_numpy(tok).long().to(DEV)
    for seq in ((False, True) if wl.T > 512 else (False,)):
        sel = np.ones(len(tok), dtype=bool) if seq else keep
        for out_f32 in (True, False):
            what = f"{name} f32={out_f32} sequential={seq}"
            got = t2f64(_run_layer(wl, g, out_f32, seq=seq)[tok_dev])
            check_out(got[sel], ref[sel], bf16_out=not out_f32, what=what,
                      flip_allowance=allow[sel])
            full = _run_layer(wl, g, out_f32, seq=seq, y_f32=True)
            got = t2f64(full[tok_dev])
            mx, rel = check_out(got[sel], ref_yf[sel], bf16_out=not out_f32,
                                what=what + " y_f32")
            print(f"{what} y_f32: {int(sel.sum())} tokens, max-abs {mx:.3e}, rel-L2 {rel:.3e}")
            # rows gathered inside the w13 matmul: every token, the same bytes
            gat = _run_layer(wl, g, out_f32, seq=seq, y_f32=True, gather_a=True)
            assert torch.equal(gat, full), what + " gather_a"


def test_shared_expert_on_second_stream_matches():
    """The shared expert on its own stream ("MoE多流并行优化") gives the same
    bits as the one-stream layer (same kernels, only the order of launches
    across streams differs)."""
    wl = SMALL[1]
    d = make_inputs(wl, 6)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    desc = _desc(wl)
    a = moe.layer_forward(desc, g["x"], _weights(g))
    s2 = torch.cuda.Stream()
    evs = [torch.cuda.Event(), torch.cuda.Event()]
    for e in evs:
        e.record()
    st = moe.new_status(DEV)
    b = moe.layer_forward(desc, g["x"], _weights(g), status=st, shared_stream=s2, events=evs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a, b)
    ref, _, _ = oracle.layer_tokens(d, wl)
    check_out(t2f64(b), ref, bf16_out=False, what="two streams")


@pytest.mark.parametrize("out_f32", [False, True], ids=["bf16", "f32"])
def test_host_pipeline_matches_device_layer(out_f32):
    """moe_layer_forward_host over several host batches (copies overlapped
    with the compute) gives, batch by batch, the device layer's bytes."""
    wl = Workload("host-pipe", T=600, H=256, E=16, k=4, I=256, I_s=128, rmsnorm=True,
                  gamma_std=0.1)
    g = make_inputs(wl, 3, device=DEV)
    xs = [make_inputs(wl, 10 + i, only=["x"])["x"].pin_memory() for i in range(5)]
    desc = _desc(wl, out_f32=out_f32)
    st = moe.new_status(DEV)
    outs = moe.layer_forward_host(desc, xs, _weights(g), status=st)
    assert int(st.item()) == 0
    for x, o in zip(xs, outs):
        ref = moe.layer_forward(desc, x.to(DEV), _weights(g))
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16 if not out_f32 else torch.int32),
                           ref.cpu().view(torch.int16 if not out_f32 else torch.int32))
    one = moe.layer_forward_host(desc, xs[0], _weights(g))       # a single tensor in, out
    assert torch.equal(one, outs[0])


GRAPH_WL = [
    WORKLOADS["tiny"],
    Workload("mid-tiled", T=700, H=256, E=32, k=4, I=128, I_s=128, rmsnorm=True, gamma_std=0.1),
    # 1024 rows per group: the CTA-pair GEMM with its per-launch tile counter
    Workload("graph-pair", T=2048, H=256, E=4, k=2, I=256, I_s=256, rmsnorm=True),
]


@pytest.mark.parametrize("wl", GRAPH_WL, ids=lambda w: w.name)
def test_layer_in_cuda_graph(wl):
    """The layer captured in a CUDA graph and replayed (new inputs copied into
    the captured buffers) gives the eager call's bytes: every launch, memset
    and tile counter of the step lives on the captured stream."""
    g = make_inputs(wl, 4, device=DEV)
    desc = _desc(wl, out_f32=False)
    w = _weights(g)
    x = g["x"].clone()
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(moe.layer_workspace_size(desc), dtype=torch.uint8, device=DEV)
    st = moe.new_status(DEV)
    moe.layer_forward(desc, x, w, out=out, workspace=ws, status=st)     # warm-up outside
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        moe.layer_forward(desc, x, w, out=out, workspace=ws, status=st)
    for seed in (5, 6):
        x.copy_(make_inputs(wl, seed, device=DEV, only=["x"])["x"])
        graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = moe.layer_forward(desc, x, w)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
