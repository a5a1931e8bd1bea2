"""GPU parity of every step of the layer against the CPU oracle, through the
C ABI (the Python binding only marshals arguments).

Small shapes span several tiles and a ragged tail; the edge cases are empty
inputs, zero-row and one-row experts, ties in the gate logits and invalid
expert ids (reported through the device status word, never a fault).
"""
import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe
import oracle
from moe_inputs import WORKLOADS, Workload, make_inputs
from tests._helpers import bf16_to_f64, bf16_ulp, check_bf16_close, t2f64, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _cuda(d):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


# ------------------------------------------------------------ rmsnorm + gate
@pytest.mark.parametrize("wl", [
    Workload("g-tiny", T=64, H=128, E=8, k=2, I=256),
    Workload("g-rms", T=77, H=320, E=13, k=3, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-bias", T=100, H=256, E=64, k=8, I=128, rmsnorm=True, skew_s=1.2, skew_beta=1.0),
    Workload("g-wideE", T=40, H=192, E=160, k=6, I=128, rmsnorm=True),
    # the small-batch router's rings: one token per CTA in 6 slots of 128
    # columns with refills (T <= SMs) or 12 slots of 64 columns (H not a
    # multiple of 128); two tokens per CTA in 5 slots of 128 columns (one
    # wave up to 2 tokens per SM, two beyond) or 10 of 64, odd T; 3 slots
    # (E=128 at the largest H); one chunk
    Workload("g-small-deep", T=100, H=1024, E=64, k=8, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-h64", T=50, H=1088, E=40, k=4, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-2cta", T=300, H=512, E=32, k=4, I=128, rmsnorm=True),
    Workload("g-small-2tok", T=201, H=1536, E=64, k=8, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-2tok-2cta", T=333, H=640, E=24, k=4, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-2tok-plain", T=157, H=192, E=16, k=2, I=128),
    Workload("g-small-2tok-h64", T=171, H=1344, E=48, k=4, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-maxH", T=24, H=8192, E=128, k=8, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-small-1chunk", T=5, H=64, E=6, k=2, I=128),
    # more than 512 tokens: the tiled router (32 tokens x 64 experts per CTA)
    Workload("g-tiled", T=700, H=256, E=64, k=8, I=128, rmsnorm=True, gamma_std=0.1),
    Workload("g-tiled-plain", T=1025, H=128, E=8, k=2, I=128),
    Workload("g-tiled-E100", T=600, H=320, E=100, k=4, I=128, rmsnorm=True, skew_s=1.2,
             skew_beta=0.7),
], ids=lambda w: w.name)
def test_rmsnorm_gate_bitexact(wl):
    d = make_inputs(wl, 1)
    g = _cuda(d)
    xn, logits = moe.rmsnorm_gate(g["x"], g["wg"], g["gamma"], g["gate_bias"], wl.eps,
                                  rmsnorm=wl.rmsnorm)
    torch.cuda.synchronize()
    xs_ref = oracle.rmsnorm(d["x"], d["gamma"], wl.eps) if wl.rmsnorm else u16(d["x"])
    if wl.rmsnorm:
        assert np.array_equal(u16(xn), xs_ref)
    lg_ref = oracle.gate_logits(xs_ref, d["wg"], d["gate_bias"])
    assert np.array_equal(logits.cpu().numpy().view(np.uint32), lg_ref.view(np.uint32))


# the RMSNorm-only pass (ahead of the tensor-core gate): one warp per row,
# rows in registers (up to 4, 8, 16 or 32 vectors per lane), many rows per
# warp, ragged vector counts (H = 384); gamma absent (all ones)
@pytest.mark.parametrize("T,H,gamma_std,with_gamma", [
    (1, 128, 0.1, True), (33, 4096, 0.1, True), (5000, 4096, 0.1, True),
    (1000, 1024, 0.0, False), (700, 8192, 0.2, True), (64, 384, 0.1, True),
    (20000, 256, 0.1, True)])
def test_rmsnorm_only_bitexact(T, H, gamma_std, with_gamma):
    wl = Workload("rn", T=T, H=H, E=4, k=1, I=128, rmsnorm=True, gamma_std=gamma_std)
    d = make_inputs(wl, 3, only=("x", "gamma"))
    gamma = d["gamma"] if with_gamma else None
    xn, lg = moe.rmsnorm_gate(d["x"].to(DEV), None, gamma.to(DEV) if gamma is not None else None,
                              None, wl.eps)
    torch.cuda.synchronize()
    assert lg is None
    ones = torch.ones(H, dtype=torch.bfloat16)
    assert np.array_equal(u16(xn), oracle.rmsnorm(d["x"], gamma if with_gamma else ones, wl.eps))


def _bf16_rows(rows):
    """float64 rows -> bf16 torch tensor (values rounded once to bf16)."""
    return torch.from_numpy(np.ascontiguousarray(rows, dtype=np.float32)).to(torch.bfloat16)


def _sumsq_cases(H):
    """Rows whose sums of squares exercise the exact rounding: random rows of
    many scales and of a 120-binade spread, exact ties and sums just above
    them, sums that the fast path cannot decide (its residual bound straddles
    a tie), largest values outside its exponent range, values below 2^-60 next
    to normal ones, bf16 subnormals, fp32 subnormal and overflowing sums,
    zeros and single nonzero values."""
    rng = np.random.default_rng(21 + H)
    rows = []
    for scale in (1.0, 2.0 ** -10, 2.0 ** 12, 2.0 ** -19, 2.0 ** 38):
        rows += [rng.standard_normal(H) * scale for _ in range(3)]
    rows.append(rng.standard_normal(H) * 2.0 ** rng.integers(-60, 60, H))
    z = np.zeros(H)

    def row(vals):
        r = z.copy()
        r[:len(vals)] = vals
        return r
    big = [2.0 ** 11] * 4
    rows.append(row(big + [1.0]))                          # 2^24 + 1: tie, to even
    rows.append(row(big + [1.0, 2.0 ** -30]))              # just above the tie
    rows.append(row(big + [1.0] * 3))                      # 2^24 + 3: tie, to even
    near = [1.0] + [2.0 ** -13] * 3 + [2.0 ** -14] * 3 + [2.0 ** -15] * 3
    rows.append(row(near + [2.0 ** -16] * 4))              # an exact tie the bound straddles
    rows.append(row(near + [2.0 ** -16] * 4 + [2.0 ** -40]))   # 2^-80 above it
    rows.append(row(near + [2.0 ** -16] * 5))              # a quarter unit above it
    rows.append(rng.standard_normal(H) * 2.0 ** 45)         # largest exponent > 40
    rows.append(rng.standard_normal(H) * 2.0 ** -40)        # largest exponent < -20
    rows.append(row([1.5, 2.0 ** -70, -(2.0 ** -80)]))     # nonzero values below 2^-60
    rows.append(row([2.0 ** -130, 3 * 2.0 ** -133, 2.0 ** -127]))   # bf16 subnormals
    rows.append(row([2.0 ** -70] * 4))                     # fp32 subnormal sum
    rows.append(row([2.0 ** -75] * 3))                     # 1.5 * 2^-149: tie to 2^-148
    rows.append(row([2.0 ** 64]))                          # overflows to infinity
    rows.append(z.copy())
    rows.append(row([-3.0]))
    return _bf16_rows(np.array(rows))


@pytest.mark.parametrize("H", [4096, 16, 136, 1024, 8192])
def test_rmsnorm_sumsq_is_the_exact_sum_rounded_once(H):
    x = _sumsq_cases(H)
    ss = moe.rmsnorm_sumsq(x.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.sumsq(x)
    got = ss.cpu().numpy()
    bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
    assert bad.size == 0, f"rows {bad.tolist()}: {got[bad]} vs {ref[bad]}"


def test_rmsnorm_only_on_exact_sum_edge_rows():
    """xn of the RMSNorm pass on the same edge rows (finite ones; ties,
    straddled bounds, subnormals) equals the oracle's bit for bit."""
    x = _sumsq_cases(4096)
    keep = np.isfinite(oracle.sumsq(x)) & (oracle.sumsq(x) > 0)
    x = x[torch.from_numpy(keep)]
    gamma = _bf16_rows(1 + 0.1 * np.random.default_rng(5).standard_normal(4096))
    for eps in (1e-6, 0.0):
        xn, _ = moe.rmsnorm_gate(x.to(DEV), None, gamma.to(DEV), None, eps)
        torch.cuda.synchronize()
        got, ref = u16(xn), oracle.rmsnorm(x, gamma, eps)
        # with eps = 0 a row whose mean of squares underflows to zero gives
        # 0 * inf = NaN: NaN in the same places (the payloads may differ)
        nan_g = (got & 0x7F80) == 0x7F80
        nan_g &= (got & 0x7F) != 0
        nan_r = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
        assert np.array_equal(nan_g, nan_r), eps
        assert np.array_equal(got[~nan_g], ref[~nan_r]), eps


def test_rmsnorm_gate_empty():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device=DEV)
    wg = torch.zeros((8, 128), dtype=torch.float32, device=DEV)
    xn, lg = moe.rmsnorm_gate(x, wg, None, None, 1e-6, rmsnorm=True)
    assert xn.shape == (0, 128) and lg.shape == (0, 8)


# ------------------------------------------------------------------- top-k
@pytest.mark.parametrize("T,E,k,renorm", [(1000, 64, 8, True), (333, 8, 2, True),
                                          (200, 64, 8, False), (97, 300, 7, True),
                                          (50, 1024, 32, True), (64, 5, 5, True)])
def test_topk(T, E, k, renorm):
    rng = np.random.default_rng(T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0] = 0.25                               # all tied -> 0..k-1
    lg[1, :] = -3.0
    lg[1, E // 2] = 1.0
    lg[1, E - 1] = 1.0                         # tie at the top
    lg[2, : min(E, 4)] = [0.0, -0.0, 0.0, -0.0][: min(E, 4)]
    lg[3] = np.round(lg[3] * 4) / 4            # many ties
    idx, w = moe.gate_topk(torch.from_numpy(lg).to(DEV), k, renorm)
    ridx, rw = oracle.topk_softmax(lg, k, renorm)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=2e-6, atol=2e-7)


# ------------------------------------------------------------------ routing
# up to 512 tokens (and 8K histogram entries) the scan counts the histogram
# itself: 77, 1, 512 tokens and 256 x 1024 experts (the largest such array);
# 384 x 1024 is past it
@pytest.mark.parametrize("T,k,E,H", [(1000, 8, 64, 256), (77, 2, 8, 128), (1, 1, 1, 64),
                                     (4097, 6, 300, 64), (513, 4, 1024, 64), (512, 8, 64, 128),
                                     (256, 3, 1024, 64), (384, 3, 1024, 64)])
def test_init_routing_bitexact(T, k, E, H):
    rng = np.random.default_rng(T * 7 + E)
    w = rng.pareto(1.2, E) + 0.01              # skewed expert popularity
    idx = np.stack([rng.choice(E, k, replace=False, p=w / w.sum()) for _ in range(T)]).astype(
        np.int32)
    x = torch.randn((T, H), dtype=torch.float32).to(torch.bfloat16)
    r = moe.init_routing(torch.from_numpy(idx).to(DEV), x.to(DEV), E)
    ref = oracle.init_routing(idx, E)
    for key in ("row_idx", "src_token", "sorted_ids", "counts", "offsets"):
        assert np.array_equal(r[key].cpu().numpy(), ref[key]), key
    assert np.array_equal(u16(r["expanded_x"]), oracle.permute(x, ref["src_token"]))
    c, o = moe.expert_tokens(r["sorted_ids"], E)
    assert np.array_equal(c.cpu().numpy(), ref["counts"])
    assert np.array_equal(o.cpu().numpy(), ref["offsets"])


def test_init_routing_bad_expert_reports():
    idx = torch.tensor([[0, 1], [2, 9], [-1, 3]], dtype=torch.int32, device=DEV)
    st = moe.new_status(DEV)
    moe.init_routing(idx, None, 4, with_rows=False, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_EXPERT_ID


def test_expert_tokens_unsorted_reports():
    ids = torch.tensor([0, 2, 1, 3], dtype=torch.int32, device=DEV)
    st = moe.new_status(DEV)
    moe.expert_tokens(ids, 4, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_UNSORTED
    c, o = moe.expert_tokens(torch.empty(0, dtype=torch.int32, device=DEV), 5)
    assert c.cpu().tolist() == [0] * 5 and o.cpu().tolist() == [0] * 6


# ------------------------------------------------------------- grouped MLP
def _grouped_case(counts, H, I, seed):
    g = torch.Generator().manual_seed(seed)
    G = len(counts)
    n = int(sum(counts))
    x = torch.randn((n, H), generator=g).to(torch.bfloat16)
    w13 = (0.05 * torch.randn((G, 2 * I, H), generator=g)).to(torch.bfloat16)
    w2 = (0.05 * torch.randn((G, H, I), generator=g)).to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return x, w13, w2, off


@pytest.mark.parametrize("counts,H,I", [
    ([300], 256, 256),                          # one group: a dense GEMM
    ([0, 1, 129, 0, 255, 37, 0, 512], 384, 256),
    ([5, 0, 0, 128, 127], 128, 384),            # H=128: 128-wide down tiles
    ([700, 3, 64], 512, 128),
    # shapes the wide pair kernel takes (I % 256 == 0, H % 512 == 0): empty,
    # one-row, half-tile (<= 128 rows) and multi-block groups
    ([0, 1, 129, 0, 255, 37, 0, 512, 300], 512, 256),
    ([1000, 600, 64, 257], 1024, 512),
    # >= 1024 rows per group on average (the wide pair kernel by default):
    # last blocks of 1, 128, 129 and 76 rows, and none
    ([1025, 1280, 1408, 1409, 1100], 512, 256),
], ids=["dense", "ragged", "h128", "mixed", "wide-ragged", "wide-big", "wide-tails"])
def test_grouped_mlp(counts, H, I):
    x, w13, w2, off = _grouped_case(counts, H, I, len(counts) * 31 + H)
    st = moe.new_status(DEV)
    act, y = moe.grouped_mlp(x.to(DEV), torch.from_numpy(off).to(DEV), w13.to(DEV), w2.to(DEV),
                             status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ract, ry = oracle.grouped_mlp(x, off, w13, w2)
    check_bf16_close(u16(act), ract, 2e-3, "act", atol_rms=2.0**-16)
    # the accepted act flips propagate into y: allow |d act| . |w2|^T on top
    dact = np.abs(t2f64(act) - bf16_to_f64(ract))
    prop = np.zeros((act.shape[0], H))
    w2a = np.abs(t2f64(w2))
    for gi in range(len(counts)):
        r0, r1 = int(off[gi]), int(off[gi + 1])
        if r1 > r0:
            prop[r0:r1] = dact[r0:r1] @ w2a[gi].T
    check_bf16_close(u16(y), ry, 2e-2, "y", atol_rms=2.0**-14, extra=1.01 * prop)
    n = int(off[-1])
    assert torch.count_nonzero(act[n:]) == 0 and torch.count_nonzero(y[n:]) == 0


def test_grouped_mlp_dense_matches_torch():
    """One group is a dense GEMM: y = bf16(act @ w2^T) with act from SwiGLU;
    checked against torch.matmul in fp32 on the same bf16 operands."""
    x, w13, w2, off = _grouped_case([1000], 512, 256, 5)
    act, y = moe.grouped_mlp(x.to(DEV), torch.from_numpy(off).to(DEV), w13.to(DEV), w2.to(DEV))
    xf = x.to(DEV).float()
    h = xf @ w13[0].to(DEV).float().T
    g, u = h[:, :256], h[:, 256:]
    ref_act = (torch.nn.functional.silu(g) * u)
    torch.testing.assert_close(act.float(), ref_act, atol=2e-2, rtol=1e-2)
    ref_y = act.float() @ w2[0].to(DEV).float().T
    torch.testing.assert_close(y.float(), ref_y, atol=1e-2, rtol=1e-2)


def test_grouped_mlp_bad_offsets_reports():
    x, w13, w2, off = _grouped_case([10, 20], 128, 128, 9)
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device=DEV)   # not monotone
    st = moe.new_status(DEV)
    moe.grouped_mlp(x.to(DEV), bad, w13.to(DEV), w2.to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & moe.DEV_BAD_OFFSETS


# ---------------------------------------------------------------- finalize
@pytest.mark.parametrize("shared", [None, "bf16", "f32"])
@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("y_f32", [False, True], ids=["ybf16", "yf32"])
def test_finalize(shared, out_f32, y_f32):
    T, H, E, k = 300, 256, 16, 4
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = oracle.topk_softmax(lg, k)
    r = oracle.init_routing(idx, E)
    y = torch.randn((T * k, H))
    if not y_f32:
        y = y.to(torch.bfloat16)
    sh = None
    sh_ref = None
    if shared == "bf16":
        sh = torch.randn((T, H)).to(torch.bfloat16)
        sh_ref = t2f64(sh)
    elif shared == "f32":
        sh = torch.randn((T, H), dtype=torch.float32)
        sh_ref = sh.double().numpy()
    out = moe.finalize_routing(y.to(DEV), torch.from_numpy(r["row_idx"]).to(DEV),
                               torch.from_numpy(w).to(DEV),
                               None if sh is None else sh.to(DEV), out_f32=out_f32)
    ref = oracle.finalize(y.double().numpy() if y_f32 else y, r["row_idx"], w, sh_ref)
    got = t2f64(out)
    if out_f32:
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)
    else:
        assert np.all(np.abs(got - ref) <= 0.5 * bf16_ulp(ref) + 1e-6 * np.abs(ref) + 1e-6)


def test_finalize_identity_experts():
    """y_exp = the permuted input rows: the renormalised weights sum to one,
    so finalize returns the input."""
    T, H, E, k = 500, 128, 32, 6
    x = torch.randn((T, H)).to(torch.bfloat16).to(DEV)
    lg = torch.randn((T, E), device=DEV)
    idx, w = moe.gate_topk(lg, k)
    r = moe.init_routing(idx, x, E)
    out = moe.finalize_routing(r["expanded_x"], r["row_idx"], w, out_f32=True)
    torch.testing.assert_close(out, x.float(), rtol=1e-6, atol=1e-6)
    out2 = moe.finalize_routing(r["expanded_x"], r["row_idx"], w, out_f32=True)
    assert torch.equal(out, out2)                       # deterministic
