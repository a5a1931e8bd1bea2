"""Shared helpers of the test suite: conversions and the output tolerances.

Tolerances (layer outputs): the fp32 output mode must be within max-abs 2e-2
and relative-L2 5e-3 of the oracle's double result; the bf16 output mode may
in addition be off by half a bf16 ulp of the oracle value (its own final
rounding).  Where the test has the oracle's routed rows, a rare element may
also be off by one bf16 ulp of each routed term (routed_flip_allowance).  act / y_exp (bf16 intermediates) may differ from the oracle by
one bf16 ulp where the fp32 tensor-core sum and the oracle's exact sum round
to neighbouring bf16 values; such flips must stay rare.  Near zero (after
cancellation in the sum) the fp32 accumulation error is absolute, not
relative, so the intermediate check adds a floor of ``atol_rms`` times the
tensor's RMS: 2^-16 for act (an fp32 sum of K <= 4096 terms is off by at
most ~K * 2^-24 of the sum of |terms|), 2^-10 for y (which also carries the
one-ulp act flips: each moves y by ~ulp(act) * |w2|); where the act
difference is known, the y check instead adds |act_gpu - act_oracle| . |w2|^T
per element, the exact first-order propagation of the accepted act flips).
"""
import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 5e-3


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def t2f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return bf16_to_f64(u16(t))
    return t.detach().cpu().to(torch.float64).numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(v), 2.0**-126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def routed_flip_allowance(y_bits, w):
    """Per output element, sum_j |w_j| * ulp_bf16(y_j): what one-ulp flips of
    the routed bf16 expert outputs y_j (the oracle's, [n, k, H] bits) can move
    the weighted sum by.  The GPU rounds its fp32 sum of each y to bf16 as the
    oracle rounds its exact sum; where the two straddle a rounding boundary
    they land one bf16 ulp apart (0.031 for |y| in [4, 8))."""
    y = bf16_to_f64(y_bits)
    return np.einsum("nk,nkh->nh", np.abs(np.asarray(w, dtype=np.float64)), bf16_ulp(y))


# elements allowed past MAX_ABS by routed one-ulp flips: must stay this rare
FLIP_FRAC = 1e-4


def check_out(gpu: np.ndarray, ref: np.ndarray, bf16_out: bool, what="", flip_allowance=None):
    """Assert the layer-output tolerance; returns (max_abs, rel_l2).  With
    ``flip_allowance`` (routed_flip_allowance of the oracle's rows) an element
    may exceed max-abs by at most that much, on at most FLIP_FRAC of the
    elements: a one-ulp flip of a bf16 routed output with a weight near 1 at
    |y| >= 4 moves the output by more than 2e-2 on its own."""
    d = np.abs(gpu - ref)
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))
    mx = float(d.max()) if d.size else 0.0
    bound = MAX_ABS + (0.5 * bf16_ulp(ref) if bf16_out else 0.0)
    over = d > bound
    if flip_allowance is not None and over.any():
        assert not (d > bound + flip_allowance).any(), (
            f"{what}: elements beyond 2e-2 plus one bf16 ulp of every routed term, max {mx}")
        assert over.mean() <= FLIP_FRAC, f"{what}: {int(over.sum())} elements past 2e-2"
    else:
        assert not over.any(), (f"{what}: {int(over.sum())} elements beyond 2e-2"
                                f"{' + ulp/2' if bf16_out else ''}, max {mx}")
    assert rel <= REL_L2, f"{what}: rel-L2 {rel} > {REL_L2}"
    return mx, rel


def check_bf16_close(gpu_bits: np.ndarray, ref_bits: np.ndarray, max_flip_frac: float,
                     what="", atol_rms=2.0**-16, extra=None):
    """bf16 tensors equal up to one-ulp flips, which must be rare.  ``extra``
    (same shape) adds a per-element allowance, e.g. the propagated effect of
    differences already accepted in an input."""
    g = bf16_to_f64(gpu_bits)
    r = bf16_to_f64(ref_bits)
    d = np.abs(g - r)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    tol = np.maximum(bf16_ulp(r), bf16_ulp(g)) * 1.0001 + atol_rms * rms
    if extra is not None:
        tol = tol + extra
    bad = d > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} differences beyond one bf16 ulp + "
                           f"{atol_rms:g} rms, max {d.max()}")
    flips = float(np.mean(d > 0)) if d.size else 0.0
    assert flips <= max_flip_frac, f"{what}: {flips:.2e} of values flipped one ulp"
    return flips


# ------------------------------------------------ the tensor-core gate
# The tensor-core gate (moe_gate_tensor, the layer's gate for T > 512) adds
# the same exact products as the oracle's sequential fp32 dot product in
# another order, so the two logits differ by rounding only.  Bound on that
# difference per logit, with S = sum_h |xs_h * wg_eh| and u = 2^-24:
#   oracle, one rounding per fused multiply-add:      H * u * S
#   tensor core, per K=16 step a block sum and one accumulation, each
#   rounded at most one fp32 ulp (2u, truncation allowed): (H/16 + 16) * 2u * S
#   (the second and third weight parts carry 2^-8 and 2^-16 of the first's
#   magnitude: a factor 1.01 covers them)
#   the combine (p1 + p2) + p3 + bias, three roundings:  4u * |logit|
# The root-mean-square difference over many logits, with independent
# rounding errors, is far smaller: at most 2 sqrt(H) u times the RMS of S.
# A gate that drops the second weight part misses by ~2^-9 / sqrt(3) of the
# logit's spread and fails that; the exact split itself (w = w1 + w2 + w3)
# is checked on its own.
def gate_tc_bound(xs_bits, wg, lg_ref):
    """-> (per-logit bound [T, E], rms bound) on |tensor-core - oracle| logits."""
    xs = bf16_to_f64(xs_bits)
    w = np.asarray(wg, dtype=np.float64)
    H = xs.shape[1]
    S = np.abs(xs) @ np.abs(w).T
    u = 2.0 ** -24
    per = ((H / 16 + 16) * 2 * u * 1.01 + H * u) * S + 4 * u * np.abs(lg_ref.astype(np.float64))
    rms = 2 * np.sqrt(H) * u * float(np.sqrt(np.mean(S * S))) if S.size else 0.0
    return per, rms


def check_gate_tc_logits(lg_gpu, lg_ref, per, rms_bound, what=""):
    d = np.abs(lg_gpu.astype(np.float64) - lg_ref.astype(np.float64))
    bad = d > per
    assert not bad.any(), (f"{what}: {int(bad.sum())} logits beyond the fp32 rounding bound, "
                           f"worst excess {float((d - per).max())}")
    rms = float(np.sqrt(np.mean(d * d))) if d.size else 0.0
    assert rms <= rms_bound, f"{what}: RMS logit difference {rms} > {rms_bound}"
    return float(d.max()) if d.size else 0.0, rms


def routing_flips(idx_gpu, idx_ref, lg_ref, per):
    """Tokens whose set of chosen experts differs from the oracle's.  Each
    such choice must be a valid top-k of the oracle's logits once every logit
    may move by its rounding bound (an ambiguous near-tie), and the slot
    order of every token must be consistent with the oracle's logits up to
    the same bound.  Returns the flipped tokens (sorted)."""
    idx_gpu = np.asarray(idx_gpu)
    idx_ref = np.asarray(idx_ref)
    T, k = idx_ref.shape
    E = lg_ref.shape[1]
    lg = lg_ref.astype(np.float64)
    assert idx_gpu.shape == (T, k)
    assert ((idx_gpu >= 0) & (idx_gpu < E)).all(), "expert id out of range"
    srt = np.sort(idx_gpu, axis=1)
    assert (np.diff(srt, axis=1) > 0).all(), "an expert chosen twice"
    flipped = np.nonzero((srt != np.sort(idx_ref, axis=1)).any(axis=1))[0]
    reordered = np.nonzero((idx_gpu != idx_ref).any(axis=1))[0]
    for t in reordered:
        g = idx_gpu[t]
        hi = lg[t] + per[t]
        lo = lg[t] - per[t]
        # slot order: descending up to the bound
        assert (hi[g[:-1]] >= lo[g[1:]]).all(), f"token {t}: slot order {g} not descending"
        # every chosen expert at least as large as every other, up to the bound
        rest = np.ones(E, dtype=bool)
        rest[g] = False
        if rest.any():
            assert hi[g].min() >= lo[rest].max(), f"token {t}: {g} is not a top-{k}"
    return flipped
