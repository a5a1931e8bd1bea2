"""Pins of the CPU oracle to things other than itself.

Each pin checks the oracle against a value worked by hand from the page
("NPU HunyuanImage-3.0模型推理优化实践", sections 'MoE TP优化 / 计算分解',
'MoE EP优化', 'GMM使能&&Routing优化', 'RmsNorm算子优化',
'消除gate计算冗余cast算子'), a closed form, an invariant, a library routine
on a special case, or brute force on tiny inputs.  ``test_mutants_are_caught``
plants plausible mistakes in temporary copies of the oracle source and checks
that every one of them fails at least one pin.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
from moe_inputs import WORKLOADS, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_f64(bits):
    return oracle.bits_to_float(bits).astype(np.float64)


# --------------------------------------------------------------------- pins
def pin_bf16_rounding():
    # hand values: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3*2^-8 ties between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6;
    # 1 + 2^-8 + 2^-40 is above the tie -> 1 + 2^-7 (a float detour would
    # round twice and give 1.0).
    got = oracle.bf16_bits([1.0, 1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-40,
                            -2.5, 0.0, 3.0e38, 3.4e38])
    assert list(got[:6]) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000], got
    # 3.0e38 = 1.7632 * 2^127 -> mantissa 97.69/128 -> 98 -> 0x7F62;
    # 3.4e38 lies above the midpoint between the largest bf16 and 2^128 -> inf
    assert got[6] == 0x7F62 and got[7] == 0x7F80, got
    # library routine: torch's fp32 -> bf16 conversion rounds to nearest even
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    assert np.array_equal(oracle.bf16_bits(v.astype(np.float64)), f32_to_bf16_bits(v))


def pin_rmsnorm():
    rng = np.random.default_rng(1)
    T, H = 8, 256
    gamma = f32_to_bf16_bits(1 + 0.1 * rng.standard_normal(H))
    # constant row 2: mean(x^2) = 4, r = 1/sqrt(4 + eps) ~ 0.5, so x*r rounds
    # to 1 in bf16 and xn = gamma exactly
    x = np.full((1, H), 0x4000, dtype=np.uint16)   # bf16 2.0
    assert np.array_equal(oracle.rmsnorm(x, gamma, 1e-6)[0], gamma)
    # eps inside the root: constant row 1 with eps = 3 gives r = 1/sqrt(4) =
    # 1/2 exactly, so xn = gamma / 2 (a power-of-two scaling of bf16, exact)
    x = np.full((1, H), 0x3F80, dtype=np.uint16)   # bf16 1.0
    half_gamma = f32_to_bf16_bits(bits_f64(gamma) * 0.5)
    assert np.array_equal(oracle.rmsnorm(x, gamma, 3.0)[0], half_gamma)
    # r = 1/sqrt(mean + eps) as two fp32 roundings (a worked case found by a
    # search over fp32 values in [1, 2)): for a row of ones and eps = 32865
    # 2^-23, sqrt(1 + eps) rounded to fp32 and its reciprocal rounded give
    # exactly 1 - 2^-9, a bf16 tie that goes to even (1.0); the reciprocal
    # square root of 1 + eps itself lies below 1 - 2^-9 and would give 1 - 2^-8
    eps = 32865 * 2.0 ** -23
    assert 1.0 / math.sqrt(1.0 + eps) < 1.0 - 2.0 ** -9 - 2.0 ** -30
    ones = np.full(H, 0x3F80, dtype=np.uint16)
    assert np.all(oracle.rmsnorm(x, ones, eps)[0] == 0x3F80)
    # xn = bf16((x r) gamma), each product rounded to fp32 (a worked case found
    # by a search, its value derived here in exact arithmetic with explicit
    # IEEE roundings): 255 ones and one x = 1.2890625 (gamma 0.7265625 there,
    # ones elsewhere), eps = 33 / 4096.  x (r gamma), and a single rounding of
    # x r gamma to bf16, both give the bf16 value one above.
    from fractions import Fraction as Fr
    assert _sqrt_rne(Fr(9, 4), 24) == Fr(3, 2)  # the exact helpers themselves
    assert float(_sqrt_rne(Fr(2), 24)) == float(np.sqrt(np.float32(2.0)))
    assert float(_rne(Fr(1, 3), 24)) == float(np.float32(1.0) / np.float32(3.0))
    xv, gv, ev = Fr(1.2890625), Fr(0.7265625), Fr(33, 4096)
    ss = 255 + xv * xv
    assert _rne(ss, 24) == ss                   # exact in fp32
    r = _rne(1 / _sqrt_rne(_rne(ss / 256 + ev, 24), 24), 24)
    want = _rne(_rne(_rne(xv * r, 24) * gv, 24), 8)
    assert _rne(_rne(xv * _rne(r * gv, 24), 24), 8) != want
    assert _rne(xv * r * gv, 8) != want
    row = np.full((1, 256), 0x3F80, dtype=np.uint16)
    row[0, 77] = 0x3FA5                         # 1.2890625
    gam = np.full(256, 0x3F80, dtype=np.uint16)
    gam[77] = 0x3F3A                            # 0.7265625
    got = oracle.rmsnorm(row, gam, float(ev))[0, 77]
    assert bits_f64(np.array([got]))[0] == float(want)
    # mean = ss / H as a rounded fp32 division (a worked case at H = 384,
    # eps = 0, exact arithmetic): 382 ones, 3.5625 and 3.984375; the output at
    # 3.5625 is 3.453125, where ss times the rounded 1/384 gives 3.4375
    av, bv = Fr(3.5625), Fr(3.984375)
    ss = 382 + av * av + bv * bv
    assert _rne(ss, 24) == ss
    r = _rne(1 / _sqrt_rne(_rne(ss / 384, 24), 24), 24)
    want = _rne(_rne(av * r, 24), 8)
    r_recip = _rne(1 / _sqrt_rne(_rne(ss * _rne(Fr(1, 384), 24), 24), 24), 24)
    assert _rne(_rne(av * r_recip, 24), 8) != want
    row = np.full((1, 384), 0x3F80, dtype=np.uint16)
    row[0, 5], row[0, 300] = 0x4064, 0x407F     # 3.5625, 3.984375
    got = oracle.rmsnorm(row, np.full(384, 0x3F80, dtype=np.uint16), 0.0)[0, 5]
    assert bits_f64(np.array([got]))[0] == float(want) == 3.453125
    # with eps = 0, scaling x by a power of two leaves xn bit-identical
    x = f32_to_bf16_bits(rng.standard_normal((T, H)))
    x4 = f32_to_bf16_bits(bits_f64(x) * 4.0)
    assert np.array_equal(oracle.rmsnorm(x, gamma, 0.0), oracle.rmsnorm(x4, gamma, 0.0))
    # library routine: torch rms_norm in fp32, within one bf16 ulp
    xt = torch.from_numpy(bits_f64(x).astype(np.float32))
    gt = torch.from_numpy(bits_f64(gamma).astype(np.float32))
    ref = torch.nn.functional.rms_norm(xt, (H,), gt, eps=1e-6).to(torch.float64).numpy()
    got = bits_f64(oracle.rmsnorm(x, gamma, 1e-6))
    ulp = np.abs(ref) * 2.0**-7
    assert np.all(np.abs(got - ref) <= ulp + 1e-30)


def _rne(S, p):
    """A positive Fraction rounded to p significant bits, nearest-even
    (normal range)."""
    from fractions import Fraction
    e = S.numerator.bit_length() - S.denominator.bit_length()
    if Fraction(2) ** e > S:
        e -= 1                               # 2^e <= S < 2^(e+1)
    q = Fraction(2) ** (e - p + 1)
    n = S / q
    m = n.numerator // n.denominator
    rem = n - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return m * q


def _sqrt_rne(S, p):
    """sqrt of a positive Fraction, correctly rounded to p significant bits
    (nearest-even), by integer square roots."""
    from fractions import Fraction
    eS = S.numerator.bit_length() - S.denominator.bit_length()
    if Fraction(2) ** eS > S:
        eS -= 1
    e = eS // 2                              # 2^e <= sqrt(S) < 2^(e+1)
    q = Fraction(2) ** (e - p + 1)
    A = S / (q * q)                          # sqrt(S) / q = sqrt(A)
    n = math.isqrt(A.numerator // A.denominator)
    half = (Fraction(2 * n + 1, 2)) ** 2
    if A > half or (A == half and n % 2 == 1):
        n += 1
    return n * q


def _f32_rne(S):
    """A Fraction rounded to the nearest fp32 (ties to even), as a float;
    infinity past the largest fp32.  Written from the IEEE definition."""
    from fractions import Fraction
    if S == 0:
        return 0.0
    e = S.numerator.bit_length() - S.denominator.bit_length()
    if Fraction(2) ** e > S:
        e -= 1                               # now 2^e <= S < 2^(e+1)
    quantum = Fraction(2) ** max(e - 23, -149)
    q = S / quantum
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * quantum
    return math.inf if v >= Fraction(2) ** 128 else float(v)


def pin_sumsq():
    """The RMSNorm's sum of squares is the exact sum of the bf16 squares,
    rounded once to fp32: checked against exact rational arithmetic on random
    rows of every scale, hand-made ties, fp32's subnormal and overflow ranges,
    and a row whose squares carry across the oracle's 64-bit limbs."""
    from fractions import Fraction

    def ref(rows):
        return np.array([_f32_rne(sum(Fraction(float(v)) ** 2 for v in r)) for r in rows],
                        dtype=np.float32)

    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(256) * 2.0 ** rng.integers(-40, 40) for _ in range(12)]
    wide = rng.standard_normal(256) * 2.0 ** rng.integers(-60, 60, 256)   # 120 binades
    rows.append(wide)
    bits = f32_to_bf16_bits(np.array(rows))
    got = oracle.sumsq(bits)
    assert np.array_equal(got.view(np.uint32), ref(bits_f64(bits)).view(np.uint32))

    def one(vals):
        return float(oracle.sumsq(f32_to_bf16_bits(np.array([vals], dtype=np.float64)))[0])
    big = [2.0 ** 11] * 4                     # squares sum to 2^24
    assert one(big + [1.0]) == 2.0 ** 24                    # 2^24 + 1: a tie, to even
    assert one(big + [1.0, 2.0 ** -30]) == 2.0 ** 24 + 2    # just above the tie
    assert one(big + [1.0] * 3) == 2.0 ** 24 + 4            # 2^24 + 3: tie, to even
    assert one([2.0 ** -70] * 4) == 2.0 ** -138             # exact subnormal
    assert one([2.0 ** -75]) == 0.0                         # half of 2^-149: tie to 0
    assert one([2.0 ** -75] * 3) == 2.0 ** -148             # 1.5 * 2^-149: tie to 2
    assert one([2.0 ** 64]) == math.inf                     # 2^128 overflows
    assert one([0.0] * 8) == 0.0
    # an exact sum just below a tie of fp32's subnormal grid (2^-149 plus
    # 2^-150 - 2^-173): rounding it to 24 bits first would land on the tie
    # and then round up; rounded once it goes down to 2^-149
    terms = [(221, 52), (141, 49), (153, 44), (247, 38), (166, 35), (169, 30), (168, 26),
             (221, 22), (141, 19), (153, 14)]
    vals = [m * 2.0 ** (E - 134) for m, E in terms]
    rest = 2 ** 117 + 2 ** 116 - 2 ** 93 - sum(m * m << (2 * E - 2) for m, E in terms)
    small = []
    while rest > 0:        # the remainder as squares of smaller bf16 values
        E = max(1, (rest.bit_length() - 16 + 2) // 2 + 1)
        while E > 1 and (128 * 128 << (2 * E - 2)) > rest:
            E -= 1
        m = 255 if E > 1 else 127
        while (m * m << (2 * E - 2)) > rest:
            m -= 1
        small.append(m * 2.0 ** (E - 134) if E > 1 or m >= 128 else m * 2.0 ** -133)
        rest -= m * m << (2 * E - 2)
    row = vals + small
    assert sum(Fraction(v) ** 2 for v in row) == Fraction(2 ** 117 + 2 ** 116 - 2 ** 93, 2 ** 266)
    assert one(row) == 2.0 ** -149
    # 4096 squares of 1.9921875 * 2^32 straddle limbs 4 and 5: carries
    carry = [1.9921875 * 2.0 ** 32] * 4096
    assert one(carry) == _f32_rne(4096 * Fraction(1.9921875 * 2.0 ** 32) ** 2)


def pin_gate():
    rng = np.random.default_rng(2)
    T, H, E = 5, 96, 7
    # small integers: every product and partial sum is exact -> exact logits
    xi = rng.integers(-3, 4, (T, H)).astype(np.float64)
    wi = rng.integers(-3, 4, (E, H)).astype(np.float32)
    b = rng.integers(-2, 3, E).astype(np.float32)
    got = oracle.gate_logits(f32_to_bf16_bits(xi), wi, b)
    assert np.array_equal(got, (xi @ wi.T.astype(np.float64) + b).astype(np.float32))
    # random values: within the fp32 error bound of an H-term sum
    x = f32_to_bf16_bits(rng.standard_normal((T, H)))
    wg = (0.02 * rng.standard_normal((E, H))).astype(np.float32)
    ref = bits_f64(x) @ wg.T.astype(np.float64)
    bound = H * 2.0**-24 * (np.abs(bits_f64(x)) @ np.abs(wg.T.astype(np.float64)))
    assert np.all(np.abs(oracle.gate_logits(x, wg) - ref) <= bound)
    # one fused multiply-add per term, ascending h (a worked case): x = [1, 1.5],
    # w = [2, m 2^-47] with m = (2^25 + 1) / 3, so the second product is
    # 2^-23 (1 + 2^-25) exactly.  An FMA chain rounds 2 + 2^-23 + 2^-48 up to
    # 2 + 2^-22; rounding the product first (2^-23) leaves an exact tie that
    # rounds to even (2), and so does the descending order (2^-23, then 2).
    m = (2 ** 25 + 1) // 3
    assert 3 * m == 2 ** 25 + 1 and m < 2 ** 24
    xw = f32_to_bf16_bits(np.array([[1.0, 1.5]]))
    ww = np.array([[2.0, m * 2.0 ** -47]], dtype=np.float32)
    assert float(ww[0, 1]) == m * 2.0 ** -47
    assert oracle.gate_logits(xw, ww)[0, 0] == np.float32(2.0 + 2.0 ** -22)


def pin_topk():
    rng = np.random.default_rng(3)
    T, E, k = 64, 16, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[0] = 0.5                      # all equal -> experts 0..k-1
    lg[1, :] = -1.0
    lg[1, [3, 9, 12]] = 2.0          # three-way tie at the top
    lg[2, :2] = [-0.0, 0.0]          # -0 and +0 compare equal
    lg[2, 2:] = -5.0
    idx, w = oracle.topk_softmax(lg, k, renorm=True)
    # numpy's stable argsort on the negated logits: lowest index first on ties
    ref_idx = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    assert np.array_equal(idx, ref_idx)
    assert list(idx[0]) == [0, 1, 2, 3] and np.allclose(w[0], 0.25)
    assert list(idx[1][:3]) == [3, 9, 12] and idx[2][0] == 0
    # renormalised weights = softmax over the chosen logits (scipy)
    ref_w = softmax(np.take_along_axis(lg, idx, 1).astype(np.float64), axis=1)
    assert np.allclose(w, ref_w, rtol=1e-6, atol=1e-7)
    assert np.allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    # without renormalisation: the full softmax probabilities of the chosen
    idx2, w2 = oracle.topk_softmax(lg, k, renorm=False)
    ref_p = np.take_along_axis(softmax(lg.astype(np.float64), axis=1), idx2, 1)
    assert np.allclose(w2, ref_p, rtol=1e-6, atol=1e-7)


def pin_routing():
    rng = np.random.default_rng(4)
    T, k, E = 300, 3, 11
    ti = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ti[:40] = ti[0]                         # many equal keys
    r = oracle.init_routing(ti, E)
    flat = ti.reshape(-1)
    order = np.argsort(flat, kind="stable")     # row -> assignment
    N = T * k
    assert np.array_equal(np.sort(r["row_idx"]), np.arange(N))
    assert np.array_equal(r["row_idx"][order], np.arange(N))
    assert np.array_equal(r["src_token"], order // k)
    assert np.array_equal(r["sorted_ids"], flat[order])
    assert np.array_equal(r["counts"], np.bincount(flat, minlength=E))
    assert r["offsets"][0] == 0 and r["offsets"][-1] == N
    assert np.array_equal(np.diff(r["offsets"]), r["counts"])
    c, o = oracle.expert_tokens(r["sorted_ids"], E)
    assert np.array_equal(c, r["counts"]) and np.array_equal(o, r["offsets"])
    bad = ti.copy()
    bad[5, 1] = E
    with pytest.raises(oracle.OracleError):
        oracle.init_routing(bad, E)


def pin_expert_mlp():
    rng = np.random.default_rng(5)
    n, H, I = 6, 40, 24              # H != I catches a transposed w2
    xe = f32_to_bf16_bits(rng.standard_normal((n, H)))
    w13 = f32_to_bf16_bits(0.2 * rng.standard_normal((2 * I, H)))
    w2 = f32_to_bf16_bits(0.2 * rng.standard_normal((H, I)))
    act, yb, yf = oracle.expert_mlp(xe, w13, w2, want_f64=True)
    X, W13, W2 = bits_f64(xe), bits_f64(w13), bits_f64(w2)
    g = X @ W13[:I].T                 # products of bf16 are exact in fp64
    u = X @ W13[I:].T
    ref_act = oracle.bf16_bits(g * expit(g) * u)   # SiLU(g) = g * sigmoid(g)
    assert np.array_equal(act, ref_act)
    ref_y = bits_f64(act) @ W2.T
    assert np.allclose(yf, ref_y, rtol=1e-12, atol=1e-15)
    assert np.array_equal(yb, oracle.bf16_bits(yf))
    # SwiGLU special cases: SiLU(0) = 0 and SiLU(g) -> g for large g
    xe1 = np.zeros((1, H), dtype=np.uint16)
    xe1[0, 0] = 0x3F80                 # one-hot 1.0
    w = np.zeros((2 * I, H), dtype=np.uint16)
    w[0, 0] = 0x4180                   # gate 16
    w[I, 0] = 0x3F80                   # up 1
    w[I + 1, 0] = 0x4000               # gate 0, up 2 -> 0
    a1, _ = oracle.expert_mlp(xe1, w, w2)
    assert a1[0, 0] == 0x4180 and a1[0, 1] == 0
    # grouped with one group == dense
    off = np.array([0, n], dtype=np.int32)
    ga, gy = oracle.grouped_mlp(xe, off, w13[None], w2[None])
    assert np.array_equal(ga, act) and np.array_equal(gy, yb)


def pin_finalize():
    rng = np.random.default_rng(6)
    T, H, E, k = 50, 32, 6, 3
    x = f32_to_bf16_bits(rng.standard_normal((T, H)))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = oracle.topk_softmax(lg, k)
    r = oracle.init_routing(idx, E)
    ex = oracle.permute(x, r["src_token"])
    # identity experts (y = expanded x): the renormalised weights sum to 1
    out = oracle.finalize(ex, r["row_idx"], w)
    assert np.allclose(out, bits_f64(x), rtol=4e-7, atol=1e-30)
    sh = rng.standard_normal((T, H))
    out2 = oracle.finalize(ex, r["row_idx"], w, sh)
    assert np.allclose(out2, bits_f64(x) + sh, rtol=1e-6, atol=1e-6)
    # unrounded routed rows (the fp32-y reading): identity experts on float64
    # rows that no bf16 value represents, and a hand-summed token
    xf = rng.standard_normal((T, H))
    exf = np.ascontiguousarray(xf[r["src_token"]])
    out3 = oracle.finalize(exf, r["row_idx"], w, sh)
    assert np.allclose(out3, xf + sh, rtol=1e-6, atol=1e-6)
    # distinct rows per slot: a token's sum taken by hand, slot by slot
    yr = rng.standard_normal((T * k, H))
    out4 = oracle.finalize(yr, r["row_idx"], w)
    for t in (0, 7, T - 1):
        hand = sum(float(w[t, j]) * yr[r["row_idx"][t * k + j]] for j in range(k))
        assert np.allclose(out4[t], hand, rtol=1e-14, atol=1e-14)


def pin_worked_example():
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        ex = json.load(f)
    s = ex["shapes"]
    T, H, E, k, I = s["T"], s["H"], s["E"], s["k"], s["I"]
    x = f32_to_bf16_bits(np.array(ex["x"], dtype=np.float32))
    wg = np.array(ex["wg"], dtype=np.float32)
    w13 = np.zeros((E, 2 * I, H), dtype=np.float32)
    w2 = np.zeros((E, H, I), dtype=np.float32)
    for e in range(E):
        w13[e, :, 0] = [e, 0, 1, 1]
        w13[e, :, 1] = [1, -1, 2, 0.5]
        w2[e, :, 0] = [1, -1, 0.5, 0]
        w2[e, :, 1] = [0, 0, 0, 1]
    from moe_inputs import Workload
    wl = Workload("worked", T=T, H=H, E=E, k=k, I=I)
    inputs = dict(x=torch.from_numpy(bits_f64(x).astype(np.float32)).to(torch.bfloat16),
                  gamma=None, wg=wg, gate_bias=None,
                  w13=torch.from_numpy(w13).to(torch.bfloat16),
                  w2=torch.from_numpy(w2).to(torch.bfloat16), w13_s=None, w2_s=None)
    out, idx, w = oracle.layer_tokens(inputs, wl)
    exp = ex["expected"]
    assert idx.tolist() == exp["topk_idx"]
    assert np.allclose(w, exp["topk_w"], rtol=1e-7, atol=0)
    assert np.allclose(out, exp["out"], rtol=0, atol=exp["out_tolerance"])
    a, _ = oracle.expert_mlp(x[:1], f32_to_bf16_bits(w13[1]), f32_to_bf16_bits(w2[1]))
    assert np.array_equal(bits_f64(a)[0], exp["act_token0_expert1"])
    a, _ = oracle.expert_mlp(x[:1], f32_to_bf16_bits(w13[3]), f32_to_bf16_bits(w2[3]))
    assert np.array_equal(bits_f64(a)[0], exp["act_token0_expert3"])
    a, _ = oracle.expert_mlp(x[1:], f32_to_bf16_bits(w13[0]), f32_to_bf16_bits(w2[0]))
    assert np.array_equal(bits_f64(a)[0], exp["act_token1"])


def pin_layer_brute_force():
    """Whole layer vs a per-token loop with no routing, no sort and no
    permutation, written with numpy matmuls (tiny workload, seed 0), with the
    routed expert outputs rounded to bf16 and, in the fp32-y reading, not."""
    wl = WORKLOADS["tiny"]
    d = make_inputs(wl, 0)
    out, idx, w = oracle.layer_tokens(d, wl)
    out_f, idx_f, w_f = oracle.layer_tokens(d, wl, y_f32=True)
    assert np.array_equal(idx_f, idx) and np.array_equal(w_f, w)
    X = d["x"].to(torch.float64).numpy()
    WG = d["wg"].to(torch.float64).numpy()
    W13 = d["w13"].to(torch.float64).numpy()
    W2 = d["w2"].to(torch.float64).numpy()
    logits = X @ WG.T
    srt = np.sort(logits, axis=1)[:, ::-1]
    margin = srt[:, wl.k - 1] - srt[:, wl.k]
    assert margin.min() > 1e-5          # no near-ties for this seed
    for t in range(wl.T):
        sel = np.argsort(-logits[t], kind="stable")[: wl.k]
        assert sorted(sel) == sorted(idx[t])
        p = softmax(logits[t, sel])
        acc = np.zeros(wl.H)
        acc_f = np.zeros(wl.H)
        for j, e in enumerate(sel):
            g = X[t] @ W13[e, : wl.I].T
            u = X[t] @ W13[e, wl.I:].T
            a = bits_f64(oracle.bf16_bits(g * expit(g) * u))
            yf = a @ W2[e].T
            acc += p[j] * bits_f64(oracle.bf16_bits(yf))
            acc_f += p[j] * yf
        assert np.allclose(out[t], acc, rtol=1e-5, atol=1e-7), t
        assert np.allclose(out_f[t], acc_f, rtol=1e-5, atol=1e-7), t
    # the two readings differ by the bf16 rounding of y only (<= half an ulp)
    assert not np.array_equal(out, out_f)


def pin_layer_shared_rmsnorm():
    """A small workload with RMSNorm, a gate offset and a shared expert:
    the layer equals the composition of its steps, and the shared term is
    exactly the shared expert's unrounded output."""
    from moe_inputs import Workload
    wl = Workload("small", T=24, H=64, E=6, k=2, I=32, I_s=48, rmsnorm=True,
                  gamma_std=0.1, skew_s=1.2, skew_beta=0.5)
    d = make_inputs(wl, 3)
    out, idx, w = oracle.layer_tokens(d, wl)
    xn = oracle.rmsnorm(d["x"], d["gamma"], wl.eps)
    lg = oracle.gate_logits(xn, d["wg"], d["gate_bias"])
    i2, w2_ = oracle.topk_softmax(lg, wl.k)
    assert np.array_equal(idx, i2) and np.array_equal(w, w2_)
    r = oracle.init_routing(i2, wl.E)
    ex = oracle.permute(xn, r["src_token"])
    _, y = oracle.grouped_mlp(ex, r["offsets"], d["w13"], d["w2"])
    _, _, ys = oracle.expert_mlp(xn, d["w13_s"], d["w2_s"], want_f64=True)
    ref = oracle.finalize(y, r["row_idx"], w, ys)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-15)
    # the fp32-y reading: the same composition over each group's unrounded rows
    yf = np.zeros((ex.shape[0], wl.H))
    w13b, w2b = d["w13"], d["w2"]
    for e in range(wl.E):
        r0, r1 = int(r["offsets"][e]), int(r["offsets"][e + 1])
        if r1 > r0:
            yf[r0:r1] = oracle.expert_mlp(ex[r0:r1], w13b[e], w2b[e], want_f64=True)[2]
    out_f, _, _ = oracle.layer_tokens(d, wl, y_f32=True)
    assert np.allclose(out_f, oracle.finalize(yf, r["row_idx"], w, ys), rtol=1e-12, atol=1e-15)
    # with the shared expert's weights zeroed the shared term vanishes
    d0 = dict(d, w2_s=torch.zeros_like(d["w2_s"]))
    out0, _, _ = oracle.layer_tokens(d0, wl)
    assert np.allclose(out - out0, ys, rtol=1e-12, atol=1e-15)
    out0_f, _, _ = oracle.layer_tokens(d0, wl, y_f32=True)
    assert np.allclose(out_f - out0_f, ys, rtol=1e-12, atol=1e-15)


def pin_ep_local_rerouting():
    """EP local steps: the rerouted order equals numpy's stable sort of the
    received rows by (local expert, source rank, arrival); finalize undoes it;
    one source rank with everything for one expert is the identity."""
    rng = np.random.default_rng(7)
    ep, El, H = 4, 6, 8
    counts = rng.integers(0, 5, (ep, El)).astype(np.int32)
    counts[1, :] = 0                      # a rank that sent nothing
    counts[2, 3] = 9
    total = int(counts.sum())
    R = total + 5
    x = rng.integers(0, 60000, (R, H)).astype(np.uint16)
    lx, src, lc, lo = oracle.local_rerouting(x, counts)
    rank = np.repeat(np.repeat(np.arange(ep), El), counts.reshape(-1))
    expert = np.repeat(np.tile(np.arange(El), ep), counts.reshape(-1))
    order = np.lexsort((np.arange(total), rank, expert))   # expert, then rank, then arrival
    assert np.array_equal(src[:total], order)
    assert np.all(src[total:] == -1)
    assert np.array_equal(lx[:total], x[order])
    assert np.array_equal(lc, counts.sum(0)) and lo[0] == 0 and lo[-1] == total
    assert np.array_equal(np.diff(lo), lc)
    back = oracle.local_finalize_rerouting(lx[:total], src, total, R)
    assert np.array_equal(back[:total], x[:total])
    one = np.array([[7]], dtype=np.int32)
    _, s1, _, _ = oracle.local_rerouting(x[:7], one)
    assert np.array_equal(s1, np.arange(7))


PINS = [pin_bf16_rounding, pin_rmsnorm, pin_sumsq, pin_gate, pin_topk, pin_routing,
        pin_expert_mlp, pin_finalize, pin_worked_example, pin_layer_brute_force,
        pin_layer_shared_rmsnorm, pin_ep_local_rerouting]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ------------------------------------------------------------------ mutants
# (original text, planted mistake) in moe_oracle.c
MUTANTS = {
    "rms_no_sqrt": ("1.0f / sqrtf(mean + eps)", "1.0f / (mean + eps)"),
    "sumsq_truncated": ("q += (uint64_t)round_up;", "q += 0;"),
    "sumsq_ties_up": ("round_up = rest || (q & 1);", "round_up = 1;"),
    "sumsq_no_subnormal": ("        lsb = 117;", "        lsb = lsb;"),
    "sumsq_carry_dropped": ("carry = (acc[j] < old || (carry && acc[j] == old)) ? 1 : 0;",
                            "carry = 0;"),
    "sumsq_square_shift": ("const int sh = 2 * (e ? e : 1) - 2;",
                           "const int sh = 2 * (e ? e : 1) - 1;"),
    "rms_no_mean": ("ss / (float)H", "ss"),
    "rms_mean_by_reciprocal": ("ss / (float)H", "ss * (1.0f / (float)H)"),
    "rms_no_eps": ("1.0f / sqrtf(mean + eps)", "1.0f / sqrtf(mean)"),
    "rms_r_in_double": ("1.0f / sqrtf(mean + eps)",
                        "(float)(1.0 / sqrt((double)mean + (double)eps))"),
    "rms_gamma_into_r": ("float v = bf16_to_float(xr[h]) * r;\n            if (gamma)\n                v = v * bf16_to_float(gamma[h]);",
                         "float v = bf16_to_float(xr[h]) * (gamma ? r * bf16_to_float(gamma[h]) : r);"),
    "rms_one_rounding": ("float v = bf16_to_float(xr[h]) * r;\n            if (gamma)\n                v = v * bf16_to_float(gamma[h]);\n            xn[t * H + h] = bf16_from_double((double)v);",
                         "double v = (double)bf16_to_float(xr[h]) * r;\n            if (gamma)\n                v = v * bf16_to_float(gamma[h]);\n            xn[t * H + h] = bf16_from_double(v);"),
    "rms_no_gamma": ("v = v * bf16_to_float(gamma[h]);", "v = v;"),
    "gate_transposed": ("wg[e * H + h], acc)", "wg[h * E + e], acc)"),
    "gate_no_bias": ("acc = acc + bias[e];", "acc = acc;"),
    "gate_mul_then_add": ("acc = fmaf(bf16_to_float(xs[t * H + h]), wg[e * H + h], acc);",
                          "acc = acc + bf16_to_float(xs[t * H + h]) * wg[e * H + h];"),
    "gate_descending_h": ("acc = fmaf(bf16_to_float(xs[t * H + h]), wg[e * H + h], acc);",
                          "acc = fmaf(bf16_to_float(xs[t * H + (H - 1 - h)]), wg[e * H + (H - 1 - h)], acc);"),
    "topk_ties_high": ("l[e] > l[best]", "l[e] >= l[best]"),
    "softmax_sign": ("exp((double)l[topk_idx[t * k + j]] - m) / den",
                     "exp(m - (double)l[topk_idx[t * k + j]]) / den"),
    "no_renorm": ("if (renorm) {", "if (0) {"),
    "renorm_inverted": ("if (renorm) {", "if (!renorm) {"),
    "topk_slots_reversed": ("topk_idx[t * k + j] = (int32_t)best;",
                            "topk_idx[t * k + (k - 1 - j)] = (int32_t)best;"),
    "finalize_unweighted": ("(double)topk_w[t * k + j] *", "1.0 *"),
    "route_src_mod": ("src_token[row] = (int32_t)(a / k);",
                      "src_token[row] = (int32_t)(a % k);"),
    "route_unstable": ("const int32_t row = offsets[e] + fill[e]++;",
                       "const int32_t row = offsets[e + 1] - ++fill[e];"),
    "swiglu_swapped": ("const bf16_t *wgate = w13 + i * H;\n            const bf16_t *wup = w13 + (I + i) * H;",
                       "const bf16_t *wup = w13 + i * H;\n            const bf16_t *wgate = w13 + (I + i) * H;"),
    "silu_sign": ("g / (1.0 + exp(-g))", "g / (1.0 + exp(g))"),
    "down_transposed": ("const bf16_t *wr = w2 + c * I;", "const bf16_t *wr = w2 + c;"),
    "finalize_no_shared": ("s += shared[t * H + c];", "s += 0.0;"),
    "finalize_weight_index": ("(double)topk_w[t * k + j] *", "(double)topk_w[j] *"),
    "bf16_truncate": ("nearbyint(ldexp(m, 8))", "floor(ldexp(m, 8))"),
    "layer_shared_dropped": ("o[c] += ys[c];", "o[c] += 0.0;"),
    "layer_y_f32_rounded": ("of[c] += (double)w[j] * yr[c];",
                            "of[c] += (double)w[j] * (double)bf16_to_float(yb[c]);"),
    "layer_y_f32_no_shared": ("of[c] += ys[c];", "of[c] += 0.0;"),
    "finalize_f64_row_ignored": ("y_exp[(int64_t)row_idx[t * k + j] * H + c];",
                                 "y_exp[(int64_t)row_idx[t * k] * H + c];"),
    "permute_reversed": ("xs + (int64_t)src_token[r] * H,", "xs + (int64_t)src_token[n - 1 - r] * H,"),
    "expert_offsets_not_cumulative": ("offsets[e + 1] = offsets[e] + counts[e];",
                                      "offsets[e + 1] = counts[e];"),
    "grouped_weights_of_group_0": ("w13 + g * 2 * I * H, w2 + g * H * I, H, I,",
                                   "w13, w2, H, I,"),
    "grouped_down_of_other_group": ("w13 + g * 2 * I * H, w2 + g * H * I, H, I,",
                                    "w13 + g * 2 * I * H, w2 + (G - 1 - g) * H * I, H, I,"),
    "ep_rank_off_by_one": ("for (int64_t rr = 0; rr < r; ++rr)",
                           "for (int64_t rr = 0; rr <= r; ++rr)"),
    "ep_finalize_wrong_side": ("memcpy(recv_y + (int64_t)local_src[d] * H, local_y + d * H,",
                               "memcpy(recv_y + d * H, local_y + (int64_t)local_src[d] * H,"),
}


def _build_mutant(src_text, tmpdir, name, old, new):
    assert src_text.count(old) >= 1, f"mutant {name}: pattern not found"
    path_c = os.path.join(tmpdir, f"{name}.c")
    with open(path_c, "w") as f:
        f.write(src_text.replace(old, new))
    path_so = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", path_so, path_c, "-lm"], check=True)
    return path_so


def test_mutants_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")).read()
    survivors = []
    tmpdir = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        for name, (old, new) in MUTANTS.items():
            so = _build_mutant(src, tmpdir, name, old, new)
            caught = False
            with oracle.using_library(so):
                for pin in PINS:
                    try:
                        pin()
                    except (AssertionError, oracle.OracleError, ValueError, IndexError):
                        caught = True
                        break
            if not caught:
                survivors.append(name)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    assert not survivors, f"mutants not caught by any pin: {survivors}"
