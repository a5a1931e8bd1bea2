"""CPU checks of the numerical argument behind the RMSNorm kernels' fast path
for the sum of squares (csrc/router.cu, "sum of squares").

The RMSNorm of "NPU HunyuanImage-3.0模型推理优化实践" (section "RmsNorm算子优化")
takes the row's sum of squares; the reading used here is the exact sum of the
bf16 squares rounded once to fp32, which the oracle computes with a
fixed-point sum.  The CUDA kernels reach the same value by one warp per row:
per lane and pair half, each square goes into an fp32 accumulator held inside
one binade (start 2^(2ex+9)), its rounding error into a second one (start
3 2^(2ex-8)) and that one's rounding error into an fp32 residual; the
accumulators' offsets become exact integers; the residual's error is bounded
by (4 vpl + 5) vpl 2^-17 units of 2^(2ex-30); the value is decided when both
ends of that interval round to the same fp32 number.

This file restates that arithmetic in numpy float32 (round to nearest, like
the packed instructions) - a model of the kernel, not the oracle - and
checks on rows of many kinds that
  - the accumulators never leave their binades and every two-sum step is
    exact (so the integer parts are exact);
  - the fp32 residual lies within the stated bound of the exact sum of the
    rounding errors;
  - every decided value equals the oracle's exactly rounded sum, and exact
    ties are never decided in the fast path.
"""
import math

import numpy as np
import pytest

import oracle

F32 = np.float32


def _bf16_rne(a):
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _u16(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _round24(v):
    """v / 2^16 (an integer v > 0 in fixed point) rounded to 24 significant
    bits, nearest-even, in units of the fixed point's integer part."""
    top = v.bit_length() - 1
    shift = top - 23
    q, rem, half = v >> shift, v & ((1 << shift) - 1), 1 << (shift - 1)
    if rem > half or (rem == half and (q & 1)):
        q += 1
    return q << (shift - 16)


def fast_path(row, check=True, s2_start=None):
    """The warp's fast path on one bf16 row (float32 values).  Returns
    (value or None when undecided, the residual's error / its bound).
    s2_start overrides the second accumulator's start (a planted mistake)."""
    H = row.size
    nvec = H // 8
    vpl = (nvec + 31) // 32
    amax = float(np.max(np.abs(row)))
    assert amax > 0
    ex = math.frexp(amax)[1] - 1
    assert -20 <= ex <= 40
    s1, s2 = F32(2.0 ** (2 * ex + 9)), F32(3 * 2.0 ** (2 * ex - 8))
    if s2_start is not None:
        s2 = F32(s2_start(ex))
    k1, k2 = F32(2.0 ** (14 - 2 * ex)), F32(2.0 ** (30 - 2 * ex))
    u2 = 2.0 ** (2 * ex - 30)
    vec = np.zeros((32 * vpl, 8), F32)
    vec[:nvec] = row.reshape(nvec, 8)
    X = vec.reshape(vpl, 32, 4, 2)          # [vector i of the lane, lane, word, pair half]
    a3 = np.zeros((32, 2), F32)
    errs = []
    n1 = n2 = 0
    for g in range(0, vpl, 16):
        a1 = np.full((32, 2), s1, F32)
        a2 = np.full((32, 2), s2, F32)
        for i in range(g, min(g + 16, vpl)):
            for j in range(4):
                x = X[i, :, j, :]
                sq = x * x
                t1 = a1 + sq
                r1 = sq - (t1 - a1)
                t2 = a2 + r1
                e = r1 - (t2 - a2)
                if check:
                    # binades: [2^(2ex+9), 2^(2ex+10)) and [2^(2ex-7), 2^(2ex-6))
                    assert np.all(np.frexp(t1)[1] - 1 == 2 * ex + 9)
                    assert np.all(np.frexp(t2)[1] - 1 == 2 * ex - 7)
                    for a, b, c, d in zip(a1.ravel(), sq.ravel(), t1.ravel(), r1.ravel()):
                        assert math.fsum([float(a), float(b), -float(c), -float(d)]) == 0.0
                    for a, b, c, d in zip(a2.ravel(), r1.ravel(), t2.ravel(), e.ravel()):
                        assert math.fsum([float(a), float(b), -float(c), -float(d)]) == 0.0
                errs.extend(float(v) for v in e.ravel())
                a3 = a3 + e
                a1, a2 = t1, t2
        d1, d2 = (a1 - s1) * k1, (a2 - s2) * k2
        assert np.all(d1 == np.rint(d1)) and np.all(d2 == np.rint(d2))
        n1 += int(np.sum(d1.astype(np.int64)))
        n2 += int(np.sum(d2.astype(np.int64)))
    r = (a3[:, 0] + a3[:, 1]).astype(F32)
    for off in (16, 8, 4, 2, 1):
        r = (r + r[np.arange(32) ^ off]).astype(F32)
    assert np.all(r == r[0])
    exact_e = math.fsum(errs)
    bound = (4 * vpl + 5) * vpl * 2.0 ** -17 * (1 + 2.0 ** -20) * u2
    seen = abs(float(r[0]) - exact_e) / bound
    T = (n1 << 16) + n2
    a16 = F32(F32(r[0] * k2) * F32(65536.0))
    err = (4 * vpl + 6) * vpl // 2 + 2
    lo = (T << 16) + math.floor(float(a16)) - err
    hi = (T << 16) + math.ceil(float(a16)) + err
    res = _round24(lo)
    if _round24(hi) != res:
        return None, seen
    return float(F32(res * u2)), seen


def _rows(H, rng):
    rows = []
    for scale in (1.0, 2.0 ** -10, 2.0 ** 12, 2.0 ** -19, 2.0 ** 38):
        rows += [rng.standard_normal(H) * scale for _ in range(2)]
    rows.append(rng.standard_normal(H) * 2.0 ** rng.integers(-60, 30, H))
    top = (2 - 2 ** -7)
    rows.append(np.full(H, top))                          # every square near the binade's top
    rows.append(np.where(np.arange(H) % 2 == 0, top, -top))
    rows.append(rng.uniform(0.9, 1.0, H) * np.sign(rng.standard_normal(H)))
    big = np.zeros(H)
    big[0] = 2.0 ** 10
    big[1:] = rng.standard_normal(H - 1) * 2.0 ** -3      # small squares next to a big one
    rows.append(big)
    rounds_up = np.full(H, 6.9375)                          # first-level errors all negative
    rounds_up[0] = 2.0 ** 10
    rows.append(rounds_up)
    return [_bf16_rne(np.asarray(r, np.float32)) for r in rows]


@pytest.mark.parametrize("H", [4096, 1024, 8192, 384])
def test_fast_path_matches_the_exactly_rounded_sum(H):
    rng = np.random.default_rng(1000 + H)
    rows = _rows(H, rng)
    ref = oracle.sumsq(np.stack([_u16(r) for r in rows]))
    decided = 0
    for k, row in enumerate(rows):
        got, seen = fast_path(row, check=(k % 4 == 0))
        assert seen <= 1.0, (k, seen)
        if got is not None:
            decided += 1
            assert np.float32(got) == ref[k], (k, got, ref[k])
    assert decided >= len(rows) - 1


def test_exact_ties_go_to_the_slow_path():
    """Sums that sit exactly on a rounding tie of fp32 are never decided by
    the fast path (the interval holds the tie)."""
    H = 256
    z = np.zeros(H, np.float32)
    cases = []
    for vals in ([2.0 ** 11] * 4 + [1.0], [2.0 ** 11] * 4 + [1.0] * 3,
                 [1.0] + [2.0 ** -13] * 3 + [2.0 ** -14] * 3 + [2.0 ** -15] * 3 + [2.0 ** -16] * 4):
        r = z.copy()
        r[:len(vals)] = vals
        cases.append(_bf16_rne(r))
    for row in cases:
        got, _ = fast_path(row)
        assert got is None


def test_second_accumulator_needs_its_centred_start():
    """The rounding errors of the first accumulator take both signs; started
    at the bottom of its binade (2^(2ex-7), as a truncating split would), the
    second accumulator leaves the binade on a row with negative errors and
    the check above catches it."""
    rng = np.random.default_rng(11)
    H = 1024
    big = np.zeros(H, np.float32)
    big[0] = 2.0 ** 10
    # squares of about 0.75 of the first grid (2^6 here): each rounds up and
    # leaves an error of about -16
    big[1:] = 6.9375 * np.sign(rng.standard_normal(H - 1))
    row = _bf16_rne(big)
    fast_path(row)                                        # the kernel's start: fine
    with pytest.raises(AssertionError):
        fast_path(row, s2_start=lambda ex: 2.0 ** (2 * ex - 7))
