"""CPU checks of the tensor-core gate's arithmetic and of the tolerance the
GPU tests hold it to (tests/_helpers.py: gate_tc_bound).

The gate of "NPU HunyuanImage-3.0模型推理优化实践" (section
"消除gate计算冗余cast算子") is an fp32 linear layer.  The tensor-core gate
splits every fp32 weight into three bf16 parts and sums the exact products
in fp32 in another order than the oracle.  Here, in numpy and independently
of the CUDA code:
  - the three-part split is exact for fp32 weights of magnitude 2^-110 and
    up (every magnitude a gate weight has), within 2^-134 below;
  - a model of the tensor-core sum (per part, blocks of 16 products summed
    exactly and rounded to fp32, accumulated in fp32; the parts added as
    (p1 + p2) + p3) stays inside the per-logit bound and the RMS bound
    against the oracle's sequential fp32 logits;
  - the RMS bound is tight enough to catch a gate that drops the second
    weight part.
"""
import numpy as np

import oracle
import pytest

from tests._helpers import bf16_to_f64, gate_tc_bound, routing_flips


def _bf16_rne(a):
    """fp32 array -> the nearest bf16 values (ties to even), as fp32."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _split3(w):
    w = np.asarray(w, dtype=np.float32)
    w1 = _bf16_rne(w)
    r1 = (w - w1).astype(np.float32)
    w2 = _bf16_rne(r1)
    r2 = (r1 - w2).astype(np.float32)
    w3 = _bf16_rne(r2)
    return w1, w2, w3, r2


def test_three_part_split_is_exact():
    """w1 = bf16(w) leaves a remainder of at most 16 significant bits, w2 =
    bf16(remainder) one of at most 8, which bf16 holds: exact, as long as the
    remainders stay above fp32's subnormal range (|w| >= 2^-110).  Below it
    the parts may be off by half a bf16 subnormal step, 2^-134 at most."""
    rng = np.random.default_rng(11)
    w = (rng.standard_normal(200000) * 0.02).astype(np.float32)
    special = np.array([1.0, -1.0, 1.0 + 2.0**-23, -(1.0 + 2.0**-23), 0.1, 1e-5, 65504.0,
                        np.float32(np.pi), 2.0**-100 * 1.2345, 2.0**-110, 0.0, -0.0],
                       dtype=np.float32)
    w = np.concatenate([w, special, rng.uniform(-1e3, 1e3, 1000).astype(np.float32)])
    w1, w2, w3, r2 = _split3(w)
    # the last remainder already fits bf16, so the third part holds it exactly
    assert np.array_equal(w3, r2)
    exact = w1.astype(np.float64) + w2.astype(np.float64) + w3.astype(np.float64)
    assert np.array_equal(exact, w.astype(np.float64))
    # and each part is a bf16 value
    for p in (w1, w2, w3):
        assert not (p.view(np.uint32) & 0xFFFF).any()
    # near fp32's underflow the split is within 2^-134
    tiny = np.array([3.0e-38, -1.3e-37, 2.0**-120 * 1.37, 1e-40, -7e-45], dtype=np.float32)
    t1, t2, t3, _ = _split3(tiny)
    err = np.abs(t1.astype(np.float64) + t2 + t3 - tiny.astype(np.float64))
    assert (err <= 2.0**-134).all()


def _tc_model_logits(xs_bits, wg, bias):
    """The tensor-core gate's arithmetic, modelled: exact products, blocks of 16
    summed exactly and rounded once to fp32, accumulated in fp32 per part."""
    xs = bf16_to_f64(xs_bits)
    T, H = xs.shape
    parts = _split3(wg)[:3]
    acc = []
    for p in parts:
        a = np.zeros((T, p.shape[0]), dtype=np.float32)
        for k0 in range(0, H, 16):
            blk = xs[:, k0:k0 + 16] @ p[:, k0:k0 + 16].astype(np.float64).T   # exact
            a = (a + blk.astype(np.float32)).astype(np.float32)
        acc.append(a)
    lg = ((acc[0] + acc[1]).astype(np.float32) + acc[2]).astype(np.float32)
    if bias is not None:
        lg = (lg + np.asarray(bias, dtype=np.float32)).astype(np.float32)
    return lg, acc


def test_bound_covers_a_blocked_fp32_sum_and_catches_a_dropped_part():
    rng = np.random.default_rng(5)
    T, H, E = 192, 1024, 24
    x = (rng.standard_normal((T, H))).astype(np.float32)
    xs_bits = (_bf16_rne(x).view(np.uint32) >> 16).astype(np.uint16)
    wg = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.5).astype(np.float32)
    lg_ref = oracle.gate_logits(xs_bits, wg, bias)
    per, rms_b = gate_tc_bound(xs_bits, wg, lg_ref)

    lg, acc = _tc_model_logits(xs_bits, wg, bias)
    d = np.abs(lg.astype(np.float64) - lg_ref.astype(np.float64))
    assert (d <= per).all()
    assert float(np.sqrt(np.mean(d * d))) <= rms_b
    # far inside the per-logit bound: rounding, not a lost term
    assert float(d.max()) < 0.05 * float(per.min())

    # a gate without the second part (bf16 weights plus the third part only)
    lg_bad = ((acc[0] + acc[2]).astype(np.float32) + bias).astype(np.float32)
    d_bad = np.abs(lg_bad.astype(np.float64) - lg_ref.astype(np.float64))
    assert float(np.sqrt(np.mean(d_bad * d_bad))) > rms_b


def test_routing_check_accepts_near_ties_and_rejects_wrong_choices():
    """routing_flips, the GPU tests' routing check, planted on CPU: a swap
    within the bound of a tie passes (reported as a flip), a clearly worse
    expert or a wrong slot order does not."""
    lg = np.array([[3.0, 2.0, 1.0000001, 1.0, -1.0],
                   [5.0, 4.0, 3.0, 2.0, 1.0]], dtype=np.float32)
    per = np.full(lg.shape, 1e-6)
    ref = np.array([[0, 1, 2], [0, 1, 2]], dtype=np.int32)
    assert len(routing_flips(ref, ref, lg, per)) == 0
    near = np.array([[0, 1, 3], [0, 1, 2]], dtype=np.int32)     # 1.0 vs 1.0000001: a near-tie
    assert list(routing_flips(near, ref, lg, per)) == [0]
    with pytest.raises(AssertionError):
        routing_flips(np.array([[0, 1, 4], [0, 1, 2]], dtype=np.int32), ref, lg, per)
    with pytest.raises(AssertionError):                            # slot order not descending
        routing_flips(np.array([[0, 1, 2], [1, 0, 2]], dtype=np.int32), ref, lg, per)
    with pytest.raises(AssertionError):                            # an expert twice
        routing_flips(np.array([[0, 1, 1], [0, 1, 2]], dtype=np.int32), ref, lg, per)
