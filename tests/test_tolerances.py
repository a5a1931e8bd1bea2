"""CPU pins of the layer-output check (tests/_helpers.py: check_out with the
routed one-ulp allowance), on planted differences."""
import numpy as np
import pytest

from tests._helpers import FLIP_FRAC, MAX_ABS, check_out, routed_flip_allowance


def _bits(v):
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_one_routed_ulp_flip_is_admitted_and_no_more():
    n, k, H = 4, 2, 4096
    rng = np.random.default_rng(3)
    y = rng.uniform(-1, 1, (n, k, H)).astype(np.float32)
    y[1, 0, 7] = -4.03125                          # |y| in [4, 8): one bf16 ulp is 2^-5
    w = np.array([[0.5, 0.5], [0.94, 0.06], [0.7, 0.3], [0.6, 0.4]], dtype=np.float32)
    ys = _bits(y)
    ref = np.einsum("nk,nkh->nh", w.astype(np.float64),
                    (ys.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    allow = routed_flip_allowance(ys, w)
    assert allow[1, 7] == pytest.approx(0.94 * 2.0**-5 + 0.06 * 2.0**-8, rel=1e-6)

    gpu = ref.copy()
    gpu[1, 7] += 0.94 * 2.0**-5                    # the routed y one ulp off: 0.029 > 2e-2
    with pytest.raises(AssertionError):
        check_out(gpu, ref, bf16_out=False)       # the bare max-abs bar refuses it
    check_out(gpu, ref, bf16_out=False, flip_allowance=allow)

    worse = gpu.copy()
    worse[1, 7] += 0.03                            # beyond one ulp of every term
    with pytest.raises(AssertionError):
        check_out(worse, ref, bf16_out=False, flip_allowance=allow)

    many = ref.copy()                              # each element within its allowance,
    cols = np.arange(0, H, 64)                     # but 1.6% of them past 2e-2
    assert len(cols) / H > FLIP_FRAC
    many[:, cols] += MAX_ABS + 0.5 * allow[:, cols]
    with pytest.raises(AssertionError):
        check_out(many, ref, bf16_out=False, flip_allowance=allow)


def test_skew_beta_is_the_committed_cuda_calibration():
    """The skewed workload's Zipf scale is the one tests/golden/calibrate_skew.py
    found on the CUDA draw (committed beside it), which leaves 16 of 64
    experts idle; the CPU draw's calibration is kept beside it for reference."""
    import json
    import os
    import moe_inputs
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    cuda = json.load(open(os.path.join(here, "skew_calibration_cuda.json")))
    cpu = json.load(open(os.path.join(here, "skew_calibration.json")))
    assert cuda["device"] == "cuda" and cpu["device"] == "cpu"
    assert cuda["beta"] == moe_inputs.SKEW_BETA_SEED0
    assert moe_inputs.WORKLOADS["skewed-32k"].skew_beta == cuda["beta"]
    assert cuda["zero_experts"] == 16 and cpu["zero_experts"] == 16
