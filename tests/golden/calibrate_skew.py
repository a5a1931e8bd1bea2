"""Calibrate the Zipf scale beta of the skewed workload (T=32768, H=4096,
E=64, k=8): the smallest beta, to 3 significant digits, for which the
seed-0 draw leaves 16 of the 64 experts (25%) without any token.

The routing decisions come from the oracle only (its fp32 gate and its
top-k); the inputs come from moe_inputs.  The result is written to
skew_calibration.json beside this script (or --out); the CUDA draw's result,
skew_calibration_cuda.json, is the value copied by hand into
moe_inputs.SKEW_BETA_SEED0.

    python tests/golden/calibrate_skew.py [--device cpu|cuda]

``--device`` picks where the seeded generator draws x and wg (a CPU draw and
a CUDA draw differ); the arithmetic always runs in the CPU oracle.
"""
import argparse
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_inputs import WORKLOADS, skew_bias, make_inputs  # noqa: E402

TARGET_ZERO = 16


def zero_experts(logits0, wl, beta, seed):
    b = skew_bias(wl.E, wl.skew_s, beta, seed).numpy()
    # the oracle adds the offset after the fp32 dot product, one fp32 add
    lg = (logits0 + b[None, :]).astype(np.float32)
    idx, _ = oracle.topk_softmax(lg, wl.k)
    counts = np.bincount(idx.reshape(-1), minlength=wl.E)
    return int((counts == 0).sum()), counts


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--device", default="cpu")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--out", default=None, help="result file (default: beside this script)")
    args = ap.parse_args()
    wl = WORKLOADS["skewed-32k"]
    d = make_inputs(wl, args.seed, device=args.device, only=("x", "wg"))
    logits0 = oracle.gate_logits(d["x"].cpu(), d["wg"].cpu(), None)
    lo, hi = 0.0, 8.0
    assert zero_experts(logits0, wl, hi, args.seed)[0] >= TARGET_ZERO
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if zero_experts(logits0, wl, mid, args.seed)[0] >= TARGET_ZERO:
            hi = mid
        else:
            lo = mid
    beta = float(np.format_float_positional(hi, precision=3, unique=False,
                                            fractional=False, trim="-"))
    while zero_experts(logits0, wl, beta, args.seed)[0] < TARGET_ZERO:
        beta = round(beta + 10 ** (np.floor(np.log10(beta)) - 2), 6)
    nz, counts = zero_experts(logits0, wl, beta, args.seed)
    res = dict(workload=wl.name, seed=args.seed, device=args.device, beta=beta,
               zero_experts=nz, top_share=float(counts.max() / counts.sum()),
               counts=counts.tolist())
    out = args.out or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                   "skew_calibration.json")
    with open(out, "w") as f:
        json.dump(res, f, indent=1)
    print(json.dumps({k: v for k, v in res.items() if k != "counts"}))


if __name__ == "__main__":
    main()
