"""Seeded synthetic inputs for the MoE feed-forward layer.

This module only draws random tensors with the shapes and value distributions
of the workloads; it holds none of the layer's arithmetic.  Both the CUDA
path (tests, bench) and the CPU oracle receive the very same tensors from it.

Workloads follow the MoE layer described on "NPU HunyuanImage-3.0模型推理优化实践"
(sections "MoE TP优化" and "GMM使能&&Routing优化"): bf16 activations and
weights, an fp32 gate weight, merged gate/up weight ``w13 [E, 2I, H]`` (rows
0..I-1 gate, I..2I-1 up) and down weight ``w2 [E, H, I]``.

Generation runs on the requested device with torch's own seeded generator
(CPU: mt19937, CUDA: Philox), so a CPU draw and a CUDA draw of the same seed
differ; every comparison uses one draw and copies it to both sides.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "skew_bias"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    H: int            # hidden size
    E: int            # routed experts
    k: int            # experts per token
    I: int            # routed expert intermediate size
    I_s: int = 0      # shared expert intermediate size (0 = no shared expert)
    rmsnorm: bool = False
    eps: float = 1e-6
    renorm: bool = True
    x_std: float = 1.0
    w_std: float = 0.02
    wg_std: float = 0.02
    gamma_std: float = 0.0      # gamma = 1 + gamma_std * N(0,1) (bf16)
    skew_s: float = 0.0         # Zipf exponent of the per-expert gate offsets
    skew_beta: float = 0.0      # scale of the offsets (calibrated, see below)
    note: str = ""

    @property
    def N(self) -> int:
        return self.T * self.k

    def flops(self) -> float:
        """Algorithmic GEMM flops of one layer pass (gate excluded)."""
        return 6.0 * self.N * self.H * self.I + 6.0 * self.T * self.H * self.I_s

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Zipf scale for the skewed workload: the smallest beta (to 3 significant
# digits) for which the seed-0 draw on a CUDA device (the draw the GPU tests
# and the benchmark use) leaves 16 of 64 experts without a token.  Found by
# tests/golden/calibrate_skew.py --device cuda, which takes the routing
# decisions from the oracle only; its output is
# tests/golden/skew_calibration_cuda.json (the seed-0 CPU draw gives 2.51,
# tests/golden/skew_calibration.json).
SKEW_BETA_SEED0 = 2.58

WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", T=64, H=128, E=8, k=2, I=256, x_std=1.0,
                 note="tiny MoE FFN, top-2, no shared expert"),
        Workload("balanced-4k", T=4096, H=2048, E=64, k=8, I=1024, x_std=0.02,
                 note="near-uniform routing, x and weights ~N(0,0.02)"),
        Workload("imagegen-16k", T=16384, H=4096, E=64, k=8, I=3072, I_s=3072,
                 rmsnorm=True, x_std=1.0, gamma_std=0.1,
                 note="image-gen MoE block: shared expert + RMSNorm"),
        Workload("skewed-32k", T=32768, H=4096, E=64, k=8, I=3072, x_std=1.0,
                 skew_s=1.2, skew_beta=SKEW_BETA_SEED0,
                 note="Zipf(1.2) gate offsets, 16/64 experts idle"),
        Workload("smallbatch-8", T=8, H=4096, E=64, k=8, I=3072, I_s=3072,
                 rmsnorm=True, x_std=1.0, gamma_std=0.1,
                 note="weight-streaming bound"),
        Workload("smallbatch-64", T=64, H=4096, E=64, k=8, I=3072, I_s=3072,
                 rmsnorm=True, x_std=1.0, gamma_std=0.1,
                 note="weight-streaming bound"),
        Workload("smallbatch-256", T=256, H=4096, E=64, k=8, I=3072, I_s=3072,
                 rmsnorm=True, x_std=1.0, gamma_std=0.1,
                 note="weight-streaming bound"),
    ]
}


def _gen(device: str, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF)
    return g


def _normal(shape, std, device, seed, stream, dtype, chunk_rows=None):
    """N(0, std^2) drawn in fp32 and rounded once to ``dtype`` (RNE)."""
    g = _gen(device, seed, stream)
    out = torch.empty(shape, dtype=dtype, device=device)
    if chunk_rows is None or shape[0] <= chunk_rows:
        out.copy_(torch.randn(shape, generator=g, device=device).mul_(std))
        return out
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        sub = (r1 - r0,) + tuple(shape[1:])
        out[r0:r1].copy_(torch.randn(sub, generator=g, device=device).mul_(std))
    return out


def skew_bias(E: int, s: float, beta: float, seed: int, device="cpu") -> torch.Tensor:
    """Per-expert gate offsets b_e = -beta * s * ln(rank_e), rank a seeded
    permutation of 1..E (the Zipf(s) log-weights, scaled by beta)."""
    g = _gen("cpu", seed, 99)
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    b = -beta * s * torch.log(rank)
    return b.to(torch.float32).to(device)


def make_inputs(w: Workload, seed: int = 0, device: str = "cpu",
                T: Optional[int] = None, only=None) -> dict:
    """Draw every input of one layer pass.  ``T`` overrides the token count
    (the weights do not depend on it); ``only`` limits the draw to the named
    tensors (the others are None).  Every tensor has its own generator
    stream, so a partial draw equals the same tensors of a full draw."""
    T = w.T if T is None else T
    H, E, I, I_s = w.H, w.E, w.I, w.I_s
    bf = torch.bfloat16
    want = (lambda n: True) if only is None else (lambda n: n in set(only))
    d = dict(x=None, gamma=None, wg=None, gate_bias=None, w13=None, w2=None,
             w13_s=None, w2_s=None)
    if want("x"):
        d["x"] = _normal((T, H), w.x_std, device, seed, 1, bf, chunk_rows=4096)
    if w.rmsnorm and want("gamma"):
        if w.gamma_std > 0:
            d["gamma"] = (1.0 + _normal((H,), w.gamma_std, device, seed, 2,
                                        torch.float32)).to(bf)
        else:
            d["gamma"] = torch.ones(H, dtype=bf, device=device)
    if want("wg"):
        d["wg"] = _normal((E, H), w.wg_std, device, seed, 3, torch.float32)
    if w.skew_s > 0 and want("gate_bias"):
        d["gate_bias"] = skew_bias(E, w.skew_s, w.skew_beta, seed, device)
    if want("w13"):
        d["w13"] = _normal((E, 2 * I, H), w.w_std, device, seed, 4, bf, chunk_rows=4)
    if want("w2"):
        d["w2"] = _normal((E, H, I), w.w_std, device, seed, 5, bf, chunk_rows=4)
    if I_s > 0 and want("w13_s"):
        d["w13_s"] = _normal((2 * I_s, H), w.w_std, device, seed, 6, bf)
    if I_s > 0 and want("w2_s"):
        d["w2_s"] = _normal((H, I_s), w.w_std, device, seed, 7, bf)
    return d
