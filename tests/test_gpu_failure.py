"""Failure detection on the GPU without a GPU fault.

The pipeline waits of every kernel are bounded: a wait that runs past its
limit records MOE_DEV_TIMEOUT in the caller's status word and the kernel
returns.  Here a kernel waits on a barrier that nothing completes (a flag
nothing sets); the test checks that the call ends on its own, that the bit
is set, and that the context still runs the layer correctly afterwards.
The other device-side checks (bad expert ids, bad group offsets, unsorted
ids) are provoked from the host with invalid inputs in test_gpu_steps.py.
"""
import os
import subprocess
import sys
import time

import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounded_wait_reports_timeout_and_context_survives():
    moe.build()
    st = moe.new_status(DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.selftest_wait_timeout(st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) & moe.DEV_TIMEOUT
    assert 0.5 < dt < 30.0, dt
    # the context is intact: a small top-k still matches its definition
    lg = torch.tensor([[0.1, 2.0, -1.0, 2.0]], device=DEV)
    idx, w = moe.gate_topk(lg, 2)
    assert idx.cpu().tolist() == [[1, 3]]
    assert torch.allclose(w.cpu(), torch.tensor([[0.5, 0.5]]))


@pytest.mark.parametrize("kernel", ["single", "pair", "wide"])
def test_each_gemm_kernel_subprocess(kernel):
    """Every grouped-GEMM kernel (one CTA per 128-row tile, CTA pairs on
    256 x 256 tiles, CTA pairs on 256 x 512 tiles where the shapes allow)
    passes the grouped-GEMM and layer parity tests when forced with
    MOE_GEMM_KERNEL (the default picks per launch; the choice is read once
    per process, hence the child process)."""
    env = dict(os.environ, MOE_GEMM_KERNEL=kernel)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_steps.py"),
           os.path.join(ROOT, "tests", "test_gpu_layer.py"),
           "-k", "grouped or small_all or second_stream"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
