"""moe_init_routing_noalloc: init_routing for callers that cannot allocate.

Some callers of this library only receive input and output pointers and have
no way to get device scratch memory (their host framework owns every
allocation, or a cudaMalloc is not allowed where they run).  The no-alloc
entry point keeps its routing histogram in a fixed array inside the library
instead of a caller workspace.  This test calls it through the C ABI twice in
a row, on different inputs, and checks that every output equals the regular
workspace entry point's (index work: bit-exact), that the largest call the
built-in array holds (its last entry in use) still matches, and that a call
one routing chunk larger is refused.

The file sorts last so that a run stopping at the first failure has already
run every other test; it passes on its own in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_routing_fp32_gb300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(topk_idx, x, E):
    T, k = topk_idx.shape
    H = x.shape[1]
    N = T * k
    out = dict(expanded_x=torch.full((N, H), -1, dtype=torch.int16, device=DEV).view(
                   torch.bfloat16),
               row_idx=torch.full((N,), -7, dtype=torch.int32, device=DEV),
               src_token=torch.full((N,), -7, dtype=torch.int32, device=DEV),
               sorted_ids=torch.full((N,), -7, dtype=torch.int32, device=DEV),
               counts=torch.full((E,), -7, dtype=torch.int32, device=DEV),
               offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=DEV))
    st = moe.new_status(DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = moe.lib().moe_init_routing_noalloc(
        _p(topk_idx), _p(x), T, H, E, k, _p(out["expanded_x"]), _p(out["row_idx"]),
        _p(out["src_token"]), _p(out["sorted_ids"]), _p(out["counts"]), _p(out["offsets"]),
        _p(st), stream)
    assert rc == 0, moe.STATUS_NAMES.get(rc, rc)
    return out, st


def _case(T, k, E, H, seed):
    rng = np.random.default_rng(seed)
    w = rng.pareto(1.2, E) + 0.01
    idx = np.stack([rng.choice(E, k, replace=False, p=w / w.sum()) for _ in range(T)])
    x = torch.randn((T, H), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    return torch.from_numpy(idx.astype(np.int32)).to(DEV), x.to(DEV)


def test_noalloc_matches_workspace_entry_point_twice():
    moe.build()
    # two calls in a row with different inputs (the second must not see the
    # first call's leftovers in the shared array)
    for T, k, E, H, seed in [(3000, 8, 64, 256, 1), (777, 4, 200, 128, 2),
                             (300, 8, 64, 128, 3)]:
        idx, x = _case(T, k, E, H, seed)
        ref = moe.init_routing(idx, x, E)
        got, st = _noalloc(idx, x, E)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for key in ("row_idx", "src_token", "sorted_ids", "counts", "offsets"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["expanded_x"].view(torch.int16),
                           ref["expanded_x"].view(torch.int16))


def test_noalloc_largest_accepted_size_matches():
    # ceil(T/32) * E == 262144: every entry of the built-in array is used
    T, k, E = 131072, 2, 64
    rng = np.random.default_rng(4)
    # k distinct experts per token, uniform
    idx = torch.from_numpy(np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)).to(DEV)
    ref = moe.init_routing(idx, None, E, with_rows=False)
    N = T * k
    got = {key: torch.full((n,), -7, dtype=torch.int32, device=DEV)
           for key, n in (("row_idx", N), ("src_token", N), ("sorted_ids", N), ("counts", E),
                          ("offsets", E + 1))}
    st = moe.new_status(DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = moe.lib().moe_init_routing_noalloc(
        _p(idx), None, T, 0, E, k, None, _p(got["row_idx"]), _p(got["src_token"]),
        _p(got["sorted_ids"]), _p(got["counts"]), _p(got["offsets"]), _p(st), stream)
    assert rc == 0, moe.STATUS_NAMES.get(rc, rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for key in ("row_idx", "src_token", "counts", "offsets"):
        assert torch.equal(got[key], ref[key]), key


def test_noalloc_rejects_sizes_beyond_its_array():
    E, k = 64, 2
    T = 32 * (262144 // E) + 1          # one chunk more than the array holds
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    x = torch.zeros((T, 128), dtype=torch.bfloat16, device=DEV)
    N = T * k
    bufs = [torch.empty(N, dtype=torch.int32, device=DEV) for _ in range(3)]
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    rc = moe.lib().moe_init_routing_noalloc(
        _p(idx), _p(x), T, 128, E, k, None, _p(bufs[0]), _p(bufs[1]), _p(bufs[2]), _p(counts),
        _p(offsets), None, None)
    assert rc == 3   # MOE_ERR_WORKSPACE_TOO_SMALL
