"""moge_permute_noalloc against moge_permute.

The no-workspace entry point serves callers that cannot allocate device memory
(a runtime whose pool owns all of HBM and hands over only inputs and outputs,
or a loop that must not call cudaMalloc).  Its scratch is a static device array
shared by every call, so two calls in a row must each match the workspace
entry point exactly: counts, offsets, pair rows, row tokens and gathered rows
are integer or copy results, compared bit for bit.

The file is named so that pytest collects it after every other test file: a
run that stops at the first failure (-x) has then run everything else before
a failure here.  The tests themselves depend on no order: each passes alone in
a fresh process as well as after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import sparse_router_gemm_global_b300 as moge
import synth
from sparse_router_gemm_global_b300 import binding

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _inputs(T, N, M, kpg, d, seed):
    c = moge.make_config(T, d, N, M, kpg, 64, "bf16")
    ws = moge.alloc_workspace(c)
    idx = torch.empty((max(T, 1), M * kpg), dtype=torch.int32, device=DEV)  # one row for T = 0: not NULL
    x = torch.zeros((max(T, 1), d), dtype=torch.bfloat16, device=DEV)
    if T > 0:
        l = synth.route_logits(seed, T, N)
        gate = torch.empty((T, M * kpg), dtype=torch.float32, device=DEV)
        moge.moge_route(c, moge.MOGE_ROUTE_GROUPED, None, None, None, torch.from_numpy(l).to(DEV), idx, gate, ws)
        x = torch.from_numpy(synth.normal(seed, synth.TID_X, (T, d), 1.0, "bf16").view(np.int16)).to(DEV)
        x = x.view(torch.bfloat16)
    return c, ws, idx, x


def _outputs(c, with_pair_row=True):
    T, K, N, d = c.T, c.M * c.k_per_group, c.N, c.d
    rows = max(T * K, 1)
    return {"counts": torch.full((N,), -1, dtype=torch.int32, device=DEV),
            "offsets": torch.full((N + 1,), -1, dtype=torch.int32, device=DEV),
            "pair_row": torch.full((max(T, 1), K), -2, dtype=torch.int32, device=DEV) if with_pair_row else None,
            "row_token": torch.full((rows,), -3, dtype=torch.int32, device=DEV),
            "x_perm": torch.zeros((rows, d), dtype=torch.bfloat16, device=DEV)}


def _run_both(c, ws, idx, x, with_pair_row=True):
    ref, got = _outputs(c, with_pair_row), _outputs(c, with_pair_row)
    moge.moge_permute(c, idx, x, ref["counts"], ref["offsets"], ref["pair_row"], ref["row_token"],
                      ref["x_perm"], ws)
    moge.moge_permute_noalloc(c, idx, x, got["counts"], got["offsets"], got["pair_row"], got["row_token"],
                              got["x_perm"])
    torch.cuda.synchronize()
    for k in ref:
        if ref[k] is not None:
            assert torch.equal(got[k], ref[k]), k
    return got


@pytest.mark.parametrize("calls", [[(5000, 64, 8, 2, 128, 1), (3001, 256, 8, 1, 64, 2)],
                                   [(300, 16, 4, 1, 64, 3), (200, 16, 4, 2, 64, 4)]])
def test_noalloc_permute_matches_workspace_permute_twice(calls):
    for (T, N, M, kpg, d, seed) in calls:
        _run_both(*_inputs(T, N, M, kpg, d, seed))


def test_noalloc_row_gather_without_pair_row():
    """Without pair_row the rows are copied row by row through row_token (the other copy path)."""
    for (T, N, M, kpg, d, seed) in [(1000, 64, 8, 2, 64, 5), (257, 32, 8, 1, 128, 6)]:
        _run_both(*_inputs(T, N, M, kpg, d, seed), with_pair_row=False)


def test_noalloc_empty_batch_zeroes_counts_and_offsets():
    """T = 0 after a non-empty call: counts and offsets are all zero, as moge_permute writes them."""
    _run_both(*_inputs(700, 64, 8, 2, 64, 7))
    got = _run_both(*_inputs(0, 64, 8, 2, 64, 8))
    assert torch.count_nonzero(got["counts"]) == 0 and torch.count_nonzero(got["offsets"]) == 0


def test_noalloc_rejects_beyond_static_scratch():
    # ceil(T/256) * N counts must fit the 256 KiB array: 65536 tokens x 1024 experts do not.  The
    # buffers are real and sized for the configuration, although the call is rejected first.
    T, N, M, kpg = 65536, 1024, 8, 1
    c = moge.make_config(T, 0, N, M, kpg, 0, "f32")
    idx = torch.zeros((T, M * kpg), dtype=torch.int32, device=DEV)
    counts = torch.zeros(N, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(N + 1, dtype=torch.int32, device=DEV)
    with pytest.raises(moge.MoGEError) as e:
        moge.moge_permute_noalloc(c, idx, None, counts, offsets, None, None, None)
    assert e.value.status == 2  # MOGE_ERR_UNSUPPORTED, raised before any launch
    assert binding.load().moge_permute_noalloc(None, None, None, None, None, None, None, None, None) == 1
