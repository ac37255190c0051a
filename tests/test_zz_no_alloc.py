"""moge_permute_noalloc against moge_permute (runs last: pytest collects this file after the others).

The no-workspace entry point serves callers that cannot allocate device memory
(a runtime whose pool owns all of HBM and hands over only inputs and outputs,
or a loop that must not call cudaMalloc).  Its scratch is a static device array
shared by every call, so two calls in a row must each match the workspace
entry point exactly: counts, offsets, pair rows, row tokens and gathered rows
are integer or copy results, compared bit for bit.
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
    l = synth.route_logits(seed, T, N)
    c = moge.make_config(T, d, N, M, kpg, 64, "bf16")
    ws = moge.alloc_workspace(c)
    idx = torch.empty((T, M * kpg), dtype=torch.int32, device=DEV)
    gate = torch.empty((T, M * kpg), dtype=torch.float32, device=DEV)
    moge.moge_route(c, moge.MOGE_ROUTE_GROUPED, None, None, None, torch.from_numpy(l).to(DEV), idx, gate, ws)
    x = torch.from_numpy(synth.normal(seed, synth.TID_X, (T, d), 1.0, "bf16").view(np.int16)).to(DEV)
    return c, ws, idx, x.view(torch.bfloat16)


def _outputs(c):
    T, K, N, d = c.T, c.M * c.k_per_group, c.N, c.d
    return {"counts": torch.full((N,), -1, dtype=torch.int32, device=DEV),
            "offsets": torch.full((N + 1,), -1, dtype=torch.int32, device=DEV),
            "pair_row": torch.full((T, K), -2, dtype=torch.int32, device=DEV),
            "row_token": torch.full((T * K,), -3, dtype=torch.int32, device=DEV),
            "x_perm": torch.zeros((T * K, d), dtype=torch.bfloat16, device=DEV)}


@pytest.mark.parametrize("calls", [[(5000, 64, 8, 2, 128, 1), (3001, 256, 8, 1, 64, 2)],
                                   [(300, 16, 4, 1, 64, 3), (200, 16, 4, 2, 64, 4)]])
def test_noalloc_permute_matches_workspace_permute_twice(calls):
    for (T, N, M, kpg, d, seed) in calls:
        c, ws, idx, x = _inputs(T, N, M, kpg, d, seed)
        ref, got = _outputs(c), _outputs(c)
        moge.moge_permute(c, idx, x, ref["counts"], ref["offsets"], ref["pair_row"], ref["row_token"],
                          ref["x_perm"], ws)
        moge.moge_permute_noalloc(c, idx, x, got["counts"], got["offsets"], got["pair_row"], got["row_token"],
                                  got["x_perm"])
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), k


def test_noalloc_rejects_beyond_static_scratch():
    # ceil(T/256) * N counts must fit the 256 KiB array: 65536 tokens x 1024 experts do not
    c = moge.make_config(65536, 0, 1024, 8, 1, 0, "f32")
    with pytest.raises(moge.MoGEError) as e:
        moge.moge_permute_noalloc(c, 0x7F0000000000, None, 0x7F0000000000, 0x7F0000000000, None, None, None)
    assert e.value.status == 2  # MOGE_ERR_UNSUPPORTED, raised before any launch
    assert binding.load().moge_permute_noalloc(None, None, None, None, None, None, None, None, None) == 1
