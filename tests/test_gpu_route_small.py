"""GPU parity of routing from x at small and medium batches, and of the fused permutation.

moge_route with x for a few tokens (T <= 64) computes the scores on CUDA cores and routes them
in the same launch; moge_layer_forward additionally permutes all tokens there.  Larger batches
take the tensor-core router and the separate permutation; the same checks hold for both:
  - scores within a few fp32 rounding steps of the oracle's double-accumulated scores;
  - routing equal to the oracle's on the GPU's own scores (bit-exact selection), and equal to
    the oracle's on its own scores except near-ties (probability gap < 1e-6);
  - counts, offsets, group loads and imbalance bit-exact against the oracle's permutation of
    the GPU routing; moge_route and moge_layer_forward agree bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, config, dev, host, routing_mismatch_ok, run_layer, upload_layer
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

SCORE_TOL = {"bf16": 1e-4, "f32": 2e-5}  # |GPU fp32 score - oracle score|, scores are O(1..10)


def route_with_x(w, d_inp, mode):
    c = config(w)
    ws = moge.alloc_workspace(c)
    logits = torch.empty((w.T, w.N), dtype=torch.float32, device=DEV)
    idx = torch.full((w.T, w.K), -5, dtype=torch.int32, device=DEV)
    gate = torch.empty((w.T, w.K), dtype=torch.float32, device=DEV)
    moge.moge_route(c, mode, d_inp["x"], d_inp["w_router"], d_inp["bias"], logits, idx, gate, ws)
    torch.cuda.synchronize()
    return host(logits), host(idx), host(gate)


@pytest.mark.parametrize("T,d,N,M,kpg,dtype", [
    (32, 4096, 64, 8, 2, "bf16"),     # the decode layer's router
    (1, 4096, 64, 8, 2, "bf16"),
    (7, 512, 24, 4, 3, "bf16"),       # ragged token and expert tiles
    (64, 256, 16, 4, 1, "f32"),       # the tiny all-fp32 layer's router
    (200, 768, 256, 8, 1, "bf16"),    # wide groups
    (256, 1024, 64, 1, 5, "bf16"),    # one group = global top-K
])
@pytest.mark.parametrize("mode", [moge.MOGE_ROUTE_GROUPED, moge.MOGE_ROUTE_GLOBAL_TOPK])
def test_small_router_scores_and_selection(T, d, N, M, kpg, dtype, mode):
    w = WORKLOADS["decode_t32"].with_(T=T, d=d, N=N, M=M, kpg=kpg, I=64, dtype=dtype)
    inp = synth.layer_inputs(w, seed=T + 3 * N, with_experts=False)
    d_inp = upload_layer(inp)
    name = "grouped" if mode == moge.MOGE_ROUTE_GROUPED else "global"
    l_gpu, idx, gate = route_with_x(w, d_inp, mode)
    l_ref = oracle.router_logits(inp["x"], inp["w_router"], inp["bias"])
    assert np.max(np.abs(l_gpu.astype(np.float64) - l_ref)) < SCORE_TOL[dtype]
    # selection and gates are exact functions of the GPU's own scores
    own = oracle.route(l_gpu, M, kpg, mode=name)
    np.testing.assert_array_equal(idx, own["idx"])
    assert np.max(np.abs(gate.astype(np.float64) - own["gate64"])) <= 1e-6
    # against the oracle's own scores only near-ties may differ
    ref = oracle.route(l_ref, M, kpg, mode=name)
    if mode == moge.MOGE_ROUTE_GROUPED:
        near = routing_mismatch_ok(idx, ref["idx"], ref["p"], M, kpg)
        assert len(near) <= max(2, T // 100)


@pytest.mark.parametrize("T", [1, 5, 32, 64, 129, 256])
def test_fused_route_and_permutation_in_layer(T):
    """Inside moge_layer_forward a few tokens are routed and permuted in one launch."""
    w = WORKLOADS["decode_t32"].with_(T=T, d=512, I=128)
    inp = synth.layer_inputs(w, seed=40 + T)
    d_inp = upload_layer(inp)
    got = run_layer(w, d_inp)
    perm = oracle.permute(got["topk_idx"], w.N)
    np.testing.assert_array_equal(got["counts"], perm["counts"])
    np.testing.assert_array_equal(got["offsets"], perm["offsets"])
    loads, score = oracle.imbalance(perm["counts"], T, w.M)
    np.testing.assert_array_equal(got["group_load"], loads)
    assert got["score"] == score == 0.0
    own = oracle.route(got["logits"], w.M, w.kpg)
    np.testing.assert_array_equal(got["topk_idx"], own["idx"])
    # the stand-alone routing call gives the same scores, indices and gates bit for bit
    l2, idx2, gate2 = route_with_x(w, d_inp, moge.MOGE_ROUTE_GROUPED)
    np.testing.assert_array_equal(l2, got["logits"])
    np.testing.assert_array_equal(idx2, got["topk_idx"])
    np.testing.assert_array_equal(gate2, got["topk_gate"])


def test_small_router_repeated_calls_reuse_the_ticket():
    """The last-CTA counter resets itself: many calls in a row on one workspace stay correct."""
    w = WORKLOADS["decode_t32"].with_(T=48, d=1024, I=64)
    inp = synth.layer_inputs(w, seed=9, with_experts=False)
    d_inp = upload_layer(inp)
    first = route_with_x(w, d_inp, moge.MOGE_ROUTE_GROUPED)
    c = config(w)
    ws = moge.alloc_workspace(c)
    logits = torch.empty((w.T, w.N), dtype=torch.float32, device=DEV)
    idx = torch.empty((w.T, w.K), dtype=torch.int32, device=DEV)
    gate = torch.empty((w.T, w.K), dtype=torch.float32, device=DEV)
    for _ in range(50):
        idx.fill_(-1)
        moge.moge_route(c, moge.MOGE_ROUTE_GROUPED, d_inp["x"], d_inp["w_router"], d_inp["bias"], logits, idx,
                        gate, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(idx), first[1])
    np.testing.assert_array_equal(host(logits), first[0])
    # the ticket word is back at zero
    assert int(host(ws[256:260].view(torch.int32))[0]) == 0
