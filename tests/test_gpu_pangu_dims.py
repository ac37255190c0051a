"""GPU parity at Pangu Pro MoE's own dimensions with top-1 per group (K' = 1, K = 8) and its 4
shared experts: hidden 5120, 64 routed experts in 8 groups, expert intermediate 1344 (not on the
pages; chosen from the parameter totals they print).  Decode batch (32 tokens) in full; prefill
batch (8192 tokens) with all routing checked and the output rows of tokens that reach every tile
of every touched routed expert and of every shared expert.  Each group receives
exactly T tokens (K' = 1), so the imbalance score is 0.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import expert_covering_tokens, upload_layer
from synth import WORKLOADS
from test_gpu_shared import check_shared, run_shared

pytestmark = pytest.mark.gpu

S = 4


@pytest.fixture(scope="module")
def prefill_inputs():
    w = WORKLOADS["pangu_k1_t8192"]
    return w, synth.layer_inputs(w, n_shared=S)


def test_pangu_dims_decode_k1_with_shared_experts(prefill_inputs):
    wp, inp_p = prefill_inputs
    w = WORKLOADS["pangu_k1_t32"]
    inp = dict(inp_p, x=inp_p["x"][: w.T].copy())
    got = run_shared(w, upload_layer(inp), S)
    check_shared(w, inp, got, S)
    counts = np.diff(got["offsets"])
    loads = counts.reshape(w.M, w.G).sum(axis=1)
    assert np.all(loads == w.T)                       # K' = 1: one expert per group per token
    assert got["score"][0] == 0.0


@pytest.mark.slow
def test_pangu_dims_prefill_k1_with_shared_experts(prefill_inputs):
    """Output rows of the tokens that reach every tile of every touched routed expert (first and
    last row, one row in every 128-row block of each segment) and every 128-row block of each
    shared expert's segment (one row per token in token order: tokens 0, 128, 256, ...)."""
    w, inp = prefill_inputs
    got = run_shared(w, upload_layer(inp), S)
    perm = oracle.permute(got["topk_idx"], w.N)
    toks, touched = expert_covering_tokens(perm["offsets"], perm["row_token"], w.T)
    toks = np.union1d(toks, np.arange(0, w.T, 128)).astype(np.int32)
    assert len(np.unique(got["topk_idx"][toks])) == touched
    check_shared(w, inp, got, S, tokens=toks)
    assert got["score"][0] == 0.0
