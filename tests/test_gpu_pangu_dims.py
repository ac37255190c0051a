"""GPU parity at Pangu Pro MoE's own dimensions with top-1 per group (K' = 1, K = 8) and its 4
shared experts: hidden 5120, 64 routed experts in 8 groups, expert intermediate 1344 (not on the
pages; chosen from the parameter totals they print).  Decode batch (32 tokens) in full; prefill
batch (8192 tokens) with all routing checked and 32 sampled output rows.  Each group receives
exactly T tokens (K' = 1), so the imbalance score is 0.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import upload_layer
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
    w, inp = prefill_inputs
    got = run_shared(w, upload_layer(inp), S)
    toks = np.sort(np.random.default_rng(5).choice(w.T, 32, replace=False))
    check_shared(w, inp, got, S, tokens=toks)
    assert got["score"][0] == 0.0
