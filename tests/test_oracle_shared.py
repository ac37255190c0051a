"""CPU pins of the oracle's shared-expert layer (every token visits every shared expert; their
SwiGLU outputs are added with weight 1 to the gated routed combine).

Pinned against special cases the definition fixes: zero shared weights leave the routed layer
unchanged; a shared expert that is a copy of routed expert e adds exactly that expert's FFN; the
shared sum does not depend on the order of the shared experts; the shared experts' output is
independent of routing (any scores give the same shared part).
"""
import numpy as np

import oracle
import synth
from synth import WORKLOADS

W = WORKLOADS["tiny_fp32"].with_(T=24, d=64, N=8, M=2, kpg=2, I=48)


def inputs(n_shared, seed=3):
    return synth.layer_inputs(W, seed=seed, n_shared=n_shared)


def layer(inp, n_shared, **kw):
    return oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                                inp["w_down"], W.M, W.kpg, n_shared=n_shared, **kw)


def test_routed_part_of_the_inputs_is_unchanged_by_shared_experts():
    a, b = inputs(0), inputs(3)
    for k in ("w_gate", "w_up", "w_down"):
        np.testing.assert_array_equal(b[k][:W.N], a[k])
        assert b[k].shape[0] == W.N + 3


def test_zero_shared_weights_leave_the_routed_layer():
    inp = inputs(2)
    for k in ("w_gate", "w_up", "w_down"):
        inp[k][W.N:] = 0
    y0 = layer(inputs(0), 0)["y"]
    np.testing.assert_array_equal(layer(inp, 2)["y"], y0)


def test_shared_copy_of_a_routed_expert_adds_that_expert():
    inp = inputs(1)
    e = 5
    for k in ("w_gate", "w_up", "w_down"):
        inp[k][W.N] = inp[k][e]
    toks = np.arange(W.T, dtype=np.int32)
    y_routed = layer(inp, 0)["y"]
    y = layer(inp, 1)["y"]
    own = oracle.expert_ffn_pairs(toks, np.full(W.T, e, dtype=np.int32), inp["x"], inp["w_gate"], inp["w_up"],
                                  inp["w_down"])
    np.testing.assert_allclose(y - y_routed, own, rtol=0, atol=1e-12)


def test_shared_sum_is_order_free_and_routing_free():
    inp = inputs(3)
    toks = np.arange(W.T, dtype=np.int32)
    a = oracle.shared_experts_tokens(toks, W.N, 3, inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    rev = {k: inp[k].copy() for k in ("w_gate", "w_up", "w_down")}
    for k in rev:
        rev[k][W.N:] = inp[k][W.N:][::-1]
    b = oracle.shared_experts_tokens(toks, W.N, 3, inp["x"], rev["w_gate"], rev["w_up"], rev["w_down"])
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    other = np.random.default_rng(0).standard_normal((W.T, W.N)).astype(np.float32)
    y1, y2 = layer(inp, 3), layer(inp, 3, logits=other)
    r1, r2 = layer(inp, 0), layer(inp, 0, logits=other)
    np.testing.assert_allclose(y1["y"] - r1["y"], y2["y"] - r2["y"], rtol=0, atol=1e-12)
