"""CPU pins of the oracle's residual add (the layer's output added once per token to a residual
stream r: y = r + sum_k gate_k FFN_k(x) + sum_s FFN_s(x)).

Pinned against what the definition fixes: bf16 residual bits decode to the values their bit
patterns define; a zero residual leaves the layer unchanged; the residual part of the output is
r itself -- added once, not per slot and not gate-weighted -- whatever the routing, the number of
shared experts or the token subset.
"""
import numpy as np

import oracle
import synth
from synth import WORKLOADS

W = WORKLOADS["tiny_fp32"].with_(T=24, d=64, N=8, M=2, kpg=2, I=48)


def layer(inp, n_shared=0, **kw):
    return oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                                inp["w_down"], W.M, W.kpg, n_shared=n_shared, **kw)


def test_bf16_bits_decode_to_their_values():
    bits = np.array([[0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000, 0x3EAA]], dtype=np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 0.0, 0.33203125]
    np.testing.assert_array_equal(oracle.values64(bits)[0], want)
    f = np.array([[1.5, -0.25]], dtype=np.float32)
    np.testing.assert_array_equal(oracle.values64(f), f.astype(np.float64))


def test_zero_residual_leaves_the_layer():
    inp = synth.layer_inputs(W, seed=4)
    y0 = layer(inp)["y"]
    np.testing.assert_array_equal(layer(inp, residual=np.zeros((W.T, W.d), np.float32))["y"], y0)


def test_residual_is_added_once_unweighted_whatever_the_routing():
    rng = np.random.default_rng(5)
    r = rng.standard_normal((W.T, W.d)).astype(np.float32)
    for n_shared, seed in ((0, 4), (2, 6)):
        inp = synth.layer_inputs(W, seed=seed, n_shared=n_shared)
        for bias in (inp["bias"], inp["bias"][::-1].copy()):  # two different routings
            inp["bias"] = bias
            y0 = layer(inp, n_shared)["y"]
            y1 = layer(inp, n_shared, residual=r)["y"]
            np.testing.assert_allclose(y1 - y0, r.astype(np.float64), rtol=0, atol=1e-12)


def test_residual_rows_follow_the_token_subset():
    inp = synth.layer_inputs(W, seed=7)
    r = synth.normal(9, synth.TID_X, (W.T, W.d), 1.0, "bf16")
    toks = np.array([3, 17, 0, 23], dtype=np.int32)
    full = layer(inp, residual=r)["y"]
    part = layer(inp, tokens=toks, residual=r)["y"]
    np.testing.assert_array_equal(part, full[toks])
