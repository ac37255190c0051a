"""Pins of the oracle's router projection, expert SwiGLU FFN and combine.

Independent checks: torch float64 library matmuls, hand closed forms, the
identical-experts closed form y = (sum_k gate_k) * FFN(x), linearity in the
gates, and exact bf16 widening.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import WORKLOADS


def torch_ffn(x, wg, wu, wd):
    x, wg, wu, wd = (torch.from_numpy(np.asarray(a, dtype=np.float64)) for a in (x, wg, wu, wd))
    a = x @ wg.T
    u = x @ wu.T
    return (torch.nn.functional.silu(a) * u) @ wd.T


def test_router_logits_vs_numpy_float64():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((40, 96)).astype(np.float32)
    w = (rng.standard_normal((12, 96)) / 10).astype(np.float32)
    b = rng.standard_normal(12).astype(np.float32)
    got = oracle.router_logits(x, w, b)
    ref = (x.astype(np.float64) @ w.astype(np.float64).T + b.astype(np.float64)).astype(np.float32)
    # both are double sums rounded once to fp32; summation order may move one ulp
    assert np.all(np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32)) <= 1)
    assert np.mean(got == ref) > 0.99


def test_ffn_vs_torch_float64():
    rng = np.random.default_rng(2)
    N, I, d = 3, 24, 40
    x = rng.standard_normal((5, d)).astype(np.float32)
    wg = (rng.standard_normal((N, I, d)) / 6).astype(np.float32)
    wu = (rng.standard_normal((N, I, d)) / 6).astype(np.float32)
    wd = (rng.standard_normal((N, d, I)) / 5).astype(np.float32)
    toks = np.array([0, 1, 2, 3, 4, 0, 4], dtype=np.int32)
    exps = np.array([0, 1, 2, 0, 1, 2, 2], dtype=np.int32)
    got = oracle.expert_ffn_pairs(toks, exps, x, wg, wu, wd)
    for i, (t, e) in enumerate(zip(toks, exps)):
        ref = torch_ffn(x[t:t + 1], wg[e], wu[e], wd[e]).numpy()[0]
        assert np.max(np.abs(got[i] - ref)) < 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_ffn_scalar_closed_form():
    # d = I = 1: o = wd * silu(wg*x) * (wu*x)
    for xv, g, u, dn in [(0.5, 2.0, -1.0, 3.0), (-1.25, 0.75, 0.5, -2.0), (0.0, 1.0, 1.0, 1.0)]:
        x = np.array([[xv]], np.float32)
        got = oracle.expert_ffn_pairs([0], [0], x, np.array([[[g]]], np.float32),
                                      np.array([[[u]]], np.float32), np.array([[[dn]]], np.float32))
        a = g * xv
        expect = dn * (a / (1 + math.exp(-a))) * (u * xv)
        assert abs(got[0, 0] - expect) < 1e-15


def test_identical_experts_closed_form():
    # all experts equal: y = (sum_k gate_k) * FFN(x)
    w = WORKLOADS["tiny_fp32"].with_(T=24, d=64, I=32)
    inp = synth.layer_inputs(w, seed=3)
    for k in ("w_gate", "w_up", "w_down"):
        inp[k] = np.ascontiguousarray(np.broadcast_to(inp[k][:1], inp[k].shape))
    r = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                             inp["w_down"], w.M, w.kpg)
    f = oracle.expert_ffn_pairs(np.arange(24), np.zeros(24), inp["x"], inp["w_gate"], inp["w_up"],
                                inp["w_down"])
    expect = r["gate64"].sum(axis=1)[:, None] * f
    assert np.max(np.abs(r["y"] - expect)) < 1e-12 * np.max(np.abs(expect))


def test_combine_linear_in_gates():
    w = WORKLOADS["tiny_fp32"].with_(T=16, d=32, I=16)
    inp = synth.layer_inputs(w, seed=4)
    r = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                             inp["w_down"], w.M, w.kpg)
    toks = np.arange(16)
    y2 = oracle.combine_tokens(toks, r["idx"], 2.5 * r["gate64"], inp["x"], inp["w_gate"],
                               inp["w_up"], inp["w_down"])
    assert np.max(np.abs(y2 - 2.5 * r["y"])) < 1e-13 * np.max(np.abs(y2))


def test_layer_vs_torch_float64_composition():
    """The whole tiny fp32 layer against an independent torch float64 chain."""
    w = WORKLOADS["tiny_fp32"]
    inp = synth.layer_inputs(w)
    r = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                             inp["w_down"], w.M, w.kpg)
    x = torch.from_numpy(inp["x"]).double()
    lg = (x @ torch.from_numpy(inp["w_router"]).double().T).float()  # fp32 scores
    p = torch.softmax(lg.double(), dim=1)
    G = w.G
    y = torch.zeros_like(x)
    for t in range(w.T):
        for g in range(w.M):
            grp = lg[t, g * G:(g + 1) * G]
            order = sorted(range(G), key=lambda j: (-float(grp[j]), j))[:w.kpg]
            for j in order:
                e = g * G + j
                f = torch_ffn(inp["x"][t:t + 1], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])[0]
                y[t] += p[t, e] * f
    ref = y.numpy()
    assert np.max(np.abs(r["y"] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_bf16_arrays_read_as_exact_values():
    w = WORKLOADS["decode_t32"].with_(T=4, d=64, N=8, M=2, I=32)
    inp = synth.layer_inputs(w, seed=8)
    widened = {k: (synth.bf16_to_f32(v) if v.dtype == np.uint16 else v) for k, v in inp.items()}
    a = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                             inp["w_down"], w.M, w.kpg)
    b = oracle.layer_forward(widened["x"], widened["w_router"], widened["bias"], widened["w_gate"],
                             widened["w_up"], widened["w_down"], w.M, w.kpg)
    np.testing.assert_array_equal(a["idx"], b["idx"])
    np.testing.assert_array_equal(a["y"], b["y"])


def identical_experts_residual(w, seed, gate_fn):
    """max |y - (sum_k p_k) FFN(x)| / max |y| for a layer whose experts all share one set of
    weights, y computed by the oracle's combine with gates gate_fn(oracle gates)."""
    inp = synth.layer_inputs(w, seed=seed)
    for k in ("w_gate", "w_up", "w_down"):
        inp[k] = np.ascontiguousarray(np.broadcast_to(inp[k][:1], inp[k].shape))
    r = oracle.route(oracle.router_logits(inp["x"], inp["w_router"], inp["bias"]), w.M, w.kpg)
    toks = np.arange(w.T)
    y = oracle.combine_tokens(toks, r["idx"], gate_fn(r["gate64"]), inp["x"], inp["w_gate"], inp["w_up"],
                              inp["w_down"])
    f = oracle.expert_ffn_pairs(toks, np.zeros(w.T), inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    expect = r["gate64"].sum(axis=1)[:, None] * f
    return np.max(np.abs(y - expect)) / np.max(np.abs(expect))


def test_planted_renormalised_gates_mistake_is_caught():
    # The closed-form check of test_identical_experts_closed_form, run on a planted variant of the
    # combine that renormalises the gates over the selected experts (a plausible misreading of
    # the explainer's section 1, which keeps the global-softmax probabilities): the check accepts
    # the oracle's gates and rejects the variant's by orders of magnitude.
    w = WORKLOADS["tiny_fp32"].with_(T=16, d=32, I=16)
    assert identical_experts_residual(w, 6, lambda g: g) < 1e-12
    assert identical_experts_residual(w, 6, lambda g: g / g.sum(axis=1, keepdims=True)) > 0.1


def test_combine_rows_equals_per_token_combine():
    # the combine step applied to permuted expert outputs gives the per-token combine
    w = WORKLOADS["tiny_fp32"].with_(T=20, d=32, I=16)
    inp = synth.layer_inputs(w, seed=9)
    r = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                             inp["w_down"], w.M, w.kpg)
    rows = oracle.expert_ffn_pairs(r["row_token"], np.repeat(np.arange(w.N), r["counts"]), inp["x"],
                                   inp["w_gate"], inp["w_up"], inp["w_down"])
    y = oracle.combine_rows(rows.astype(np.float32), r["pair_row"], r["gate64"])
    assert np.max(np.abs(y - r["y"])) < 1e-6 * np.max(np.abs(r["y"]))
    # hand case: two rows, weights 0.5 and 2
    rows2 = np.array([[1.0, -2.0], [4.0, 0.5]], dtype=np.float32)
    y2 = oracle.combine_rows(rows2, np.array([[1, 0]]), np.array([[0.5, 2.0]]))
    assert np.array_equal(y2, np.array([[4.0, -3.75]]))
