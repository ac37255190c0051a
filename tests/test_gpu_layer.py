"""GPU parity of the expert FFN, the combine and the whole layer against the oracle.

Tolerances: max|y - ref| <= 2e-2 * max|ref| for bf16 (fp32 accumulation),
<= 1e-5 * max|ref| for the all-fp32 layer.  End-to-end routing may differ from
the oracle's only on near-ties (oracle probability gap < 1e-6); such tokens are
left out of the output comparison and counted.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import (DEV, as_f64, config, dev, expert_covering_tokens, host, max_rel_err, routing_mismatch_ok,
                      run_layer, torch_dtype, upload_layer)
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


def check_layer(w, inp, got, tokens=None, seed_note=""):
    """Routing of all tokens and outputs of `tokens` (all if None) vs the oracle."""
    T = w.T
    ref = oracle.route(oracle.router_logits(inp["x"], inp["w_router"], inp["bias"]), w.M, w.kpg)
    near = routing_mismatch_ok(got["topk_idx"], ref["idx"], ref["p"], w.M, w.kpg)
    assert len(near) <= max(2, T // 1000), f"too many near-tie tokens: {len(near)}"
    # the permutation and loads follow the GPU's own routing exactly
    perm = oracle.permute(got["topk_idx"], w.N)
    np.testing.assert_array_equal(got["counts"], perm["counts"])
    np.testing.assert_array_equal(got["offsets"], perm["offsets"])
    loads, score = oracle.imbalance(perm["counts"], T, w.M)
    np.testing.assert_array_equal(got["group_load"], loads)
    assert got["score"] == 0.0 and np.all(loads == T * w.kpg)
    # gates: the GPU's fp32 softmax of its own scores vs the oracle's, for agreeing tokens
    ok = np.array([t not in near for t in range(T)])
    gate_tol = 2e-4 if w.dtype == "bf16" else 1e-5  # scores differ by accumulation order
    assert np.max(np.abs(got["topk_gate"][ok] - ref["gate64"][ok])) < gate_tol
    # outputs
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    toks = np.array([t for t in toks if t not in near], dtype=np.int32)
    y_ref = oracle.combine_tokens(toks, ref["idx"], ref["gate64"], inp["x"], inp["w_gate"], inp["w_up"],
                                  inp["w_down"])
    err = max_rel_err(got["y"][toks], y_ref)
    assert err <= TOL[w.dtype], f"{w.name}: max rel err {err:.3e} {seed_note}"
    return err, toks


def check_layer_every_expert(w, inp, got):
    """check_layer on the tokens that reach every tile of every touched expert (first and last
    row, and one row in every 128-row block, of each expert's segment of the GPU's permutation):
    every expert the batch touches has its output rows compared."""
    perm = oracle.permute(got["topk_idx"], w.N)
    toks, touched = expert_covering_tokens(perm["offsets"], perm["row_token"], w.T)
    err, compared = check_layer(w, inp, got, tokens=toks)
    checked = np.unique(got["topk_idx"][compared])
    print(f"{w.name}: {len(compared)} tokens compared, {len(checked)} of {touched} touched experts, "
          f"max rel err {err:.3e}")
    assert len(checked) == touched == int(np.count_nonzero(perm["counts"]))
    return err


def test_tiny_fp32_layer():
    w = WORKLOADS["tiny_fp32"]
    inp = synth.layer_inputs(w)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)
    # the fp32 scores themselves: within a few ulp of the oracle's double-then-fp32 scores
    l_ref = oracle.router_logits(inp["x"], inp["w_router"], inp["bias"])
    assert np.max(np.abs(got["logits"] - l_ref)) < 1e-5


@pytest.mark.parametrize("T,d,N,M,kpg,I", [
    (300, 256, 16, 4, 2, 192),     # ragged rows and a ragged intermediate tile
    (129, 512, 32, 8, 1, 256),
    (1, 128, 16, 4, 4, 64),        # one token, K' = G
    (64, 384, 24, 1, 3, 320),      # a single group = global top-K
    (520, 256, 256, 8, 1, 128),    # wide groups (G = 32), many empty experts
    (700, 264, 16, 4, 2, 136),     # hidden size not a multiple of the 64-wide k-block (zero-filled tail)
    (1100, 1024, 64, 8, 2, 256),   # several 256-row tiles per expert, gathered token rows
    (512, 64, 16, 4, 2, 128),      # CTA-pair tiles with a one-k-block gate/up: the next tile id is taken
                                   # and published at the first k-block, the producer runs tiles ahead
])
def test_bf16_layer_shapes(T, d, N, M, kpg, I):
    w = WORKLOADS["decode_t32"].with_(name=f"bf16_{T}_{d}_{N}_{M}_{kpg}_{I}", T=T, d=d, N=N, M=M, kpg=kpg, I=I)
    inp = synth.layer_inputs(w, seed=T + d + N)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)


def test_decode_t32_full():
    w = WORKLOADS["decode_t32"]
    inp = synth.layer_inputs(w)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)


def test_prefill_t8192_every_expert():
    w = WORKLOADS["prefill_t8192"]
    inp = synth.layer_inputs(w)
    got = run_layer(w, upload_layer(inp))
    check_layer_every_expert(w, inp, got)


def test_layer_is_deterministic():
    w = WORKLOADS["decode_t32"].with_(T=700, d=512, I=256)
    d_inp = upload_layer(synth.layer_inputs(w, seed=21))
    a = run_layer(w, d_inp)
    b = run_layer(w, d_inp)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_expert_ffn_and_combine_on_oracle_permutation():
    """moge_expert_ffn on the oracle's own permutation, then moge_combine, each vs the oracle."""
    w = WORKLOADS["decode_t32"].with_(T=333, d=256, I=192)
    inp = synth.layer_inputs(w, seed=5)
    ref = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                               inp["w_down"], w.M, w.kpg)
    c = config(w)
    ws = moge.alloc_workspace(c)
    x_perm = dev(inp["x"][ref["row_token"]])
    y_perm = torch.empty((w.P, w.d), dtype=torch.bfloat16, device=DEV)
    d_inp = upload_layer(inp)
    moge.moge_expert_ffn(c, x_perm, dev(ref["offsets"]), d_inp["w_gate"], d_inp["w_up"], d_inp["w_down"],
                         y_perm, ws)
    torch.cuda.synchronize()
    yp = host(y_perm)
    experts = np.repeat(np.arange(w.N, dtype=np.int32), ref["counts"])
    rows_ref = oracle.expert_ffn_pairs(ref["row_token"], experts, inp["x"], inp["w_gate"], inp["w_up"],
                                       inp["w_down"])
    assert max_rel_err(yp, rows_ref) <= TOL["bf16"]
    # combine of the GPU rows vs the oracle's combine of the same rows
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=DEV)
    moge.moge_combine(c, y_perm, dev(ref["pair_row"]), dev(ref["gate"]), y)
    torch.cuda.synchronize()
    y_ref = oracle.combine_rows(yp, ref["pair_row"], ref["gate"].astype(np.float64))
    # fp32 accumulation of bf16 rows, one final bf16 rounding: within 2 bf16 ulps
    assert np.max(np.abs(as_f64(host(y)) - y_ref) / (np.abs(y_ref) + 1e-3)) < 2 ** -7


def test_empty_layer():
    w = WORKLOADS["decode_t32"].with_(T=0)
    c = config(w)
    ws = moge.alloc_workspace(c)
    d_inp = upload_layer(synth.layer_inputs(w.with_(T=1)))
    y = torch.empty((0, w.d), dtype=torch.bfloat16, device=DEV)
    counts = torch.full((w.N,), 3, dtype=torch.int32, device=DEV)
    moge.moge_layer_forward(c, d_inp["x"], d_inp["w_router"], d_inp["bias"], d_inp["w_gate"], d_inp["w_up"],
                            d_inp["w_down"], y, ws, aux={"counts": counts})
    torch.cuda.synchronize()
    assert np.all(host(counts) == 0)


@pytest.mark.slow
def test_stress_n256_every_expert():
    w = WORKLOADS["stress_n256"]
    inp = synth.layer_inputs(w)
    got = run_layer(w, upload_layer(inp))
    check_layer_every_expert(w, inp, got)


@pytest.mark.parametrize("T", [16, 17, 32, 33, 64, 65, 128, 192, 193, 256, 257, 384, 416, 417])
def test_bf16_layer_at_path_boundaries(T):
    """Token counts on both sides of every switch (K=16 of N=64 experts: T/4 rows per expert on
    average): weights-as-M tile widths 16/32 and the in-GEMM row gather (T <= 32), the small
    router (64/65), 64-token tiles -> 128-token tiles (192/193: 48 rows per expert), one vs several
    permutation chunks (256/257), several 128-token blocks per expert (384), weights-as-M ->
    tokens-as-M tiles (416/417: 104 rows per expert)."""
    w = WORKLOADS["decode_t32"].with_(name=f"edge_{T}", T=T, d=384, I=192)
    inp = synth.layer_inputs(w, seed=100 + T)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)


def test_fp32_layer_many_tokens():
    w = WORKLOADS["tiny_fp32"].with_(name="fp32_t300", T=300, d=128, I=64)
    inp = synth.layer_inputs(w, seed=12)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)


@pytest.mark.parametrize("T", [5, 48])
def test_expert_ffn_standalone_few_tokens(T):
    """moge_expert_ffn on an oracle permutation at weights-as-M sizes (rows read from x_perm)."""
    w = WORKLOADS["decode_t32"].with_(T=T, d=256, I=192)
    inp = synth.layer_inputs(w, seed=6 + T)
    ref = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                               inp["w_down"], w.M, w.kpg)
    c = config(w)
    ws = moge.alloc_workspace(c)
    x_perm = dev(inp["x"][ref["row_token"]])
    y_perm = torch.empty((w.P, w.d), dtype=torch.bfloat16, device=DEV)
    d_inp = upload_layer(inp)
    moge.moge_expert_ffn(c, x_perm, dev(ref["offsets"]), d_inp["w_gate"], d_inp["w_up"], d_inp["w_down"],
                         y_perm, ws)
    torch.cuda.synchronize()
    experts = np.repeat(np.arange(w.N, dtype=np.int32), ref["counts"])
    rows_ref = oracle.expert_ffn_pairs(ref["row_token"], experts, inp["x"], inp["w_gate"], inp["w_up"],
                                       inp["w_down"])
    assert max_rel_err(host(y_perm), rows_ref) <= TOL["bf16"]


@pytest.mark.parametrize("T,dtype", [(5, "bf16"), (333, "bf16"), (2000, "bf16"), (64, "f32")])
def test_expert_ffn_clamps_offsets_to_the_rows(T, dtype):
    """Offsets that no permutation wrote -- a negative start, an empty expert, an end past P -- are
    clamped to [0, P): every row keeps the FFN of the expert whose clamped segment holds it, and
    no row outside y_perm is written (guard rows on both sides, wider than the overshoot, so an
    unclamped store would land in them)."""
    w = WORKLOADS["decode_t32"].with_(T=T, d=256, I=192, dtype=dtype)
    inp = synth.layer_inputs(w, seed=50 + T)
    P, N = w.P, w.N
    rng = np.random.default_rng(T)
    cuts = np.sort(rng.choice(np.arange(1, P), N - 1, replace=False)).astype(np.int32)
    offsets = np.concatenate([[-7], cuts, [P + 300]]).astype(np.int32)
    offsets[5] = offsets[4]                                   # expert 4 empty
    begin = np.clip(offsets[:-1], 0, P)
    end = np.clip(np.maximum(offsets[1:], begin), 0, P)
    experts = np.repeat(np.arange(N, dtype=np.int32), end - begin)
    assert len(experts) == P
    tokens = rng.integers(0, T, size=P).astype(np.int32)
    c = config(w)
    ws = moge.alloc_workspace(c)
    d_inp = upload_layer(inp)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    guard = 512
    buf = torch.full((P + 2 * guard, w.d), 5.0, dtype=tdt, device=DEV)
    moge.moge_expert_ffn(c, dev(inp["x"][tokens]), dev(offsets), d_inp["w_gate"], d_inp["w_up"],
                         d_inp["w_down"], buf[guard:guard + P], ws)
    torch.cuda.synchronize()
    got = host(buf)
    sentinel = host(torch.full((1, w.d), 5.0, dtype=tdt))[0]
    assert np.all(got[:guard] == sentinel) and np.all(got[guard + P:] == sentinel)
    rows_ref = oracle.expert_ffn_pairs(tokens, experts, inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    assert max_rel_err(got[guard:guard + P], rows_ref) <= TOL[dtype]


def test_combine_treats_out_of_range_rows_as_absent():
    """pair_row entries outside [0, T*K) (-1 from a skipped expert id, or past the last row) add
    nothing to the token's output."""
    w = WORKLOADS["decode_t32"].with_(T=200, d=256, I=64)
    rng = np.random.default_rng(3)
    yp = synth.normal(8, synth.TID_X, (w.P, w.d), 1.0, "bf16")
    pair_row = rng.permutation(w.P).astype(np.int32).reshape(w.T, w.K)
    gate = rng.random((w.T, w.K)).astype(np.float32)
    absent = rng.random(pair_row.shape) < 0.15
    pair_row[absent] = np.resize(np.array([-1, w.P, w.P + 7, 1 << 30], dtype=np.int32), int(absent.sum()))
    c = config(w)
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=DEV)
    moge.moge_combine(c, dev(yp), dev(pair_row), dev(gate), y)
    torch.cuda.synchronize()
    y_ref = oracle.combine_rows(yp, np.where(absent, 0, pair_row), np.where(absent, 0.0, gate.astype(np.float64)))
    assert np.max(np.abs(as_f64(host(y)) - y_ref) / (np.abs(y_ref) + 1e-3)) < 2 ** -7


def test_layer_with_1024_experts():
    """The largest expert count the library takes (N=1024; scores on CUDA cores for N > 256)."""
    w = WORKLOADS["decode_t32"].with_(name="n1024", T=300, d=256, N=1024, M=8, kpg=1, I=128)
    inp = synth.layer_inputs(w, seed=31)
    got = run_layer(w, upload_layer(inp))
    check_layer(w, inp, got)


@pytest.mark.slow
def test_layer_with_half_a_million_rows():
    """T=32768 tokens x K=16: 524288 (token, expert) rows, ~2000 CTA-pair tiles per GEMM;
    every token's routing checked, output rows of tokens reaching every tile of every expert."""
    w = WORKLOADS["prefill_t8192"].with_(name="rows512k", T=32768, d=256, I=128)
    inp = synth.layer_inputs(w, seed=32)
    got = run_layer(w, upload_layer(inp))
    check_layer_every_expert(w, inp, got)


@pytest.mark.parametrize("d,I", [(256, 192), (384, 136), (256, 64), (256, 384)])
def test_expert_ffn_per_expert_tile_shapes(d, I):
    """Experts whose row counts sit on both sides of every per-expert switch of the grouped GEMM
    (the batch holds > 104 rows per expert on average, so the tile shape is chosen per expert on
    the device): weights-as-M tiles of 32 tokens for experts of at most 64 rows (1, 31, 32, 33,
    63, 64), CTA-pair tiles above (65, 127, 128, 129, 255, 256, 257, 511, 512, 1000), with a ragged
    intermediate size and an empty expert; every row against the oracle.  The gate/up pair tiles
    hold two regions of 128 features: a partly filled second region (I = 192, 136), a half-filled
    first region and no second one (I = 64), and a last feature block of one region (I = 384)."""
    counts = np.array([1, 31, 32, 33, 63, 64, 0, 65, 127, 128, 129, 255, 256, 257, 511, 512, 1000, 0, 7, 5],
                      dtype=np.int64)
    N, M, kpg = 20, 4, 1
    P = int(counts.sum())
    T = P // (M * kpg)
    assert T * M * kpg == P and P / N > 104
    w = WORKLOADS["decode_t32"].with_(T=T, d=d, N=N, M=M, kpg=kpg, I=I)
    inp = synth.layer_inputs(w, seed=d + I)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    experts = np.repeat(np.arange(N, dtype=np.int32), counts)
    tokens = np.random.default_rng(d).integers(0, T, size=P).astype(np.int32)
    c = config(w)
    ws = moge.alloc_workspace(c)
    d_inp = upload_layer(inp)
    y_perm = torch.empty((P, w.d), dtype=torch.bfloat16, device=DEV)
    moge.moge_expert_ffn(c, dev(inp["x"][tokens]), dev(offsets), d_inp["w_gate"], d_inp["w_up"], d_inp["w_down"],
                         y_perm, ws)
    torch.cuda.synchronize()
    assert moge.moge_query_device_status(ws) == 0
    got = host(y_perm)
    rows_ref = oracle.expert_ffn_pairs(tokens, experts, inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    for e in range(N):  # per expert, so that a failing tile shape is named
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            err = max_rel_err(got[a:b], rows_ref[a:b])
            assert err <= TOL["bf16"], f"expert {e} ({counts[e]} rows): max rel err {err:.3e}"


def test_grouped_gemm_tile_counters_return_to_zero():
    """The CTA-pair GEMM launches take their tiles from two counters in the workspace's status page
    (bytes 512 and 768: next tile, finished CTAs); each launch returns them to zero before it ends,
    so back-to-back layers and CUDA-graph replays start from zero.  Checked after three layers of
    the per-expert plan on one workspace."""
    w = WORKLOADS["decode_t32"].with_(T=1500, d=256, I=192)
    d_inp = upload_layer(synth.layer_inputs(w, seed=77))
    ws = moge.alloc_workspace(config(w))
    for _ in range(3):
        run_layer(w, d_inp, ws=ws)
        page = host(ws[:1024].view(torch.int32))
        assert np.all(page[128:132] == 0) and np.all(page[192:196] == 0), page[128:200]
