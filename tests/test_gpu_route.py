"""GPU parity of moge_route / moge_permute / moge_imbalance_score against the oracle.

Given the same fp32 scores, routing indices, counts, offsets, pair rows and
group loads are bit-exact; gates agree within 1e-6 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, dev, host

pytestmark = pytest.mark.gpu

GATE_TOL = 1e-6


def gpu_route(logits: np.ndarray, M: int, kpg: int, mode: int):
    T, N = logits.shape
    K = M * kpg
    c = moge.make_config(T, 0, N, M, kpg, 0, "f32")
    ws = moge.alloc_workspace(c)
    d_l = dev(logits)
    idx = torch.full((T, K), -7, dtype=torch.int32, device=DEV)
    gate = torch.empty((T, K), dtype=torch.float32, device=DEV)
    counts = torch.empty(N, dtype=torch.int32, device=DEV)
    offsets = torch.empty(N + 1, dtype=torch.int32, device=DEV)
    pair_row = torch.empty((T, K), dtype=torch.int32, device=DEV)
    row_token = torch.empty(T * K, dtype=torch.int32, device=DEV)
    loads = torch.empty(M, dtype=torch.int32, device=DEV)
    score = torch.empty(4, dtype=torch.float32, device=DEV)
    moge.moge_route(c, mode, None, None, None, d_l, idx, gate, ws)
    moge.moge_permute(c, idx, None, counts, offsets, pair_row, row_token, None, ws)
    moge.moge_imbalance_score(c, counts, loads, score)
    torch.cuda.synchronize()
    return {"idx": host(idx), "gate": host(gate), "counts": host(counts), "offsets": host(offsets),
            "pair_row": host(pair_row), "row_token": host(row_token), "group_load": host(loads),
            "score": host(score)[0]}


def check(got, ref, T):
    np.testing.assert_array_equal(got["idx"], ref["idx"])
    assert np.max(np.abs(got["gate"].astype(np.float64) - ref["gate64"])) <= GATE_TOL
    for k in ("counts", "offsets", "pair_row", "row_token", "group_load"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    loads = ref["group_load"].astype(np.int64)
    expect = np.float32(loads.max() - loads.min()) / np.float32(T) if T else np.float32(0)
    assert got["score"] == expect


@pytest.mark.parametrize("kpg", [2, 1])
@pytest.mark.parametrize("mode", [moge.MOGE_ROUTE_GROUPED, moge.MOGE_ROUTE_GLOBAL_TOPK])
def test_routing_16k_bit_exact(kpg, mode):
    """The routing-only workload: T=16384, N=64 in 8 groups, skewed fp32 scores."""
    T, N, M = 16384, 64, 8
    l = synth.route_logits(synth.DEFAULT_SEED, T, N)
    ref = oracle.route(l, M, kpg, mode="grouped" if mode == moge.MOGE_ROUTE_GROUPED else "global")
    got = gpu_route(l, M, kpg, mode)
    check(got, ref, T)
    if mode == moge.MOGE_ROUTE_GROUPED:
        assert got["score"] == 0.0 and np.all(got["group_load"] == T * kpg)
    else:
        assert got["score"] > 0.5


@pytest.mark.parametrize("T,N,M,kpg", [
    (1, 64, 8, 2), (255, 64, 8, 2), (256, 64, 8, 2), (257, 16, 4, 1), (1000, 12, 3, 2),
    (777, 256, 8, 1), (300, 256, 8, 32), (513, 40, 1, 7), (100, 8, 8, 1), (64, 1024, 4, 3)])
def test_routing_shapes_and_ties(T, N, M, kpg):
    rng = np.random.default_rng(T * 7 + N)
    l = rng.integers(-3, 4, size=(T, N)).astype(np.float32)   # heavy ties
    l[::2] += rng.standard_normal((l[::2].shape)).astype(np.float32) * 0.5
    for mode, name in ((moge.MOGE_ROUTE_GROUPED, "grouped"), (moge.MOGE_ROUTE_GLOBAL_TOPK, "global")):
        check(gpu_route(l, M, kpg, mode), oracle.route(l, M, kpg, mode=name), T)


def test_one_expert_takes_every_token():
    T, N, M = 600, 16, 4
    l = np.zeros((T, N), dtype=np.float32)
    l[:, 5] = 10.0
    ref = oracle.route(l, M, 1)
    got = gpu_route(l, M, 1, moge.MOGE_ROUTE_GROUPED)
    check(got, ref, T)
    assert got["counts"][5] == T


@pytest.mark.parametrize("T,d,dtype", [
    (700, 256, "bf16"),    # one 32-vector chunk per row, destinations split in 4 groups per token
    (5, 4104, "bf16"),     # rows of 513 vectors: three chunks, the last ragged; 16 destination groups
    (3000, 4104, "bf16"),  # one destination group
    (300, 1028, "f32"),    # fp32 rows, ragged chunk
])
@pytest.mark.parametrize("with_pair_row", [True, False])
def test_permute_gathers_rows_exactly(T, d, dtype, with_pair_row):
    """x_perm[r] = x[row_token[r]] bit for bit: the token-major copy when pair_row is an output, the
    row-major gather through row_token when it is not."""
    w = synth.WORKLOADS["decode_t32"].with_(T=T, d=d)
    x = synth.normal(3, synth.TID_X, (w.T, w.d), 1.0, dtype)
    l = synth.route_logits(4, w.T, w.N)
    ref = oracle.route(l, w.M, w.kpg)
    c = moge.make_config(w.T, w.d, w.N, w.M, w.kpg, w.I, dtype)
    ws = moge.alloc_workspace(c)
    idx = dev(ref["idx"])
    counts = torch.empty(w.N, dtype=torch.int32, device=DEV)
    offsets = torch.empty(w.N + 1, dtype=torch.int32, device=DEV)
    pair_row = torch.empty((w.T, w.K), dtype=torch.int32, device=DEV) if with_pair_row else None
    row_token = torch.empty(w.P, dtype=torch.int32, device=DEV)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x_perm = torch.full((w.P, w.d), 7.0, dtype=tdt, device=DEV)
    moge.moge_permute(c, idx, dev(x), counts, offsets, pair_row, row_token, x_perm, ws)
    torch.cuda.synchronize()
    perm = oracle.permute(ref["idx"], w.N)
    if with_pair_row:
        np.testing.assert_array_equal(host(pair_row), perm["pair_row"])
    np.testing.assert_array_equal(host(row_token), perm["row_token"])
    np.testing.assert_array_equal(host(x_perm), x[perm["row_token"]])


@pytest.mark.parametrize("with_pair_row", [True, False])
def test_permute_skips_out_of_range_ids_and_writes_nothing_else(with_pair_row):
    """Ids outside [0, N) own no row: pair_row = -1 there, the other pairs keep the order of the
    definition, and the row copy writes rows [0, valid pairs) only.  x_perm is a view one row into
    a larger buffer, so a store to row -1 or past the last row would show in the guard rows."""
    T, d, N, M, kpg = 300, 264, 16, 4, 1
    w = synth.WORKLOADS["decode_t32"].with_(T=T, d=d, N=N, M=M, kpg=kpg)
    x = synth.normal(5, synth.TID_X, (T, d), 1.0, "bf16")
    idx = oracle.route(synth.route_logits(6, T, N), M, kpg)["idx"].copy()
    bad = np.random.default_rng(1).random(idx.shape) < 0.2
    idx[bad] = np.resize(np.array([-1, N, 1000, -7], dtype=np.int32), int(bad.sum()))
    # the definition on the valid pairs, in (token, slot) order
    valid = (idx >= 0) & (idx < N)
    counts = np.bincount(idx[valid], minlength=N).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    pair_row_ref = np.full(idx.shape, -1, dtype=np.int32)
    fill = offsets[:-1].copy()
    for t in range(T):
        for k in range(w.K):
            e = idx[t, k]
            if 0 <= e < N:
                pair_row_ref[t, k] = fill[e]
                fill[e] += 1
    pv = int(offsets[N])
    row_token_ref = np.empty(pv, dtype=np.int32)
    row_token_ref[pair_row_ref[valid]] = np.nonzero(valid)[0]
    c = moge.make_config(T, d, N, M, kpg, 64, "bf16")
    ws = moge.alloc_workspace(c)
    cnt = torch.empty(N, dtype=torch.int32, device=DEV)
    off = torch.empty(N + 1, dtype=torch.int32, device=DEV)
    pair_row = torch.empty((T, w.K), dtype=torch.int32, device=DEV) if with_pair_row else None
    row_token = torch.full((T * w.K,), -9, dtype=torch.int32, device=DEV)
    buf = torch.full((T * w.K + 2, d), 3.0, dtype=torch.bfloat16, device=DEV)
    moge.moge_permute(c, dev(idx), dev(x), cnt, off, pair_row, row_token, buf[1:], ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(cnt), counts)
    np.testing.assert_array_equal(host(off), offsets)
    if with_pair_row:
        np.testing.assert_array_equal(host(pair_row), pair_row_ref)
    np.testing.assert_array_equal(host(row_token)[:pv], row_token_ref)
    got = host(buf)
    np.testing.assert_array_equal(got[1:pv + 1], x[row_token_ref])
    guard = host(torch.full((1, d), 3.0, dtype=torch.bfloat16))
    assert np.all(got[0] == guard[0]) and np.all(got[pv + 1:] == guard[0])


def test_empty_batch():
    c = moge.make_config(0, 0, 16, 4, 1, 0, "f32")
    ws = moge.alloc_workspace(c)
    counts = torch.full((16,), 9, dtype=torch.int32, device=DEV)
    offsets = torch.full((17,), 9, dtype=torch.int32, device=DEV)
    idx = torch.empty((1, 4), dtype=torch.int32, device=DEV)
    moge.moge_permute(c, idx, None, counts, offsets, None, None, None, ws)
    score = torch.full((4,), 5.0, dtype=torch.float32, device=DEV)
    moge.moge_imbalance_score(c, counts, None, score)
    torch.cuda.synchronize()
    assert np.all(host(counts) == 0) and np.all(host(offsets) == 0) and host(score)[0] == 0.0
