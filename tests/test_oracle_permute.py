"""Pins of the oracle's permutation and imbalance score.

Permutation: a stable counting sort of (token, slot) pairs by expert (reading:
ascending token inside an expert).  Imbalance: busiest minus idlest group load
over a batch ('Pangu Pro MoE explainer', section 1), divided by T.
"""
import numpy as np
import pytest

import oracle
import synth


def definition_pair_row(idx, N):
    """pair_row straight from its definition, by counting (O(P*T))."""
    T, K = idx.shape
    counts = np.array([(idx == e).sum() for e in range(N)])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    out = np.empty_like(idx)
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            out[t, k] = offsets[e] + sum(e in idx[tp] for tp in range(t))
    return counts, offsets, out


@pytest.mark.parametrize("mode", ["grouped", "global"])
def test_pair_row_definition_small(mode):
    l = synth.route_logits(5, 40, 16)
    idx = oracle.select_grouped(l, 4, 2) if mode == "grouped" else oracle.select_global(l, 8)
    perm = oracle.permute(idx, 16)
    c, o, pr = definition_pair_row(idx, 16)
    np.testing.assert_array_equal(perm["counts"], c)
    np.testing.assert_array_equal(perm["offsets"], o)
    np.testing.assert_array_equal(perm["pair_row"], pr)


def test_permutation_invariants_large():
    T, N, M, kpg = 4096, 64, 8, 2
    l = synth.route_logits(9, T, N)
    idx = oracle.select_grouped(l, M, kpg)
    perm = oracle.permute(idx, N)
    P = T * M * kpg
    counts, offsets, pr, rt = perm["counts"], perm["offsets"], perm["pair_row"], perm["row_token"]
    assert counts.sum() == P and offsets[-1] == P and offsets[0] == 0
    assert np.all(np.diff(offsets) == counts)
    # bijection onto [0, P)
    assert np.array_equal(np.sort(pr.ravel()), np.arange(P))
    # row_token inverts pair_row, and each row lies in its expert's segment
    tok = np.repeat(np.arange(T), M * kpg).reshape(T, -1)
    assert np.array_equal(rt[pr], tok)
    assert np.all(pr >= offsets[idx]) and np.all(pr < offsets[idx + 1])
    # ascending tokens inside every expert segment
    for e in range(N):
        seg = rt[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_experts_with_zero_and_all_tokens():
    T = 33
    idx = np.zeros((T, 2), dtype=np.int32)
    idx[:, 0] = 3          # every token to expert 3
    idx[:, 1] = 5          # and to expert 5
    perm = oracle.permute(idx, 8)
    assert list(perm["counts"]) == [0, 0, 0, T, 0, T, 0, 0]
    assert list(perm["pair_row"][:, 0]) == list(range(T))
    assert list(perm["pair_row"][:, 1]) == list(range(T, 2 * T))


def test_imbalance_hand_values():
    loads, s = oracle.imbalance(np.array([3, 0, 1, 4], dtype=np.int32), T=2, M=2)
    assert list(loads) == [3, 5] and s == 1.0
    loads, s = oracle.imbalance(np.array([2, 2, 2, 2, 2, 2], dtype=np.int32), T=4, M=3)
    assert list(loads) == [4, 4, 4] and s == 0.0
    loads, s = oracle.imbalance(np.array([7, 0, 0], dtype=np.int32), T=7, M=3)
    assert list(loads) == [7, 0, 0] and s == 1.0
