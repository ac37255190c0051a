"""Pins of the oracle's routing: softmax, group top-K', global top-K, gates.

Each check is independent of the oracle's own code: a hand-worked fixture,
brute-force enumeration, closed forms, or a library routine (numpy sort).
Routing rule: 'Pangu Pro MoE explainer', section 1 (global softmax over all
N experts, then top-K' = K/M inside each of M equal groups); section 6 (no
co-activation inside a group when K'=1).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_tiny.json")


def _ranks_before(l, a, b):
    return l[a] > l[b] or (l[a] == l[b] and a < b)


def brute_force_group_topk(l, lo, hi, k):
    """The unique k-subset of [lo,hi) whose members all rank before all
    non-members, found by enumerating every subset; returned in rank order."""
    members = range(lo, hi)
    valid = []
    for S in itertools.combinations(members, k):
        rest = [e for e in members if e not in S]
        if all(_ranks_before(l, a, b) for a in S for b in rest):
            valid.append(S)
    assert len(valid) == 1, "the rank rule must define exactly one subset"
    S = list(valid[0])
    # rank order: the number of members ranking before each one
    return sorted(S, key=lambda a: sum(_ranks_before(l, b, a) for b in S))


def brute_force_route(logits, M, kpg):
    T, N = logits.shape
    G = N // M
    out = np.empty((T, M * kpg), dtype=np.int32)
    for t in range(T):
        for g in range(M):
            out[t, g * kpg:(g + 1) * kpg] = brute_force_group_topk(logits[t], g * G, (g + 1) * G, kpg)
    return out


def test_golden_tiny_grouped_and_global():
    gold = json.load(open(GOLDEN))
    l = np.array(gold["logits"], dtype=np.float32)
    for mode in ("grouped", "global"):
        r = oracle.route(l, gold["M"], gold["kpg"], mode=mode)
        exp = gold[mode]
        for key in ("idx", "counts", "offsets", "pair_row", "row_token", "group_load"):
            np.testing.assert_array_equal(r[key], np.array(exp[key]), err_msg=f"{mode}:{key}")
        assert r["score"] == exp["score"]
        # gates are the plain softmax probabilities (closed form, math.exp)
        for t in range(gold["T"]):
            z = sum(math.exp(v) for v in gold["logits"][t])
            for k, e in enumerate(exp["idx"][t]):
                assert abs(r["gate64"][t, k] - math.exp(gold["logits"][t][e]) / z) < 1e-15


@pytest.mark.parametrize("kpg", [1, 2, 3, 4])
def test_exhaustive_tie_patterns_g4(kpg):
    # every pattern of {0,1,2}^4 in group 0 and its reverse in group 1
    pats = np.array(list(itertools.product([0.0, 1.0, 2.0], repeat=4)), dtype=np.float32)
    l = np.concatenate([pats, pats[:, ::-1]], axis=1)
    got = oracle.select_grouped(l, M=2, kpg=kpg)
    np.testing.assert_array_equal(got, brute_force_route(l, 2, kpg))


@pytest.mark.parametrize("N,M,kpg", [(12, 3, 2), (16, 4, 1), (8, 1, 3), (10, 5, 2), (32, 4, 3)])
def test_random_ties_vs_brute_force(N, M, kpg):
    rng = np.random.default_rng(N * 100 + M * 10 + kpg)
    l = rng.integers(-2, 3, size=(150, N)).astype(np.float32)  # many ties
    l[::3] += rng.standard_normal((50, N)).astype(np.float32)   # and some without
    np.testing.assert_array_equal(oracle.select_grouped(l, M, kpg), brute_force_route(l, M, kpg))


def test_exactly_kpg_per_group_and_zero_imbalance():
    l = synth.route_logits(7, 2048, 64)
    for kpg in (1, 2):
        idx = oracle.select_grouped(l, 8, kpg)
        grp = idx // 8
        for g in range(8):
            assert np.all((grp[:, g * kpg:(g + 1) * kpg] == g)), "slot block g holds group g"
        assert np.all(np.sort(idx, axis=1)[:, 1:] != np.sort(idx, axis=1)[:, :-1]), "distinct"
        perm = oracle.permute(idx, 64)
        loads, score = oracle.imbalance(perm["counts"], 2048, 8)
        assert np.all(loads == 2048 * kpg) and score == 0.0


def test_kpg1_no_coactivation_inside_group():
    l = synth.route_logits(11, 1024, 64)
    idx = oracle.select_grouped(l, 8, 1)
    assert np.all(np.diff(idx // 8, axis=1) == 1)  # one expert from each group, in order


def test_single_group_equals_global_topk_and_numpy_sort():
    rng = np.random.default_rng(3)
    l = rng.integers(-3, 4, size=(300, 20)).astype(np.float32)
    a = oracle.select_grouped(l, M=1, kpg=6)
    b = oracle.select_global(l, K=6)
    np.testing.assert_array_equal(a, b)
    # library routine: stable lexicographic sort on (-score, index)
    ref = np.stack([np.lexsort((np.arange(20), -row))[:6] for row in l]).astype(np.int32)
    np.testing.assert_array_equal(b, ref)


def test_kpg_equals_group_size_selects_all_in_rank_order():
    rng = np.random.default_rng(5)
    l = rng.standard_normal((64, 16)).astype(np.float32)
    idx = oracle.select_grouped(l, M=4, kpg=4)
    for t in range(64):
        for g in range(4):
            blk = idx[t, 4 * g:4 * g + 4]
            assert sorted(blk) == list(range(4 * g, 4 * g + 4))
            assert all(l[t, blk[i]] >= l[t, blk[i + 1]] for i in range(3))


def test_selection_matches_probability_order():
    # the selection uses fp32 logits; the softmax is increasing, so the same
    # experts are the K' most probable ones of each group
    l = synth.route_logits(13, 512, 64)
    p = oracle.softmax(l)
    idx = oracle.select_grouped(l, 8, 2)
    for t in range(0, 512, 7):
        for g in range(8):
            pg = p[t, 8 * g:8 * g + 8]
            best2 = set(np.argsort(-pg, kind="stable")[:2] + 8 * g)
            assert best2 == set(idx[t, 2 * g:2 * g + 2])


def test_softmax_closed_forms():
    rng = np.random.default_rng(1)
    l = (rng.standard_normal((100, 64)) * 3).astype(np.float32)
    p = oracle.softmax(l)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-12
    assert np.all(p > 0)
    # N=2 is the logistic function of the difference
    l2 = np.array([[0.0, 1.5], [2.0, -1.0], [3.25, 3.25]], dtype=np.float32)
    p2 = oracle.softmax(l2)
    for t in range(3):
        expect = 1.0 / (1.0 + math.exp(float(l2[t, 1]) - float(l2[t, 0])))
        assert abs(p2[t, 0] - expect) < 1e-15
    # uniform logits give 1/N
    assert np.allclose(oracle.softmax(np.full((2, 7), 0.3, np.float32)), 1 / 7, rtol=0, atol=1e-15)
    # invariance to an exactly representable shift
    li = rng.integers(-8, 8, size=(50, 16)).astype(np.float32)
    assert np.max(np.abs(oracle.softmax(li) - oracle.softmax(li + np.float32(16.0)))) < 1e-14


def test_gates_are_unrenormalised_probabilities():
    l = synth.route_logits(17, 256, 64)
    r = oracle.route(l, 8, 2)
    p = r["p"]
    for t in range(0, 256, 5):
        for k in range(16):
            assert r["gate64"][t, k] == p[t, r["idx"][t, k]]
            assert r["gate"][t, k] == np.float32(p[t, r["idx"][t, k]])
    s = r["gate64"].sum(axis=1)
    assert np.all(s < 1.0) and np.all(s > 0.0)  # 16 of 64 experts: not renormalised


def test_global_topk_imbalance_positive_on_skewed_scores():
    # conventional top-K routing on the same scores is (almost always) unbalanced
    l = synth.route_logits(synth.DEFAULT_SEED, 16384, 64)
    for kpg in (1, 2):
        g = oracle.route(l, 8, kpg, mode="global")
        m = oracle.route(l, 8, kpg, mode="grouped")
        assert m["score"] == 0.0 and np.all(m["group_load"] == 16384 * kpg)
        assert g["score"] > 0.5
        assert g["group_load"].sum() == 16384 * 8 * kpg


# -- a planted mistake must trip the pins -------------------------------------------

def test_planted_tie_break_mistake_is_caught():
    gold = json.load(open(GOLDEN))
    l = np.array(gold["logits"], dtype=np.float32)
    good = oracle.select_grouped(l, 2, 2)
    # the same rule with ties to the HIGHER index, written as a mutant
    bad = np.stack([
        np.concatenate([sorted(range(g * 4, g * 4 + 4), key=lambda e: (-l[t, e], -e))[:2]
                        for g in range(2)]) for t in range(2)]).astype(np.int32)
    assert not np.array_equal(bad, np.array(gold["grouped"]["idx"]))
    np.testing.assert_array_equal(good, np.array(gold["grouped"]["idx"]))
