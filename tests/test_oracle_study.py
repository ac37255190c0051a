"""CPU pins of the imbalance Monte-Carlo study's inputs and of its expected outcome.

The study's scores are an Irwin-Hall approximation of N(0, 1): twelve 16-bit uniforms
(u + 1/2)/2^16 from three splitmix64 words per element, minus 6.  Pinned here against
that definition written out in numpy (uint64 arithmetic), against the moments and
support of the Irwin-Hall distribution, and the study's claim (Pangu Pro MoE explainer,
section 1: conventional top-K routing is almost always imbalanced, MoGE never) against
the oracle's routing of a few batches.
"""
import numpy as np

import oracle
import synth

M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def mix64_np(z):
    """splitmix64 (Steele, Lea and Flood, 2014) on uint64 arrays, wrap-around arithmetic."""
    with np.errstate(over="ignore"):
        z = z + np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def test_study_scores_follow_their_definition():
    seed, T, N = 11, 3, 5
    key = mix64_np(np.array([seed ^ synth.TID_STUDY], dtype=np.uint64))[0]
    got = synth.study_scores(seed, 2, 2, T, N)          # batches 2 and 3
    i = np.arange(2 * T * N, 4 * T * N, dtype=np.uint64)
    S = np.zeros(i.shape, dtype=np.int64)
    for j in range(3):
        with np.errstate(over="ignore"):
            w = mix64_np(key + np.uint64(3) * i + np.uint64(j))
        for k in range(4):
            S += ((w >> np.uint64(16 * k)) & np.uint64(0xFFFF)).astype(np.int64)
    want = ((2 * S + 12) / 2.0 ** 17 - 6.0).reshape(2, T, N)
    np.testing.assert_array_equal(got.astype(np.float64), want)


def test_study_scores_moments_and_support():
    z = synth.study_scores(3, 0, 4, 4096, 64).astype(np.float64).ravel()
    n = z.size
    assert abs(z.mean()) < 5 / np.sqrt(n)                  # mean 0
    assert abs(z.var() - 1.0) < 0.01                        # variance 12 * 1/12 = 1
    kurt = np.mean(z ** 4) / z.var() ** 2
    assert abs(kurt - (3 - 6 / 60)) < 0.03                  # Irwin-Hall(12): excess kurtosis -1/10
    assert z.min() > -6 and z.max() < 6
    assert np.all(np.mod((z + 6) * 2 ** 17, 1) == 0)        # exact grid of 2^-17


def test_study_batches_are_independent_streams():
    a = synth.study_scores(5, 0, 3, 100, 16)
    b = synth.study_scores(5, 1, 1, 100, 16)
    np.testing.assert_array_equal(a[1], b[0])
    assert not np.array_equal(a[0], a[1])


def test_conventional_routing_is_imbalanced_and_moge_is_not():
    """Section 1's Monte-Carlo claim on a few batches of the routing workload's shape."""
    T, N, M, kpg, B = 2048, 64, 8, 2, 6
    bias = synth.router_bias(synth.DEFAULT_SEED, N)
    z = synth.study_scores(synth.DEFAULT_SEED, 0, B, T, N)
    for b in range(B):
        l = (z[b] + bias[None, :]).astype(np.float32)
        g = oracle.route(l, M, kpg, mode="grouped")
        c = oracle.route(l, M, kpg, mode="global")
        assert g["score"] == 0.0 and np.all(g["group_load"] == T * kpg)
        assert c["score"] > 0.0 and c["group_load"].sum() == T * M * kpg
