"""Pins of the oracle's posterior evaluation and KV compaction (CPU).

Typical acceptance ("大模型推理 memory bandwidth bound (5) - Medusa", 一.3
Typical acceptance, 二.6 evaluate_posterior()): hand-computed distributions.
Uniform over V tokens: p = 1/V, H = -ln(1/V + 1e-5), exp(-H) = 1/V + 1e-5, so
tau = min(eps, delta (1/V + 1e-5)).
Greedy acceptance: hand-built trees with known accept lengths.
KV compaction (二.7 update_inference_inputs()): hand-written integer cases,
including a path whose source and destination rows overlap.
"""
import math

import numpy as np

import synth
from oracle.kv import kv_compact
from oracle.posterior import GREEDY, TYPICAL, evaluate_posterior, node_stats
from oracle.tree import tree_buffers


def test_typical_uniform_closed_form():
    for V in (4, 32000):
        st = node_stats(np.zeros((1, V)), TYPICAL, 1.0, 0.09, 0.3)
        assert math.isclose(st["entropy"][0], -math.log(1 / V + 1e-5), rel_tol=1e-12)
        assert math.isclose(st["tau"][0], min(0.09, 0.3 * (1 / V + 1e-5)), rel_tol=1e-12)
    st = node_stats(np.zeros((1, 4)), TYPICAL)
    assert abs(st["tau"][0] - 0.075003) < 1e-12 and abs(st["entropy"][0] - 1.386254) < 1e-6
    st = node_stats(np.zeros((1, 32000)), TYPICAL)
    assert abs(st["entropy"][0] - 10.095859) < 1e-6 and abs(st["tau"][0] - 1.2375e-5) < 1e-15
    assert st["p"][0, 0] > st["tau"][0]                         # 3.125e-5 > 1.2375e-5: accepted


def test_typical_hand_values():
    # logits [2,1,0,-1]: p = [.643914, .236883, .087144, .032059], H = .947497 -> tau = eps = .09
    st = node_stats(np.array([[2.0, 1, 0, -1]]), TYPICAL, 1.0)
    assert np.allclose(st["p"][0], [0.643914, 0.236883, 0.087144, 0.032059], atol=1e-6)
    assert abs(st["entropy"][0] - 0.947497) < 1e-6 and st["tau"][0] == 0.09
    assert (st["p"][0] > st["tau"][0]).tolist() == [True, True, False, False]
    # temperature 0.7 divides the logits first: p = [.762865, .182821, .043813, .0105]
    st = node_stats(np.array([[2.0, 1, 0, -1]]), TYPICAL, 0.7)
    assert np.allclose(st["p"][0], [0.762865, 0.182821, 0.043813, 0.0105], atol=1e-6)
    assert (st["p"][0] > st["tau"][0]).tolist() == [True, True, False, False]
    # a peaked row: H = .001461, only rank 0 passes
    st = node_stats(np.array([[10.0, 0, 0, 0]]), TYPICAL, 1.0)
    assert abs(st["entropy"][0] - 0.001461) < 1e-6
    assert (st["p"][0] > st["tau"][0]).tolist() == [True, False, False, False]


def _dense_tree():
    return tree_buffers(synth.dense_tree_choices([2, 3]), 10)   # 9 nodes, 6 paths


def test_greedy_accept_lengths_by_hand():
    t = _dense_tree()          # node order: 0 root, 1 (0,), 2 (1,), 3..5 (0,r), 6..8 (1,r)
    V = 16
    tokens = np.array([0, 5, 6, 7, 8, 9, 10, 11, 12])
    z = np.zeros((9, V))
    z[0, 6] = 1.0              # root predicts token 6 = node 2 (rank 1 of head 1)
    z[2, 11] = 1.0             # node 2 predicts token 11 = node 7 ((1,1))
    r = evaluate_posterior(z, tokens, t["retrieve"], GREEDY)
    assert r["acc"] == 2 and r["nodes"].tolist() == [0, 2, 7] and r["next_node"] == 7
    assert t["retrieve"][r["best"]].tolist() == [0, 2, 7]
    assert sorted(r["accept_len"].tolist()) == [0, 0, 0, 1, 1, 2]
    z[2, 11] = 0.0             # only depth 1 accepted: first row among the three (1, .) paths
    r = evaluate_posterior(z, tokens, t["retrieve"], GREEDY)
    assert r["acc"] == 1 and r["nodes"].tolist() == [0, 2]
    assert r["best"] == min(i for i, row in enumerate(t["retrieve"]) if row[1] == 2)
    r = evaluate_posterior(np.zeros((9, V)) + np.eye(V)[15], tokens, t["retrieve"], GREEDY)
    assert r["acc"] == 0 and r["best"] == 0 and r["nodes"].tolist() == [0]


def test_padding_is_never_accepted():
    # a path shorter than the tree depth: retrieve pads with -1; the page's code would map
    # the pad to token 0 and compare it with the last node's argmax
    t = tree_buffers([(0,), (1,), (0, 0)], 10)                    # rows [0,1,3], [0,2,-1]
    tokens = np.array([9, 1, 2, 3])
    z = np.zeros((4, 8))
    z[0, 2] = 5.0              # root -> node 2 (token 2), a leaf at depth 1
    z[3, 0] = 5.0              # the last node predicts token 0 (the pad token)
    r = evaluate_posterior(z, tokens, t["retrieve"], GREEDY)
    assert r["acc"] == 1 and r["nodes"].tolist() == [0, 2]


def test_typical_likelihood_tie_break():
    t = _dense_tree()
    V = 8
    tokens = np.array([0, 1, 2, 3, 4, 5, 3, 4, 5])
    z = np.full((9, V), -20.0)
    z[0, [1, 2]] = [0.0, 0.0]                     # both depth-1 nodes accepted, equal p
    z[1, [3, 4]] = [0.0, 0.0]                     # under node 1: two children at p = .5 each
    z[2, [3, 4, 5]] = [1.0, 0.0, 0.0]             # under node 2: child token 3 at p = .576 (wins)
    r = evaluate_posterior(z, tokens, t["retrieve"], TYPICAL, 1.0, 0.09, 0.3)
    assert r["acc"] == 2
    assert r["nodes"].tolist() == [0, 2, 6]
    # the same two-way tie with equal likelihood goes to the first row
    z[2, [3, 4, 5]] = [0.0, 0.0, -20.0]
    r = evaluate_posterior(z, tokens, t["retrieve"], TYPICAL, 1.0, 0.09, 0.3)
    assert r["acc"] == 2 and r["best"] == min(np.flatnonzero(r["accept_len"] == 2))


def test_kv_compact_overlapping_rows():
    # path [0, 3, 26, 56] at prefix 10: row 10+3 is both a source (j=1) and a destination (j=3)
    S = 10 + 64
    cache = np.arange(2 * S * 2, dtype=np.float64).reshape(2, S, 2)  # [heads, S, D]
    out, L = kv_compact(cache, 10, [0, 3, 26, 56])
    assert L == 14
    for j, node in enumerate([0, 3, 26, 56]):
        assert (out[:, 10 + j] == cache[:, 10 + node]).all()
    assert (out[:, :10] == cache[:, :10]).all() and (out[:, 14:] == cache[:, 14:]).all()
    out, L = kv_compact(cache, 10, [0])                       # nothing accepted: length + 1
    assert L == 11 and (out == cache).all()


def test_margins_by_hand():
    # The margin of each decision ("大模型推理 memory bandwidth bound (5) - Medusa", 二.6 evaluate_posterior()):
    # greedy top-1 - top-2 when the candidate is the argmax (accepted), top-1 - its logit when it is not; typical
    # |ln p(candidate) - ln tau|. Every decision up to a row's first rejection is listed, and none after it.
    t = tree_buffers([(0,), (1,)], 10)                   # retrieve rows [0, 2] and [0, 1]
    # an exact tie at the top: tokens 3 and 5 share the largest logit; the argmax is the lower id (3)
    z = np.zeros((3, 8))
    z[0, [3, 5]] = 1.0
    r = evaluate_posterior(z, np.array([0, 3, 5]), t["retrieve"], GREEDY)
    m = {(p, j): v for (p, j, v) in r["margins"]}
    assert m == {(0, 0): 0.0, (1, 0): 0.0}
    assert r["accept_len"].tolist() == [0, 1] and r["nodes"].tolist() == [0, 1]
    # the row [2, 1, 0, -1]: candidate token 0 accepted with margin 2 - 1; candidate token 2 rejected, 2 - 0
    z = np.full((3, 4), -5.0)
    z[0] = [2.0, 1.0, 0.0, -1.0]
    r = evaluate_posterior(z, np.array([9, 0, 2]) % 4, t["retrieve"], GREEDY)
    m = {(p, j): v for (p, j, v) in r["margins"]}
    assert m == {(0, 0): 2.0, (1, 0): 1.0}
    # typical at T = 1 on the same row: p = [.643914, .236883, .087144, .032059], tau = eps = .09;
    # token 2 is rejected by ln(.09 / .087144) = .032244, token 1 accepted by ln(.236883 / .09) = .967756
    r = evaluate_posterior(z, np.array([0, 1, 2]), t["retrieve"], TYPICAL, 1.0, 0.09, 0.3)
    m = {(p, j): v for (p, j, v) in r["margins"]}
    assert abs(m[(0, 0)] - 0.032244) < 1e-6 and abs(m[(1, 0)] - 0.967756) < 1e-6
    assert r["accept_len"].tolist() == [0, 1]
    # a rejection ends the row: with the depth-1 candidate of row [0, 1, 3] rejected, its depth-2 decision is
    # never made (no margin listed for it); the other row is accepted at depth 1 and ends there
    t = tree_buffers([(0,), (1,), (0, 0)], 10)          # rows [0, 1, 3] and [0, 2, -1]
    z = np.zeros((4, 8))
    z[0, 6] = 3.0                                       # root predicts token 6 = node 2
    z[1, 7] = 3.0
    r = evaluate_posterior(z, np.array([0, 5, 6, 7]), t["retrieve"], GREEDY)
    assert sorted((p, j) for (p, j, _) in r["margins"]) == [(0, 0), (1, 0)]
    m = {(p, j): v for (p, j, v) in r["margins"]}
    assert m[(0, 0)] == 3.0 and m[(1, 0)] == 3.0        # rejected: 3 - z[5] = 3; accepted: 3 - 0 = 3
