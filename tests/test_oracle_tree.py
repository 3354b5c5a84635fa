"""Pins of the oracle's tree buffers (CPU).

* The page's printed 64-node example ("大模型推理 memory bandwidth bound (5) -
  Medusa", 二.2 generate_medusa_buffers()) must come out bit-exactly.
* The dense head1 top-2 x head2 top-3 tree (same page, 一.2 Tree attention)
  must give exactly the Cartesian product of paths.
* The synthetic 64-node tree is checked against a brute-force ranking that
  multiplies the scores out in floating point.
"""
import itertools
import json
import math
import os

import numpy as np

import synth
from oracle.tree import sort_choices, tree_buffers


def _page():
    with open(os.path.join(os.path.dirname(__file__), "golden", "page4_tree.json")) as f:
        return json.load(f)


def test_page_example_bit_exact():
    g = _page()
    choices = [tuple(c) for c in g["medusa_choices"]]
    assert len(choices) == 63
    assert [list(c) for c in sort_choices(choices)] == g["sorted_medusa_choices"]
    t = tree_buffers(choices, g["topk"])
    assert t["n_nodes"] == 64 and t["depth"] == 4
    assert t["tree_indices"].tolist() == g["tree_indices"]
    assert t["position_ids"].tolist() == g["medusa_position_ids"]
    assert t["retrieve"].tolist() == g["retrieve_indices"]
    for row, first, last in g["attn_mask_rows_shown"]["rows"]:
        assert t["attn_mask"][row, :3].tolist() == first
        assert t["attn_mask"][row, -3:].tolist() == last
    assert t["attn_mask"][:, 0].all()                     # the root column is all ones


def test_mask_is_ancestor_closure_of_parent():
    t = tree_buffers([tuple(c) for c in _page()["medusa_choices"]], 10)
    n = t["n_nodes"]
    for i in range(n):
        anc, j = {i}, i
        while t["parent"][j] >= 0:
            j = int(t["parent"][j])
            anc.add(j)
        assert set(np.flatnonzero(t["attn_mask"][i]).tolist()) == anc
        assert len(anc) == t["position_ids"][i] + 1


def test_every_node_on_some_path_and_paths_are_leaves():
    t = tree_buffers([tuple(c) for c in _page()["medusa_choices"]], 10)
    r = t["retrieve"]
    assert sorted(set(r[r >= 0].tolist())) == list(range(t["n_nodes"]))
    leaves = r[np.arange(len(r)), (r >= 0).sum(1) - 1]
    assert list(leaves) == sorted(leaves, reverse=True)
    assert set(leaves.tolist()).isdisjoint(set(t["parent"].tolist()))


def test_dense_tree_is_cartesian_product():
    t = tree_buffers(synth.dense_tree_choices([2, 3]), 10)
    assert t["n_nodes"] == 9 and len(t["retrieve"]) == 6
    assert t["tree_indices"].tolist() == [0, 1, 2, 11, 12, 13, 11, 12, 13]
    # symbolic tokens: root R, head-1 rank r -> 100+r, head-2 rank r -> 200+r
    cand = np.array([7] + [100 + r for r in range(10)] + [200 + r for r in range(10)])
    tree_tokens = cand[t["tree_indices"]]
    paths = {tuple(tree_tokens[p] for p in row if p >= 0) for row in t["retrieve"]}
    assert paths == {(7, 100 + a, 200 + b) for a, b in itertools.product(range(2), range(3))}


def test_synthetic_tree_brute_force():
    ch = synth.synthetic_tree_choices(64, 4, 10)
    assert len(ch) == 63
    t = tree_buffers(ch, 10)
    assert np.bincount(t["position_ids"]).tolist() == [1, 7, 21, 30, 5]
    assert len(t["retrieve"]) == 41
    # brute force: product of per-level factors, ranked with lexicographic ties
    allp = [c for D in range(1, 5) for c in itertools.product(range(10), repeat=D)]
    score = {c: math.prod(0.7 ** (d + 1) * 0.5 ** r for d, r in enumerate(c)) for c in allp}
    chosen = set(ch)
    worst_in = min(score[c] for c in chosen)
    best_out = max(score[c] for c in allp if c not in chosen)
    assert worst_in >= best_out * (1 - 1e-12)
    tied = [c for c in allp if abs(score[c] - worst_in) <= 1e-12 * worst_in]
    kept = sorted(c for c in tied if c in chosen)
    assert kept == sorted(tied)[: len(kept)]               # ties resolved lexicographically


def test_tree_rejects_bad_input():
    import pytest
    with pytest.raises(ValueError):
        tree_buffers([(0, 0)], 10)                        # not prefix-closed
    with pytest.raises(ValueError):
        tree_buffers([(0,), (0,)], 10)                    # duplicate
    with pytest.raises(ValueError):
        tree_buffers([(10,)], 10)                         # rank >= topk
