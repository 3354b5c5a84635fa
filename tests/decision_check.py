"""Per-decision comparison of a GPU posterior result with the oracle's (test helper, not a test module).

"大模型推理 memory bandwidth bound (5) - Medusa", 二.6 evaluate_posterior(): along every retrieve row the
candidate at position j + 1 is accepted or rejected against the distribution of the node at position j, and a
row stops at its first rejection. The bar: a GPU acceptance decision may differ from the oracle's only where
the oracle's margin for that same decision is below MARGIN (greedy: top-1 minus top-2 when accepted, top-1
minus the candidate's logit when rejected; typical: |ln p(candidate) - ln tau|). So each row is walked
decision by decision; at the first decision where the two sides differ, that decision's oracle margin must be
below MARGIN (the rest of that row legitimately diverges). When no decision differs, the results must be
equal, except that typical acceptance may pick another row between likelihood sums within MARGIN.

The GPU side's decisions come from the GPU's own per-node outputs: the posterior kernel's node argmax and
statistics, or (for a whole verify step) the GPU's logits rows. The acceptance rule is restated here in a few
lines for that purpose; nothing is taken from the oracle module.
"""
from __future__ import annotations

import numpy as np

MARGIN = 1e-3
GREEDY, TYPICAL = 0, 1


def decisions_from_logits(logits, tree_tokens, mode, temperature=0.7, eps=0.09, delta=0.3):
    """accepts(node, child) -> bool, computed in float64 from the GPU's fp32 logits rows [n, V]."""
    z = np.asarray(logits, dtype=np.float64)
    tok = np.asarray(tree_tokens, dtype=np.int64)
    if mode == GREEDY:
        am = np.argmax(z, axis=1)  # first largest, as the kernels break ties
        return lambda node, child: int(tok[child]) == int(am[node])
    y = z / temperature
    y = y - y.max(axis=1, keepdims=True)
    lse = np.log(np.exp(y).sum(axis=1))
    p = np.exp(y - lse[:, None])
    H = -np.sum(p * np.log(p + 1e-5), axis=1)
    ltau = np.log(np.minimum(eps, delta * np.exp(-H)))
    return lambda node, child: bool(y[node, tok[child]] - lse[node] > ltau[node])


def decisions_from_stats(logits, tree_tokens, mode, node_argmax, node_stats, temperature=0.7):
    """accepts(node, child) from the posterior kernel's own outputs: its node argmax (greedy), or its node
    statistics (max, log normaliser of z/T relative to the max, H, tau) with the candidate's logit (typical)."""
    tok = np.asarray(tree_tokens, dtype=np.int64)
    if mode == GREEDY:
        am = np.asarray(node_argmax)
        return lambda node, child: int(tok[child]) == int(am[node])
    z = np.asarray(logits, dtype=np.float64)
    st = np.asarray(node_stats, dtype=np.float64)

    def acc(node, child):
        lp = (z[node, tok[child]] - st[node, 0]) / temperature - st[node, 1]
        return bool(lp > np.log(st[node, 3]))

    return acc


def check(res, accepts, ref, retrieve, mode):
    """Asserts the bar above for one verification; returns the list of (row, position, oracle margin) where a
    row's first differing decision was found (empty when every decision matched)."""
    retrieve = np.asarray(retrieve)
    n_paths, width = retrieve.shape
    margins = {(p, j): m for (p, j, m) in ref["margins"]}
    oacc = np.asarray(ref["accept_len"])
    gacc = np.zeros(n_paths, dtype=np.int64)  # the GPU side's accept lengths
    diverged = []
    for p in range(n_paths):
        agreed = True
        for j in range(width - 1):
            node, child = int(retrieve[p, j]), int(retrieve[p, j + 1])
            if child < 0:
                break
            g = accepts(node, child)
            if agreed:
                o = j < oacc[p]
                if g != o:
                    m = margins[(p, j)]
                    assert m < MARGIN, f"row {p} position {j}: GPU {'accepts' if g else 'rejects'}, the oracle " \
                                       f"does not, and the oracle's margin there is {m:.3g} >= {MARGIN}"
                    diverged.append((p, j, m))
                    agreed = False
            if not g:
                break
            gacc[p] += 1
    # the GPU result follows from its own decisions: the longest accepted row, a prefix of a retrieve row
    acc = int(res["acc"])
    assert acc == int(gacc.max()), (acc, int(gacc.max()))
    nodes = list(res["nodes"])
    rows = [p for p in range(n_paths) if gacc[p] == acc and retrieve[p, : acc + 1].tolist() == nodes]
    assert rows, ("GPU nodes are no accepted row prefix", nodes)
    if mode == GREEDY:
        assert int(res["best"]) == int(np.argmax(gacc)), (res["best"], int(np.argmax(gacc)))
    if not diverged:
        same = res["best"] == ref["best"] and acc == ref["acc"] and nodes == ref["nodes"].tolist()
        if not same:
            assert mode == TYPICAL and acc == ref["acc"], (res, ref["best"], ref["acc"])
            cand = np.flatnonzero(oacc == ref["acc"])
            like = np.sort(np.asarray(ref["likelihood"])[cand])[::-1]
            assert len(like) > 1 and like[0] - like[1] < MARGIN, like[:2]
    return diverged
