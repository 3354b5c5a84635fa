"""Static token-tree buffers from a list of rank tuples (oracle; test infrastructure only).

Follows "大模型推理 memory bandwidth bound (5) - Medusa", 二.2
generate_medusa_buffers(): the input is a list of rank tuples (root excluded),
e.g. (0, 1) = "rank 1 of head 2 under rank 0 of head 1"; the outputs are the
ancestor mask, tree_indices, position ids and retrieve indices.

Readings where the page prints values but not the rule:
* node order: the root is node 0, then the tuples sorted by (length, tuple);
* retrieve rows: one per leaf (a node that is no proper prefix of another),
  leaves in descending node order; each row is the root-to-leaf node list
  padded with -1 to ``max_depth + 1`` entries. This reproduces the printed
  42 x 5 table of the page exactly.
"""
from __future__ import annotations

import numpy as np


def sort_choices(choices):
    """Tuples sorted by (length, lexicographic) -- the page's sorted_medusa_choices."""
    return sorted((tuple(c) for c in choices), key=lambda c: (len(c), c))


def tree_buffers(choices, topk: int):
    """All static buffers of the tree given by ``choices`` (rank tuples, root excluded).

    Returns a dict:
      n_nodes, depth (max tuple length), sorted (node -> tuple, root = ()),
      attn_mask  [n, n] uint8: 1 where column j is an ancestor of row i or i itself
                 (the root is an ancestor of every node, so column 0 is all ones),
      tree_indices [n] int64: index into [root token, head-1 top-k, head-2 top-k, ...];
                 the root maps to 0 and a node at depth L with last rank r to
                 1 + topk*(L-1) + r (page: "each head takes 10; the token's index
                 among all 1+10+10+... tokens"),
      position_ids [n] int64: depth of each node (root 0),
      retrieve   [n_leaves, depth+1] int64, -1 padded,
      parent     [n] int64 (-1 for the root).
    """
    srt = sort_choices(choices)
    if len(set(srt)) != len(srt):
        raise ValueError("duplicate choice")
    node_of = {(): 0}
    for i, c in enumerate(srt):
        node_of[c] = i + 1
    for c in srt:
        if len(c) == 0 or c[:-1] not in node_of:
            raise ValueError(f"choices are not prefix-closed at {c}")
        if max(c) >= topk or min(c) < 0:
            raise ValueError(f"rank out of range in {c}")
    nodes = [()] + srt
    n = len(nodes)
    depth = max(len(c) for c in nodes)

    mask = np.zeros((n, n), dtype=np.uint8)
    for i, ci in enumerate(nodes):
        for j, cj in enumerate(nodes):
            if ci[: len(cj)] == cj:          # cj is a prefix of ci (root = () is a prefix of all)
                mask[i, j] = 1

    tree_indices = np.array([0] + [1 + topk * (len(c) - 1) + c[-1] for c in srt], dtype=np.int64)
    position_ids = np.array([len(c) for c in nodes], dtype=np.int64)
    parent = np.array([-1] + [node_of[c[:-1]] for c in srt], dtype=np.int64)

    is_prefix_of_other = set()
    for c in srt:
        for L in range(len(c)):
            is_prefix_of_other.add(c[:L])
    leaves = [i for i in range(n) if nodes[i] not in is_prefix_of_other]
    retrieve = np.full((len(leaves), depth + 1), -1, dtype=np.int64)
    for row, leaf in enumerate(sorted(leaves, reverse=True)):
        c = nodes[leaf]
        for L in range(len(c) + 1):
            retrieve[row, L] = node_of[c[:L]]
    return dict(n_nodes=n, depth=depth, sorted=nodes, attn_mask=mask, tree_indices=tree_indices,
                position_ids=position_ids, retrieve=retrieve, parent=parent, topk=topk)
