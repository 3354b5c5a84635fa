"""Posterior evaluation: greedy and typical acceptance (oracle; test infrastructure only).

"大模型推理 memory bandwidth bound (5) - Medusa", 一.3 Typical acceptance and
二.6 evaluate_posterior(). For every path (a row of retrieve) and position j,
the candidate token of the path's node j+1 is checked against the target
distribution computed at the path's node j:

* greedy (temperature 0): accepted iff it equals argmax of node j's logits;
* typical ("fast" branch): with p = softmax(logits / T),
  H = -sum p log(p + 1e-5) and tau = min(eps, delta * exp(-H)), accepted iff
  p(candidate) > tau (eta-sampling's allow set).

accept length of a path = number of consecutive accepted positions from the
start. The best path has the largest accept length; greedy takes the first
such row, typical takes the row with the largest sum of log p(candidate)
over its accepted positions (first row on equal likelihood). With nothing
accepted the best row is 0.

Readings: positions past the end of a path (retrieve = -1) are never
accepted (the page's code maps them to token 0 and to the last node's logits,
which could accept a node that does not exist). The page's default arguments
(0.09 / 0.3) are swapped between functions and its comment writes
alpha * H; the formula of 一.3 is delta * exp(-H), with eps = 0.09 and
delta = 0.3 the defaults of medusa_generate().
"""
from __future__ import annotations

import numpy as np

GREEDY, TYPICAL = 0, 1


def node_stats(logits, mode, temperature=1.0, eps=0.09, delta=0.3):
    """Per-node statistics in float64.

    greedy: dict(argmax [n], top1 [n], top2 [n]) (top2 = second-largest value).
    typical: dict(logp [n, V] = log softmax(z/T), entropy [n], tau [n]).
    """
    z = np.asarray(logits, dtype=np.float64)
    if mode == GREEDY:
        am = np.argmax(z, axis=1)
        srt = np.sort(z, axis=1)
        return dict(argmax=am, top1=srt[:, -1], top2=srt[:, -2])
    y = z / temperature
    y = y - y.max(axis=1, keepdims=True)
    p = np.exp(y)
    p = p / p.sum(axis=1, keepdims=True)
    H = -np.sum(p * np.log(p + 1e-5), axis=1)
    tau = np.minimum(eps, delta * np.exp(-H))
    return dict(logp=np.log(p), p=p, entropy=H, tau=tau)


def evaluate_posterior(logits, tree_tokens, retrieve, mode, temperature=1.0, eps=0.09, delta=0.3):
    """Best path, accept length and accepted nodes; also every decision's margin.

    logits [n, V] (one row per tree node), tree_tokens [n] (candidate token of
    each node), retrieve [n_paths, depth+1] (-1 padded). Returns dict(best,
    acc, nodes (retrieve[best, :acc+1]), next_node (retrieve[best, acc]),
    accept_len [n_paths], margins (list of (path, j, margin)) -- the margin of
    the decision at position j: greedy: top1 - logit(candidate) if rejected,
    top1 - top2 if accepted; typical: |ln p(candidate) - ln tau|.
    """
    st = node_stats(logits, mode, temperature, eps, delta)
    retrieve = np.asarray(retrieve)
    n_paths, width = retrieve.shape
    z = np.asarray(logits, dtype=np.float64)
    acc = np.zeros(n_paths, dtype=np.int64)
    like = np.zeros(n_paths)
    margins = []
    for p in range(n_paths):
        for j in range(width - 1):
            node, child = retrieve[p, j], retrieve[p, j + 1]
            if child < 0:
                break
            tok = int(tree_tokens[child])
            if mode == GREEDY:
                ok = tok == int(st["argmax"][node])
                m = (st["top1"][node] - st["top2"][node]) if ok else (st["top1"][node] - z[node, tok])
            else:
                lp, lt = st["logp"][node, tok], np.log(st["tau"][node])
                ok = lp > lt
                m = abs(lp - lt)
            margins.append((p, j, float(m)))
            if not ok:
                break
            acc[p] += 1
            if mode == TYPICAL:
                like[p] += st["logp"][node, tok]
    amax = int(acc.max())
    if amax == 0:
        best = 0
    elif mode == GREEDY:
        best = int(np.argmax(acc))
    else:
        cands = np.flatnonzero(acc == amax)
        best = int(cands[np.argmax(like[cands])])
    nodes = retrieve[best, : amax + 1].copy()
    return dict(best=best, acc=amax, nodes=nodes, next_node=int(nodes[-1]), accept_len=acc,
                likelihood=like, margins=margins, stats=st)
