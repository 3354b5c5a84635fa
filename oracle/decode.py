"""Candidates, the verify step and the greedy decode loops (oracle; test infrastructure only).

"大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate() and
its steps: 二.3 initialize_medusa() (prefill; root = argmax of the last LM
logits, head top-k of the last Medusa logits), 二.4 generate_candidates()
(candidates = [root] + per-head top-k flattened; tree_candidates =
candidates[tree_indices]; cart_candidates = tree_candidates padded with token
0, indexed by retrieve), 二.5 tree_decoding(), 二.6 evaluate_posterior(),
二.7 update_inference_inputs() (append cart[best, :acc+1]; compact the KV
cache; the next LM/Medusa logits are those of node retrieve[best, acc]).

The reference evaluates the Medusa heads on all tree nodes and keeps the row
of node retrieve[best, acc]; here the heads run on that node only, which is
the same consumed value. The root is the argmax of the LM logits (the
temperature-0 / "fast" branch of generate_candidates()), or drawn by a root
sampler of ``sampling`` (the branch for temperature > 0 without "fast").

Greedy equivalence ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu",
2️⃣: under greedy decoding the output is identical token for token) is the
pin between ``medusa_greedy_decode`` and ``ar_greedy_decode``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .kv import kv_compact
from .model import Backbone, KVCache, argmax_first, medusa_heads, topk_ids
from .posterior import GREEDY, evaluate_posterior


def generate_candidates(root, head_topk, tree):
    """(tree_tokens [n], cart [n_paths, depth+1]) from the root token and head_topk [K, topk]."""
    cand = np.concatenate([[int(root)], np.asarray(head_topk, dtype=np.int64).reshape(-1)])
    tree_tokens = cand[tree["tree_indices"]]
    ext = np.concatenate([tree_tokens, [0]])
    cart = ext[tree["retrieve"]]          # retrieve = -1 picks the appended 0
    return tree_tokens, cart


@dataclass
class DecodeState:
    cache: KVCache
    cur_len: int
    root: int
    head_topk: np.ndarray     # [K, topk]


def chain_mask(n):
    """Causal mask of a chain of n tokens (lower triangle, diagonal included)."""
    return np.tril(np.ones((n, n), dtype=np.uint8))


def prefill(model: Backbone, prompt, s_max, topk, root=None):
    """Forward the prompt causally; root = argmax of its last logits (or ``root(logits row)``, e.g. a
    ``sampling.RootSampler``), heads on its last state."""
    cache = KVCache(model.dims, s_max)
    P = len(prompt)
    h, logits = model.forward(np.asarray(prompt), np.arange(P), cache, 0, chain_mask(P))
    z = medusa_heads(model.get, model.dims.n_medusa, h[-1])
    r0 = argmax_first(logits[-1]) if root is None else root(logits[-1])
    return DecodeState(cache, P, r0, np.stack([topk_ids(r, topk) for r in z]))


def verify_step(model: Backbone, st: DecodeState, tree, mode=GREEDY, temperature=1.0, eps=0.09, delta=0.3,
                root=None):
    """One Medusa verify step. Returns (accepted tokens, details) and advances ``st``. The next root is the
    argmax of node retrieve[best, acc]'s logits, or ``root(that row)`` when a root sampler is given."""
    tree_tokens, cart = generate_candidates(st.root, st.head_topk, tree)
    pos = st.cur_len + tree["position_ids"]
    h, logits = model.forward(tree_tokens, pos, st.cache, st.cur_len, tree["attn_mask"])
    post = evaluate_posterior(logits, tree_tokens, tree["retrieve"], mode, temperature, eps, delta)
    st.cache.data, new_len = kv_compact(st.cache.data, st.cur_len, post["nodes"])
    out = cart[post["best"], : post["acc"] + 1].copy()
    nn = post["next_node"]
    z = medusa_heads(model.get, model.dims.n_medusa, h[nn])
    prev_len = st.cur_len
    st.cur_len = new_len
    st.root = argmax_first(logits[nn]) if root is None else root(logits[nn])
    st.head_topk = np.stack([topk_ids(r, tree["topk"]) for r in z])
    return out, dict(post=post, tree_tokens=tree_tokens, cart=cart, logits=logits, hidden=h,
                     prefix_len=prev_len, head_logits=z)


def medusa_greedy_decode(model: Backbone, prompt, n_new, tree, s_max):
    """Greedy Medusa decoding of exactly ``n_new`` tokens (the last step's tokens are truncated)."""
    st = prefill(model, prompt, s_max, tree["topk"])
    out, accs = [], []
    while len(out) < n_new:
        toks, info = verify_step(model, st, tree, GREEDY)
        out.extend(int(t) for t in toks)
        accs.append(info["post"]["acc"])
    return np.asarray(out[:n_new]), accs


def ar_greedy_decode(model: Backbone, prompt, n_new, s_max):
    """Plain greedy autoregressive decoding, one token per forward, with a KV cache."""
    cache = KVCache(model.dims, s_max)
    P = len(prompt)
    _, logits = model.forward(np.asarray(prompt), np.arange(P), cache, 0, chain_mask(P))
    cur, out = P, []
    tok = argmax_first(logits[-1])
    for _ in range(n_new):
        out.append(tok)
        _, logits = model.forward(np.asarray([tok]), np.asarray([cur]), cache, cur, chain_mask(1))
        cur += 1
        tok = argmax_first(logits[-1])
    return np.asarray(out)


def teacher_forced_logits(model: Backbone, prompt, generated, s_max):
    """LM logits of one causal forward over prompt + generated; row i predicts generated[i]."""
    seq = np.concatenate([np.asarray(prompt), np.asarray(generated)])
    cache = KVCache(model.dims, s_max)
    _, logits = model.forward(seq, np.arange(len(seq)), cache, 0, chain_mask(len(seq)))
    P = len(prompt)
    return logits[P - 1: P - 1 + len(generated)]
