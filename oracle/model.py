"""Llama-style backbone, tree attention and Medusa heads in float64 (oracle; test infrastructure only).

* Medusa head k on hidden state h: ``z_k = W2_k (SiLU(W1_k h) + h)`` with
  W1_k d x d and W2_k taking d to the vocabulary -- "大模型推理 memory
  bandwidth bound (5) - Medusa", 一.1 Medusa heads. The softmax of that
  formula is monotone, so the per-head top-k taken on ``z_k`` is the top-k of
  p^(k) (二.4 generate_candidates() takes torch.topk on the head logits).
* Tree attention: the tree is flattened into a sequence and each node attends
  to the whole cached prefix plus its own root-to-node path, never to
  siblings -- same page, 一.2 Tree attention and 二.2 (the mask's ones);
  "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 4️⃣.
* Tree decoding positions: ``position_ids = medusa_position_ids + prefix
  length`` -- same page, 二.5 tree_decoding().

The backbone itself is not on the pages; the plainest Llama reading is used:
pre-norm RMSNorm (eps 1e-5, gains 1), rotary embedding with theta 10000 and
rotate-half pairing (i, i + D/2), SiLU-gated FFN, untied LM head, no biases,
attention scale 1/sqrt(head_dim). The Medusa heads read the final-normed
hidden state, the same vector the LM head reads.
"""
from __future__ import annotations

import numpy as np


def rms_norm(x, eps):
    """x / sqrt(mean(x^2) + eps) along the last axis (gain 1)."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def silu(x):
    """SiLU(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    return x / (1.0 + np.exp(-x))


def rope(x, pos, theta):
    """Rotary embedding of x [n, H, D] at integer positions pos [n].

    Pair (i, i + D/2) is rotated by the angle pos * theta**(-2i/D).
    """
    D = x.shape[-1]
    half = D // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / D)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]       # [n, half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def masked_attention(q, k, v, allowed, scale):
    """softmax(q k^T * scale) v per head, over keys where ``allowed[i, j]``.

    q [nq, H, D], k/v [nk, H, D], allowed [nq, nk] bool. Every query row must
    allow at least one key.
    """
    s = np.einsum("ihd,jhd->hij", q, k) * scale                   # [H, nq, nk]
    s = np.where(allowed[None], s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return np.einsum("hij,jhd->ihd", p, v)


def tree_attention(q, k_cache, v_cache, prefix_len, attn_mask, scale):
    """Tree attention of the n tree queries q [n, H, D].

    k_cache/v_cache are [S, H, D] and already hold the tree block's keys and
    values at rows prefix_len .. prefix_len+n-1. Node i sees every prefix row
    and tree row prefix_len + j where attn_mask[i, j] = 1.
    """
    n = q.shape[0]
    allowed = np.zeros((n, prefix_len + n), dtype=bool)
    allowed[:, :prefix_len] = True
    allowed[:, prefix_len:] = attn_mask.astype(bool)
    return masked_attention(q, k_cache[: prefix_len + n], v_cache[: prefix_len + n], allowed, scale)


class KVCache:
    """Keys and values of every layer: data[l, 0] = K, data[l, 1] = V, each [H, S_max, D]."""

    def __init__(self, dims, s_max, data=None):
        self.dims = dims
        shape = (dims.n_layers, 2, dims.n_heads, s_max, dims.head_dim)
        self.data = np.zeros(shape) if data is None else np.array(data, dtype=np.float64)
        assert self.data.shape == shape

    def k(self, l):  # [S, H, D] view
        return self.data[l, 0].transpose(1, 0, 2)

    def v(self, l):
        return self.data[l, 1].transpose(1, 0, 2)


def _exact(name, v):
    return v


class Backbone:
    """The decoder. ``get(name)`` returns the float64 weight ``name`` (see synth.weight_names).

    ``store(name, v)`` is applied to each intermediate that a path keeps in memory between its stages: the
    normalised projection operands ("a"), the rotated queries and keys and the values ("q", "k", "v"), the
    attention output ("o") and the SiLU-gate product ("act"). It is the identity by default, so the oracle is
    exact; rounding there to a storage precision measures how sensitive the model's outputs are to that
    precision (it changes no arithmetic step).
    """

    def __init__(self, dims, get, store=_exact):
        self.dims, self.get, self.store = dims, get, store

    def forward(self, tokens, positions, cache: KVCache, cache_len, block_mask):
        """Run ``tokens`` [n] at ``positions`` [n] after ``cache_len`` cached rows.

        Their keys/values are written to cache rows cache_len .. cache_len+n-1;
        token i attends to every cached row and to new row j where
        block_mask[i, j] = 1 (lower-triangular for a causal chunk, the tree's
        ancestor mask for a tree). Returns (h, logits): the final-normed
        hidden states [n, d] and the LM-head logits [n, V].
        """
        D, H, g, st = self.dims.head_dim, self.dims.n_heads, self.get, self.store
        eps, n = self.dims.norm_eps, len(tokens)
        x = g("embed")[np.asarray(tokens)]
        for l in range(self.dims.n_layers):
            a = st("a", rms_norm(x, eps))
            q = (a @ g(f"layer{l}.wq").T).reshape(n, H, D)
            k = (a @ g(f"layer{l}.wk").T).reshape(n, H, D)
            v = (a @ g(f"layer{l}.wv").T).reshape(n, H, D)
            q, k = rope(q, positions, self.dims.rope_theta), rope(k, positions, self.dims.rope_theta)
            q, k, v = st("q", q), st("k", k), st("v", v)
            cache.k(l)[cache_len:cache_len + n] = k
            cache.v(l)[cache_len:cache_len + n] = v
            o = st("o", tree_attention(q, cache.k(l), cache.v(l), cache_len, block_mask, 1.0 / np.sqrt(D)))
            x = x + o.reshape(n, H * D) @ g(f"layer{l}.wo").T
            a = st("a", rms_norm(x, eps))
            u = st("act", silu(a @ g(f"layer{l}.w_gate").T) * (a @ g(f"layer{l}.w_up").T))
            x = x + u @ g(f"layer{l}.w_down").T
        h = st("a", rms_norm(x, eps))
        return h, h @ g("lm_head").T


def medusa_heads(get, n_medusa, h):
    """Head logits z [K, V] on one hidden state h [d]: z_k = W2_k (SiLU(W1_k h) + h)."""
    return np.stack([get(f"medusa{k}.w2") @ (silu(get(f"medusa{k}.w1") @ h) + h) for k in range(n_medusa)])


def topk_ids(z, k):
    """Indices of the k largest entries of z, largest first; equal values: lower index first."""
    order = sorted(range(len(z)), key=lambda i: (-z[i], i)) if len(z) <= 64 else \
        np.lexsort((np.arange(len(z)), -np.asarray(z)))
    return np.asarray(order[:k], dtype=np.int64)


def argmax_first(z):
    """Index of the largest entry; the lowest such index on ties (torch.argmax semantics)."""
    return int(np.argmax(z))
