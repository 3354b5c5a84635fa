"""Pins of the oracle's backbone pieces, tree attention and Medusa heads (CPU).

Each function is tied to a closed form, a library routine or an invariant
the pages state, never to a retyped copy of itself:
* RMSNorm, SiLU, RoPE: closed forms and torch.nn.functional.
* masked attention: torch.nn.functional.scaled_dot_product_attention.
* tree attention: every node equals its root-to-node path run as an
  independent causal sequence ("大模型推理 memory bandwidth bound (5) -
  Medusa", 一.2 Tree attention; "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 4️⃣).
* Medusa head: a hand-built case with SiLU(ln 3) = 0.75 ln 3 (一.1 Medusa heads).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle.decode import chain_mask
from oracle.model import (Backbone, KVCache, argmax_first, masked_attention, medusa_heads, rms_norm,
                          rope, silu, topk_ids, tree_attention)
from oracle.tree import tree_buffers


def test_rms_norm_closed_form_and_library():
    x = np.full((1, 8), 3.0)
    assert np.allclose(rms_norm(x, 1e-5), 3.0 / math.sqrt(9.0 + 1e-5), rtol=0, atol=1e-15)
    y = np.random.default_rng(0).normal(size=(5, 33))
    ref = F.rms_norm(torch.tensor(y), (33,), eps=1e-5).numpy()
    assert np.allclose(rms_norm(y, 1e-5), ref, rtol=1e-14, atol=1e-14)


def test_silu_closed_form():
    v = silu(np.array([math.log(3), 0.0, -math.log(3)]))
    assert np.allclose(v, [0.75 * math.log(3), 0.0, -0.25 * math.log(3)], rtol=0, atol=1e-15)
    z = np.linspace(-8, 8, 101)
    assert np.allclose(silu(z), F.silu(torch.tensor(z)).numpy(), rtol=1e-14, atol=1e-15)


def test_rope_closed_form():
    # D=4, theta=100: pair (0,2) turns by pos * 1 rad, pair (1,3) by pos * 0.1 rad
    x = np.array([[[1.0, 0.0, 0.0, 0.0]], [[0.0, 1.0, 0.0, 0.0]]])
    out = rope(x, [1, 1], 100.0)
    assert np.allclose(out[0, 0], [0.5403023058681398, 0, 0.8414709848078965, 0], atol=1e-15)
    assert np.allclose(out[1, 0], [0, 0.9950041652780258, 0, 0.09983341664682815], atol=1e-15)
    assert np.allclose(rope(x, [0, 0], 100.0), x)           # position 0 is the identity


def test_rope_relative_position():
    rng = np.random.default_rng(1)
    q, k = rng.normal(size=(1, 1, 16)), rng.normal(size=(1, 1, 16))
    d1 = (rope(q, [7], 1e4) * rope(k, [3], 1e4)).sum()
    d2 = (rope(q, [104], 1e4) * rope(k, [100], 1e4)).sum()
    assert abs(d1 - d2) < 1e-12                              # depends on m - n only


def test_masked_attention_vs_sdpa():
    rng = np.random.default_rng(2)
    n, H, D = 11, 3, 8
    q, k, v = (rng.normal(size=(n, H, D)) for _ in range(3))
    out = masked_attention(q, k, v, np.tril(np.ones((n, n), bool)), 1 / math.sqrt(D))
    t = lambda a: torch.tensor(a).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_tree_attention_equals_independent_paths():
    rng = np.random.default_rng(3)
    tree = tree_buffers(synth.synthetic_tree_choices(64, 4, 10), 10)
    n, H, D, P = tree["n_nodes"], 2, 16, 9
    q = rng.normal(size=(n, H, D))
    kc, vc = rng.normal(size=(P + n, H, D)), rng.normal(size=(P + n, H, D))
    out = tree_attention(q, kc, vc, P, tree["attn_mask"], 0.25)
    t = lambda a: torch.tensor(a).permute(1, 0, 2)[None]
    for row in tree["retrieve"]:
        path = [int(p) for p in row if p >= 0]
        rows = list(range(P)) + [P + p for p in path]
        # the path as its own causal sequence after the prefix: query of path node j sees rows[:P+j+1]
        L = len(rows)
        allowed = np.tril(np.ones((L, L), bool))
        qq = np.concatenate([rng.normal(size=(P, H, D)), q[path]])
        ref = F.scaled_dot_product_attention(t(qq), t(kc[rows]), t(vc[rows]),
                                             attn_mask=torch.tensor(allowed), scale=0.25)[0].permute(1, 0, 2)
        assert np.allclose(out[path], ref[P:].numpy(), rtol=1e-12, atol=1e-12)


def test_single_node_tree_is_decode_attention():
    rng = np.random.default_rng(4)
    P, H, D = 20, 2, 8
    q, kc, vc = rng.normal(size=(1, H, D)), rng.normal(size=(P + 1, H, D)), rng.normal(size=(P + 1, H, D))
    out = tree_attention(q, kc, vc, P, np.ones((1, 1), np.uint8), 0.3)
    t = lambda a: torch.tensor(a).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(t(q), t(kc), t(vc), scale=0.3)[0].permute(1, 0, 2).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_medusa_head_hand_case():
    # d = 3, V = 4: W1 h = [ln3, 0, -ln3]; u = SiLU(W1 h) + h; W2 picks / sums entries of u
    h = np.array([1.0, 2.0, -1.0])
    W1 = np.diag([math.log(3), 0.0, math.log(3)])
    W2 = np.array([[1, 0, 0], [0, 1, 0], [0, 0, 1], [1, 1, 1]], float)
    w = {"medusa0.w1": W1, "medusa0.w2": W2}
    z = medusa_heads(w.__getitem__, 1, h)[0]
    u = [0.75 * math.log(3) + 1.0, 0.0 + 2.0, -0.25 * math.log(3) - 1.0]
    assert np.allclose(z, [u[0], u[1], u[2], sum(u)], rtol=0, atol=1e-14)
    # W1 = 0: SiLU(0) = 0, so z = W2 h
    w0 = {"medusa0.w1": np.zeros((3, 3)), "medusa0.w2": W2}
    assert np.allclose(medusa_heads(w0.__getitem__, 1, h)[0], [1, 2, -1, 2])


def test_topk_and_argmax_ties():
    z = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert topk_ids(z, 3).tolist() == [1, 2, 4]
    assert topk_ids(z, 5).tolist() == [1, 2, 4, 3, 0]
    assert argmax_first(z) == 1
    big = np.zeros(1000)
    big[[5, 900, 17]] = [2.0, 2.0, 1.0]
    assert topk_ids(big, 4).tolist() == [5, 900, 17, 0]


def _tiny_model():
    dims = synth.TINY
    w = {k: v.double().numpy() for k, v in synth.model_weights(dims, seed=0).items()}
    return dims, w


def test_backbone_residual_structure():
    # with every output projection zero the layers add nothing: logits = rmsnorm(E[t]) W_lm^T
    dims, w = _tiny_model()
    w0 = dict(w)
    for l in range(dims.n_layers):
        w0[f"layer{l}.wo"] = np.zeros_like(w[f"layer{l}.wo"])
        w0[f"layer{l}.w_down"] = np.zeros_like(w[f"layer{l}.w_down"])
    m = Backbone(dims, w0.__getitem__)
    toks = np.array([3, 17, 400])
    h, logits = m.forward(toks, np.arange(3), KVCache(dims, 8), 0, chain_mask(3))
    e = w["embed"][toks]
    hh = e / np.sqrt((e * e).mean(1, keepdims=True) + 1e-5)
    assert np.allclose(h, hh, rtol=1e-13, atol=1e-13)
    assert np.allclose(logits, hh @ w["lm_head"].T, rtol=1e-12, atol=1e-13)


def test_backbone_layer_vs_torch_functional():
    """One decoder layer against the same layer assembled from torch.nn.functional routines."""
    dims, w = _tiny_model()
    one = synth.ModelDims(d=dims.d, n_layers=1, n_heads=dims.n_heads, head_dim=dims.head_dim,
                          ffn=dims.ffn, vocab=dims.vocab, n_medusa=0)
    m = Backbone(one, w.__getitem__)
    n, H, D = 6, one.n_heads, one.head_dim
    toks = np.array([1, 5, 9, 200, 301, 7])
    h, _ = m.forward(toks, np.arange(n), KVCache(one, 8), 0, chain_mask(n))
    T = lambda a: torch.tensor(a)
    x = T(w["embed"][toks])
    a = F.rms_norm(x, (one.d,), eps=1e-5)
    q, k, v = (F.linear(a, T(w[f"layer0.w{c}"])).view(n, H, D) for c in "qkv")
    # rotary via complex multiplication of (x_i + i x_{i+D/2}) by e^{i pos theta^{-2i/D}}
    ang = torch.arange(n, dtype=torch.float64)[:, None] * (1e4 ** (-torch.arange(0, D, 2, dtype=torch.float64) / D))
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    cplx = lambda t: torch.complex(t[..., : D // 2], t[..., D // 2:]) * rot
    q, k = (torch.cat([c.real, c.imag], -1) for c in (cplx(q), cplx(k)))
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), k.permute(1, 0, 2), v.permute(1, 0, 2),
                                       is_causal=True).permute(1, 0, 2).reshape(n, H * D)
    x = x + F.linear(o, T(w["layer0.wo"]))
    a = F.rms_norm(x, (one.d,), eps=1e-5)
    x = x + F.linear(F.silu(F.linear(a, T(w["layer0.w_gate"]))) * F.linear(a, T(w["layer0.w_up"])),
                     T(w["layer0.w_down"]))
    ref = F.rms_norm(x, (one.d,), eps=1e-5).numpy()
    assert np.allclose(h, ref, rtol=1e-11, atol=1e-12)


def test_backbone_store_hook_placement():
    """The storage hook sits on the named intermediates: zeroing one of them equals zeroing the weight that
    produces it (or the one that consumes it), and the default hook changes nothing."""
    dims, w = _tiny_model()
    toks, n = np.array([3, 17, 400, 9]), 4

    def run(weights, store=None):
        m = Backbone(dims, weights.__getitem__) if store is None else Backbone(dims, weights.__getitem__, store)
        return m.forward(toks, np.arange(n), KVCache(dims, 8), 0, chain_mask(n))[1]

    base = run(w)
    assert np.array_equal(run(w, lambda name, v: v), base)
    for name, zeroed in (("o", "wo"), ("v", "wo"), ("act", "w_down")):
        wz = dict(w)
        for l in range(dims.n_layers):
            wz[f"layer{l}.{zeroed}"] = np.zeros_like(w[f"layer{l}.{zeroed}"])
        got = run(w, lambda nm, v, name=name: np.zeros_like(v) if nm == name else v)
        assert np.allclose(got, run(wz), rtol=1e-12, atol=1e-13), name
    # rounding the stored intermediates to bf16 moves the tiny model's logits by a small, nonzero amount
    bf = lambda nm, v: torch.tensor(v).to(torch.bfloat16).double().numpy()
    rel = np.linalg.norm(run(w, bf) - base) / np.linalg.norm(base)
    assert 1e-5 < rel < 2e-2, rel
