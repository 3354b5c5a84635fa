"""Pins of the oracle's root samplers (CPU).

"大模型推理 memory bandwidth bound (5) - Medusa", 二.4 generate_candidates()
(get_typical_one_token / get_nucleus_one_token for temperature > 0) and 一.3
(typical acceptance = eta-sampling's allow set); nucleus sampling as defined
by Holtzman et al. (2020): the smallest leading set of the tokens, largest
probability first, whose mass reaches top_p.

* hand-computed allow sets and draws (typical on logits [2, 1, 0, -1];
  nucleus on p = [.05, .5, .2, .25] at T = 1 and T = 0.5; tied logits);
* the nucleus set against its definition on random rows: its mass reaches
  top_p and dropping its least likely member falls below it; every kept token
  is at least as likely as every dropped one;
* the typical set always holds the argmax (Jensen bound of the readings);
* the draw: on a grid of N uniforms each token is drawn N q_k +- 1 times,
  q the renormalised kept distribution;
* the uniform: counter 0 under key 0 is the published first SplitMix64 word;
* a nucleus decode with top_p -> 0 keeps only the argmax, so it reproduces
  greedy autoregressive decoding of the tiny decoder.
"""
import math

import numpy as np
import torch

import synth
from oracle.decode import ar_greedy_decode, prefill, verify_step
from oracle.model import Backbone
from oracle.posterior import GREEDY
from oracle.sampling import (NUCLEUS, TYPICAL_ONE, RootSampler, inverse_cdf, nucleus_allow, sample_root,
                             softmax_t, typical_allow, uniform)
from oracle.tree import tree_buffers


def test_typical_one_token_hand_values():
    # p = [.643914, .236883, .087144, .032059], H = .947497, tau = eps = .09: allow {0, 1}, q0 = e / (e + 1)
    z = np.array([2.0, 1.0, 0.0, -1.0])
    allow, margin = typical_allow(z, 1.0, 0.09, 0.3)
    assert allow.tolist() == [True, True, False, False]
    assert abs(margin[2] - math.log(0.087144 / 0.09)) < 1e-5
    q0 = math.e / (math.e + 1.0)                                  # 0.7310585786
    for u, tok in [(0.0, 0), (0.5, 0), (q0 - 1e-9, 0), (q0 + 1e-9, 1), (0.999999, 1)]:
        assert sample_root(z, TYPICAL_ONE, 1.0, 0.09, 0.3, u=u) == tok, u
    # eps = 0: tau = 0, every token is kept: the draw is the plain categorical inverse CDF of softmax(z)
    p = np.exp(z) / np.exp(z).sum()
    assert sample_root(z, TYPICAL_ONE, 1.0, 0.0, 0.3, u=p[0] + p[1] + 1e-9) == 2


def test_nucleus_hand_values():
    p = np.array([0.05, 0.5, 0.2, 0.25])
    z = np.log(p)
    # order 1, 3, 2, 0 with mass before 0, .5, .75, .95: top_p .8 keeps {1, 3, 2}
    allow, before = nucleus_allow(z, 1.0, 0.8)
    assert allow.tolist() == [False, True, True, True]
    assert np.allclose(before, [0.95, 0.0, 0.75, 0.5])
    c1, c2 = 0.5 / 0.95, 0.7 / 0.95                              # cumulative in vocabulary order
    for u, tok in [(0.1, 1), (c1 - 1e-9, 1), (c1 + 1e-9, 2), (0.6, 2), (c2 + 1e-9, 3), (0.9, 3)]:
        assert sample_root(z, NUCLEUS, 1.0, top_p=0.8, u=u) == tok, u
    # top_p .7: {1, 3}, q = [0, 2/3, 0, 1/3]; top_p .45: {1} only
    assert nucleus_allow(z, 1.0, 0.7)[0].tolist() == [False, True, False, True]
    assert [sample_root(z, NUCLEUS, 1.0, top_p=0.7, u=u) for u in (0.6, 0.7)] == [1, 3]
    assert {sample_root(z, NUCLEUS, 1.0, top_p=0.45, u=u) for u in np.linspace(0, 0.999, 11)} == {1}
    # T = 0.5 squares p: [.0025, .25, .04, .0625] / .355 = [.00704, .70423, .11268, .17606]: top_p .8 keeps {1, 3}
    assert np.allclose(softmax_t(z, 0.5), [0.0025 / 0.355, 0.25 / 0.355, 0.04 / 0.355, 0.0625 / 0.355])
    assert nucleus_allow(z, 0.5, 0.8)[0].tolist() == [False, True, False, True]


def test_nucleus_ties_lower_index_first():
    # logits [1, 3, 3, 0]: p1 = p2 = e^3 / (e + 2 e^3 + 1) = .457640; top_p .3 keeps token 1 only, .5 keeps 1 and 2
    z = np.array([1.0, 3.0, 3.0, 0.0])
    assert nucleus_allow(z, 1.0, 0.3)[0].tolist() == [False, True, False, False]
    assert nucleus_allow(z, 1.0, 0.5)[0].tolist() == [False, True, True, False]
    assert abs(softmax_t(z, 1.0)[1] - 0.457640) < 1e-6


def test_nucleus_set_is_the_smallest_leading_set():
    for seed in range(6):
        z = synth.normal(seed, "nucleus", (1000,), 2.0, dtype=torch.float64).numpy()
        for T, top_p in [(0.7, 0.8), (1.0, 0.5), (0.3, 0.95), (2.0, 0.8)]:
            p = softmax_t(z, T)
            allow, _ = nucleus_allow(z, T, top_p)
            mass = p[allow].sum()
            assert mass >= top_p - 1e-12
            assert mass - p[allow].min() < top_p
            assert p[allow].min() >= p[~allow].max()
            k = int(np.argmax(z))
            assert allow[k]


def test_typical_set_holds_the_argmax():
    for seed in range(6):
        for scale in (0.01, 1.0, 5.0):
            z = synth.normal(seed, "typical", (32000,), scale, dtype=torch.float64).numpy()
            for T in (0.3, 0.7, 1.5):
                allow, margin = typical_allow(z, T, 0.09, 0.3)
                assert allow[int(np.argmax(z))]
                assert (allow == (margin > 0)).all()


def test_draw_follows_the_kept_distribution():
    N = 20000
    us = (np.arange(N) + 0.5) / N
    for seed, mode in [(0, TYPICAL_ONE), (1, NUCLEUS), (2, NUCLEUS)]:
        z = synth.normal(seed, "draw", (40,), 1.5, dtype=torch.float64).numpy()
        p = softmax_t(z, 0.7)
        allow = typical_allow(z, 0.7, 0.09, 0.3)[0] if mode == TYPICAL_ONE else nucleus_allow(z, 0.7, 0.8)[0]
        q = np.where(allow, p, 0.0) / p[allow].sum()
        counts = np.bincount([sample_root(z, mode, 0.7, 0.09, 0.3, 0.8, u) for u in us], minlength=40)
        assert (counts[~allow] == 0).all()
        assert np.abs(counts - N * q).max() <= 1.0 + 1e-9


def test_inverse_cdf_edges():
    p = np.array([0.25, 0.25, 0.5])
    allow = np.array([True, False, True])
    assert inverse_cdf(p, allow, 0.0) == 0
    assert inverse_cdf(p, allow, 1.0 / 3.0 + 1e-12) == 2
    assert inverse_cdf(p, allow, 1.0 - 2 ** -53) == 2
    assert inverse_cdf(p, np.zeros(3, dtype=bool), 0.5) == 2   # nothing kept: the argmax


def test_uniform_is_the_published_splitmix_word():
    assert uniform(0, 0) == (0xE220A8397B1DCDAF >> 11) * 2.0 ** -53
    us = [uniform(12345, c) for c in range(2000)]
    assert min(us) >= 0.0 and max(us) < 1.0 and abs(np.mean(us) - 0.5) < 0.02
    assert len(set(us)) == len(us)


def test_nucleus_decode_with_tiny_top_p_is_greedy():
    dims = synth.TINY
    w = {k: v.double().numpy() for k, v in synth.model_weights(dims, seed=0, dtype=torch.float32).items()}
    m = Backbone(dims, w.__getitem__)
    t = tree_buffers(synth.dense_tree_choices([2, 3]), 10)
    prompt = synth.prompt_tokens(0, 32, dims.vocab).numpy()
    ar = ar_greedy_decode(m, prompt, 12, 96)
    rs = RootSampler(NUCLEUS, 0.7, top_p=1e-9, key=7, counter=3)
    st = prefill(m, prompt, 96, 10, root=rs)
    out = []
    while len(out) < 12:
        toks, _ = verify_step(m, st, t, GREEDY, root=rs)
        out.extend(int(x) for x in toks)
    assert out[:12] == ar.tolist()
    assert [c for c, _, _ in rs.draws] == list(range(3, 3 + len(rs.draws)))
