"""Stochastic root of a verify step: typical and nucleus one-token sampling (oracle; test infrastructure only).

"大模型推理 memory bandwidth bound (5) - Medusa", 二.4 generate_candidates():
with temperature > 0 and without the "fast" flag the root token (the first
candidate) is drawn by get_typical_one_token(logits, T, eps, delta) or
get_nucleus_one_token(logits, T, top_p); 二.1 medusa_generate() gives the
defaults top_p = 0.8 and sampling = 'typical'. The pages name the two
functions and their arguments but do not print their bodies. Readings (the
plainest ones the rest of the pages support):

* typical one token: 一.3 explains typical acceptance as eta-sampling's allow
  set. The one-token sampler draws from p = softmax(z / T) restricted to that
  same set, {p > tau} with tau = min(eps, delta * exp(-H)) and
  H = -sum p log(p + 1e-5) (the quantities of the posterior), renormalised.
  By Jensen's inequality exp(-H) <= p_max + 1e-5, so the argmax is in the set
  whenever p_max > delta * 1e-5 / (1 - delta): for delta = 0.3, any
  vocabulary below 233,000 tokens. An empty set falls back to the argmax.
* nucleus one token (top-p, Holtzman et al., "The Curious Case of Neural Text
  Degeneration", 2020): tokens ordered by logit, largest first, equal logits
  by lower index first; a token is kept iff the probability mass of the
  tokens before it in that order is below top_p (the smallest leading set
  whose mass reaches top_p); renormalised.
* the draw: one uniform u in [0, 1) per root; the token is the first index k
  in vocabulary order whose cumulative kept probability exceeds u (the
  inverse of the kept distribution's CDF).
* u is word ``counter`` of the counter-based SplitMix64 stream of ``synth``
  under a 64-bit key, top 53 bits: u = (w >> 11) * 2**-53. A decode takes
  counter c0 for the prefill root and c0 + 1 + i for the root of step i.
* the verify step keeps the "fast" typical acceptance of 二.6 when the root is
  sampled: the non-fast mask get_typical_posterior_mask is not defined on the
  pages.
"""
from __future__ import annotations

import numpy as np

import synth

from .posterior import TYPICAL, node_stats

ARGMAX, TYPICAL_ONE, NUCLEUS = 0, 1, 2


def uniform(key: int, counter: int) -> float:
    """u in [0, 1) of the root drawn with ``counter`` under ``key`` (top 53 bits of the SplitMix64 word)."""
    w = int(synth.hash_words(key, counter, 1)[0]) % 2 ** 64
    return (w >> 11) * 2.0 ** -53


def softmax_t(z, temperature):
    """float64 p = softmax(z / T) of one logits row."""
    y = np.asarray(z, dtype=np.float64) / temperature
    e = np.exp(y - y.max())
    return e / e.sum()


def typical_allow(z, temperature, eps, delta):
    """Allow set {p > tau} of the typical one-token sampler, and ln p - ln tau per token."""
    st = node_stats(np.asarray(z, dtype=np.float64)[None, :], TYPICAL, temperature, eps, delta)
    p, tau = st["p"][0], st["tau"][0]
    with np.errstate(divide="ignore"):
        margin = np.log(p) - np.log(tau)
    return p > tau, margin


def nucleus_order(z):
    """Token order of the nucleus: logit descending, equal logits by ascending index."""
    z = np.asarray(z, dtype=np.float64)
    return np.lexsort((np.arange(len(z)), -z))


def nucleus_allow(z, temperature, top_p):
    """Allow set of the nucleus sampler and, per token, the mass of the tokens before it in the order."""
    p = softmax_t(z, temperature)
    order = nucleus_order(z)
    before_sorted = np.concatenate([[0.0], np.cumsum(p[order])[:-1]])
    before = np.empty_like(before_sorted)
    before[order] = before_sorted
    return before < top_p, before


def inverse_cdf(p, allow, u):
    """First index k (vocabulary order) whose cumulative renormalised kept probability exceeds u."""
    q = np.where(allow, np.asarray(p, dtype=np.float64), 0.0)
    tot = q.sum()
    if not tot > 0.0:
        return int(np.argmax(p))
    c = np.cumsum(q / tot)
    k = int(np.searchsorted(c, u, side="right"))
    if k >= len(c):                      # u beyond the last rounded cumulative: the last kept token
        k = int(np.flatnonzero(allow)[-1])
    return k


def sample_root(z, mode, temperature=0.7, eps=0.09, delta=0.3, top_p=0.8, u=0.0):
    """The root token drawn from logits row z (mode ARGMAX, TYPICAL_ONE or NUCLEUS) with uniform u."""
    z = np.asarray(z, dtype=np.float64)
    if mode == ARGMAX:
        return int(np.argmax(z))
    p = softmax_t(z, temperature)
    if mode == TYPICAL_ONE:
        allow, _ = typical_allow(z, temperature, eps, delta)
    elif mode == NUCLEUS:
        allow, _ = nucleus_allow(z, temperature, top_p)
    else:
        raise ValueError(f"unknown root mode {mode}")
    if not allow.any():
        return int(np.argmax(z))
    return inverse_cdf(p, allow, u)


class RootSampler:
    """Draws successive roots of a decode: counter c0 first, then c0 + 1, ... (see the module readings)."""

    def __init__(self, mode, temperature=0.7, eps=0.09, delta=0.3, top_p=0.8, key=0, counter=0):
        self.mode, self.temperature, self.eps, self.delta, self.top_p = mode, temperature, eps, delta, top_p
        self.key, self.counter = key, counter
        self.draws = []                  # (counter, u, token) of every draw

    def __call__(self, z):
        u = uniform(self.key, self.counter)
        tok = sample_root(z, self.mode, self.temperature, self.eps, self.delta, self.top_p, u)
        self.draws.append((self.counter, u, tok))
        self.counter += 1
        return tok
