"""Seeded synthetic inputs for the Medusa tree-verify workloads.

This module is the only code shared by the CPU oracle and the GPU path. It holds
none of the method's arithmetic: it draws random numbers, builds prompt tokens,
weight tensors and tree choice lists, and plants agreements into logits. Every
value is a pure function of (seed, tensor name, element index), so the same
tensor comes out of every call on every device.

Generator
---------
Counter-based: element ``i`` of the stream named ``name`` under ``seed`` is the
SplitMix64 output function (Steele, Lea and Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014) applied to
``key(seed, name) + (i + 1) * 0x9E3779B97F4A7C15`` modulo 2**64. Normal variates
use the Box-Muller transform (Box and Muller, "A Note on the Generation of
Random Normal Deviates", 1958) in float64 on two such words, cosine branch
only: ``z_i = sqrt(-2 ln u1) cos(2 pi u2)`` with ``u1`` in (0, 1] from word
``2i`` and ``u2`` in [0, 1) from word ``2i+1`` (top 53 bits each). The result
is rounded once to the requested dtype (round-to-nearest-even).

The integer part is exact on any device (int64 arithmetic wraps modulo 2**64
in PyTorch on CPU and CUDA; right shifts are made logical by masking).
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass

import torch

__all__ = [
    "GAMMA", "stream_key", "hash_words", "normal", "uniform01", "randint",
    "ModelDims", "TINY", "SMALL64", "LLAMA7B", "model_weights", "weight_names",
    "dense_tree_choices", "synthetic_tree_choices", "prompt_tokens",
    "planted_tokens_and_logits", "kv_cache", "packed_weights",
]

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _s64(u: int) -> int:
    """Unsigned 64-bit Python int -> the int64 with the same bits."""
    u &= MASK64
    return u - (1 << 64) if u >= (1 << 63) else u


def _mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, name: str) -> int:
    """64-bit key of the stream ``name`` under ``seed`` (FNV-1a of the name, mixed)."""
    h = 0xCBF29CE484222325
    for b in name.encode():
        h = ((h ^ b) * 0x100000001B3) & MASK64
    return _mix64_int(h ^ _mix64_int(seed & MASK64))


def _lsr(x: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> s) & ((1 << (64 - s)) - 1)


def hash_words(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Words ``start .. start+count-1`` of the stream with 64-bit ``key`` (int64 bit patterns)."""
    idx = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = idx * _s64(GAMMA) + _s64(key)
    z = (z ^ _lsr(z, 30)) * _s64(_M1)
    z = (z ^ _lsr(z, 27)) * _s64(_M2)
    return z ^ _lsr(z, 31)


_CHUNK = 1 << 24


def uniform01(key: int, count: int, device="cpu", open_low=False) -> torch.Tensor:
    """float64 uniforms from the top 53 bits of each word: [0,1), or (0,1] if ``open_low``."""
    w = hash_words(key, 0, count, device)
    u = _lsr(w, 11).to(torch.float64)
    if open_low:
        u = u + 1.0
    return u * (2.0 ** -53)


def normal(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0,
           dtype=torch.float32, device="cpu") -> torch.Tensor:
    """``shape`` normal variates N(mean, std^2) of stream ``name`` (see module doc)."""
    n = math.prod(shape)
    key = stream_key(seed, name)
    out = torch.empty(n, dtype=dtype, device=device)
    for c0 in range(0, n, _CHUNK):
        c = min(_CHUNK, n - c0)
        w = hash_words(key, 2 * c0, 2 * c, device).view(c, 2)
        u1 = (_lsr(w[:, 0], 11).to(torch.float64) + 1.0) * (2.0 ** -53)
        u2 = _lsr(w[:, 1], 11).to(torch.float64) * (2.0 ** -53)
        z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
        out[c0:c0 + c] = (z * std + mean).to(dtype)
    return out.view(*shape)


def randint(seed: int, name: str, count: int, low: int, high: int, device="cpu") -> torch.Tensor:
    """``count`` integers uniform on [low, high) (floor of a 53-bit uniform times the range)."""
    u = uniform01(stream_key(seed, name), count, device)
    return (low + torch.floor(u * (high - low))).to(torch.int64)


# --------------------------------------------------------------------------------------------
# model shapes and weights
# --------------------------------------------------------------------------------------------

@dataclass(frozen=True)
class ModelDims:
    """Shape of a Llama-style decoder with Medusa heads."""
    d: int            # hidden size
    n_layers: int
    n_heads: int      # attention heads (q heads == kv heads)
    head_dim: int
    ffn: int          # SiLU-gated FFN inner size
    vocab: int
    n_medusa: int     # Medusa heads
    std: float = 0.02  # every weight matrix and the embedding ~ N(0, std^2); norm gains are 1
    rope_theta: float = 10000.0
    norm_eps: float = 1e-5


# Tiny decoder: d=64, 4 heads x 16, FFN 128, vocab 512, 2 layers, 2 Medusa heads.
TINY = ModelDims(d=64, n_layers=2, n_heads=4, head_dim=16, ffn=128, vocab=512, n_medusa=2)
# Small decoder with 64-wide heads: d=256, 4 heads x 64, FFN 512, vocab 1024, 2 layers, 2 Medusa heads.
SMALL64 = ModelDims(d=256, n_layers=2, n_heads=4, head_dim=64, ffn=512, vocab=1024, n_medusa=2)
# Llama-7B shape: d=4096, 32 layers, 32 heads x 128, FFN 11008, vocab 32000, 4 Medusa heads.
LLAMA7B = ModelDims(d=4096, n_layers=32, n_heads=32, head_dim=128, ffn=11008, vocab=32000, n_medusa=4)


def weight_names(dims: ModelDims):
    """(name, shape) of every weight; matrices are [out, in] (row = output feature)."""
    d, f, v = dims.d, dims.ffn, dims.vocab
    qd = dims.n_heads * dims.head_dim
    out = [("embed", (v, d))]
    for l in range(dims.n_layers):
        out += [(f"layer{l}.wq", (qd, d)), (f"layer{l}.wk", (qd, d)), (f"layer{l}.wv", (qd, d)),
                (f"layer{l}.wo", (d, qd)), (f"layer{l}.w_gate", (f, d)), (f"layer{l}.w_up", (f, d)),
                (f"layer{l}.w_down", (d, f))]
    out += [("lm_head", (v, d))]
    for k in range(dims.n_medusa):
        out += [(f"medusa{k}.w1", (d, d)), (f"medusa{k}.w2", (v, d))]
    return out


def model_weights(dims: ModelDims, seed: int = 0, dtype=torch.float32, device="cpu", names=None):
    """Random-init weights ~N(0, std^2), rounded once to ``dtype``; dict name -> tensor."""
    sel = None if names is None else set(names)
    return {n: normal(seed, n, s, dims.std, dtype=dtype, device=device)
            for n, s in weight_names(dims) if sel is None or n in sel}


def packed_weights(dims: ModelDims, seed: int = 0, dtype=torch.bfloat16, device="cpu"):
    """The same weights as ``model_weights``, laid out for the verify library.

    wqkv[l] = rows of wq, then wk, then wv of layer l (one [3*H*D, d] matrix); medusa_w1 / medusa_w2 stack the
    heads ([K, d, d] / [K, V, d]). Pure layout: every value is the one ``model_weights`` draws.
    """
    d, qd, v, K = dims.d, dims.n_heads * dims.head_dim, dims.vocab, dims.n_medusa
    g = lambda name, shape: normal(seed, name, shape, dims.std, dtype=dtype, device=device)
    w = {"embed": g("embed", (v, d)), "lm_head": g("lm_head", (v, d)),
         "wqkv": [], "wo": [], "w_gate": [], "w_up": [], "w_down": []}
    for l in range(dims.n_layers):
        qkv = torch.empty(3 * qd, d, dtype=dtype, device=device)
        for i, c in enumerate("qkv"):
            qkv[i * qd:(i + 1) * qd] = g(f"layer{l}.w{c}", (qd, d))
        w["wqkv"].append(qkv)
        w["wo"].append(g(f"layer{l}.wo", (d, qd)))
        w["w_gate"].append(g(f"layer{l}.w_gate", (dims.ffn, d)))
        w["w_up"].append(g(f"layer{l}.w_up", (dims.ffn, d)))
        w["w_down"].append(g(f"layer{l}.w_down", (d, dims.ffn)))
    w1 = torch.empty(K, d, d, dtype=dtype, device=device)
    w2 = torch.empty(K, v, d, dtype=dtype, device=device)
    for k in range(K):
        w1[k] = g(f"medusa{k}.w1", (d, d))
        w2[k] = g(f"medusa{k}.w2", (v, d))
    w["medusa_w1"], w["medusa_w2"] = w1, w2
    return w


def unpacked_getter(dims: ModelDims, w):
    """name -> float64 numpy view of one logical weight of a ``packed_weights`` dict (for the oracle)."""
    qd = dims.n_heads * dims.head_dim
    cache = {}

    def get(name):
        if name in cache:
            return cache[name]
        if name.startswith("layer"):
            l, key = name[5:].split(".")
            l = int(l)
            if key in ("wq", "wk", "wv"):
                i = "qkv".index(key[1])
                t = w["wqkv"][l][i * qd:(i + 1) * qd]
            else:
                t = w[key][l]
        elif name.startswith("medusa"):
            k, key = name[6:].split(".")
            t = w["medusa_" + key][int(k)]
        else:
            t = w[name]
        a = t.double().cpu().numpy()
        if len(cache) > 64:
            cache.clear()
        cache[name] = a
        return a

    return get


def prompt_tokens(seed: int, n: int, vocab: int, name: str = "prompt", device="cpu") -> torch.Tensor:
    """A random prompt: ``n`` token ids uniform on [0, vocab)."""
    return randint(seed, name, n, 0, vocab, device)


def kv_cache(seed: int, shape, dtype=torch.bfloat16, device="cpu", name="kv") -> torch.Tensor:
    """A KV cache filled with N(0,1) values."""
    return normal(seed, name, shape, 1.0, dtype=dtype, device=device)


# --------------------------------------------------------------------------------------------
# tree choice lists (inputs: the structure of the static token tree)
# --------------------------------------------------------------------------------------------

def dense_tree_choices(widths):
    """Every rank tuple of the dense tree whose depth-k level takes the top ``widths[k-1]``.

    ``[2, 3]`` is the head1 top-2 x head2 top-3 tree (8 choices; 9 nodes with the root).
    """
    out = []
    for depth in range(1, len(widths) + 1):
        out += list(itertools.product(*[range(w) for w in widths[:depth]]))
    return out


def synthetic_tree_choices(n_nodes: int = 64, depth: int = 4, topk: int = 10):
    """The ``n_nodes - 1`` highest-scoring rank paths of a ``topk``-ary tree of ``depth`` levels.

    Path (r_1..r_D) scores prod_{d=1..D} 0.7**d * 0.5**r_d. Ties go to the
    lexicographically smaller tuple. The score is 0.7**a * 0.5**b with the
    integers a = D(D+1)/2 and b = sum(r); it is ordered by a*ln(0.7) + b*ln(0.5),
    which separates distinct (a, b) pairs far above float64 rounding.
    """
    paths = []
    for D in range(1, depth + 1):
        for t in itertools.product(range(topk), repeat=D):
            a, b = D * (D + 1) // 2, sum(t)
            paths.append((-(a * math.log(0.7) + b * math.log(0.5)), t))
    paths.sort()
    return [t for _, t in paths[: n_nodes - 1]]


# --------------------------------------------------------------------------------------------
# posterior workload: logits with planted agreements along a path
# --------------------------------------------------------------------------------------------

def planted_tokens_and_logits(seed: int, n_nodes: int, vocab: int, path, plant_len: int,
                              std: float = 3.0, bump: float = 2.0, device="cpu"):
    """Node tokens and fp32 logits [n_nodes, vocab] ~ N(0, std^2) with a planted agreement.

    ``path`` lists node indices root-first. For j < ``plant_len`` the logit of
    the token of ``path[j+1]`` in row ``path[j]`` is set to that row's maximum
    plus ``bump``, so it becomes the row's argmax. Node tokens are distinct
    draws from [0, vocab) (the root's token included).
    """
    logits = normal(seed, "posterior_logits", (n_nodes, vocab), std, dtype=torch.float32, device="cpu")
    perm = torch.argsort(uniform01(stream_key(seed, "node_tokens"), vocab))
    tokens = perm[:n_nodes].to(torch.int64)
    for j in range(plant_len):
        row, child = int(path[j]), int(path[j + 1])
        logits[row, tokens[child]] = logits[row].max() + bump
    return tokens.to(device), logits.to(device)
