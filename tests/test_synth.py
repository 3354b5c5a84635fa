"""The seeded input generator against its published definition (CPU)."""
import math

import torch

import synth


def _splitmix_ref(key, i):
    """SplitMix64 (Steele, Lea and Flood 2014) output for counter i, in Python integers."""
    z = (key + (i + 1) * 0x9E3779B97F4A7C15) % 2 ** 64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) % 2 ** 64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) % 2 ** 64
    return z ^ (z >> 31)


def test_hash_words_match_definition():
    key = synth.stream_key(0, "x")
    w = synth.hash_words(key, 5, 40)
    for j in range(40):
        assert int(w[j]) % 2 ** 64 == _splitmix_ref(key, 5 + j)
    # the published first output of SplitMix64 seeded with 0 is 0xE220A8397B1DCDAF
    assert int(synth.hash_words(0, 0, 1)[0]) % 2 ** 64 == 0xE220A8397B1DCDAF


def test_normal_moments_and_determinism():
    a = synth.normal(0, "w", (1 << 16,), std=0.02)
    b = synth.normal(0, "w", (1 << 16,), std=0.02)
    assert torch.equal(a, b)
    assert abs(a.mean().item()) < 3 * 0.02 / math.sqrt(a.numel())
    assert abs(a.std().item() / 0.02 - 1) < 0.02
    assert not torch.equal(a, synth.normal(1, "w", (1 << 16,), std=0.02))


def test_randint_range():
    r = synth.randint(0, "p", 10000, 0, 512)
    assert r.min() >= 0 and r.max() < 512 and len(set(r.tolist())) > 400
