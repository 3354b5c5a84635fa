"""Pins of the oracle's decode loop (CPU).

* Greedy Medusa decoding is token-identical to plain greedy autoregressive
  decoding of the same model ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu",
  2️⃣; "大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate()).
  Checked on the tiny 2-layer decoder with the dense 1 x 2 x 3 tree, 16 steps.
* Forced acceptance: with the head top-k replaced by the true greedy
  continuation at rank 0, every step accepts the whole depth; compaction and
  multi-token acceptance must still reproduce the autoregressive stream.
"""
import numpy as np

import synth
from oracle.decode import ar_greedy_decode, generate_candidates, medusa_greedy_decode, prefill, verify_step
from oracle.model import Backbone
from oracle.tree import tree_buffers


def _tiny(dtype="fp32"):
    dims = synth.TINY
    import torch
    dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    w = {k: v.double().numpy() for k, v in synth.model_weights(dims, seed=0, dtype=dt).items()}
    return dims, Backbone(dims, w.__getitem__)


def test_generate_candidates_dense():
    t = tree_buffers(synth.dense_tree_choices([2, 3]), 10)
    topk = np.array([[100 + r for r in range(10)], [200 + r for r in range(10)]])
    tt, cart = generate_candidates(7, topk, t)
    assert tt.tolist() == [7, 100, 101, 200, 201, 202, 200, 201, 202]
    assert {tuple(r) for r in cart.tolist()} == {(7, 100 + a, 200 + b) for a in range(2) for b in range(3)}


def test_greedy_equivalence_tiny():
    dims, m = _tiny()
    t = tree_buffers(synth.dense_tree_choices([2, 3]), 10)
    prompt = synth.prompt_tokens(0, 32, dims.vocab).numpy()
    ar = ar_greedy_decode(m, prompt, 16, 96)
    md, accs = medusa_greedy_decode(m, prompt, 16, t, 96)
    assert md.tolist() == ar.tolist()


def test_forced_acceptance_reproduces_ar():
    dims, m = _tiny()
    t = tree_buffers(synth.dense_tree_choices([2, 3]), 10)
    prompt = synth.prompt_tokens(0, 32, dims.vocab).numpy()
    ar = ar_greedy_decode(m, prompt, 24, 128)
    st = prefill(m, prompt, 128, 10)
    out = []
    while len(out) < 18:
        k = len(out)
        # rank 0 of head j := the true token at offset j+1 after the root
        st.head_topk[:, 0] = ar[k + 1: k + 1 + dims.n_medusa]
        assert st.root == ar[k]
        toks, info = verify_step(m, st, t)
        assert info["post"]["acc"] == t["depth"]
        out.extend(toks.tolist())
    assert out == ar[: len(out)].tolist()
