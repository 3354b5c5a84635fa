"""Batch > 1 verify: several independent sequences in one session, one backbone pass per step for all of them.

The pages' code verifies one sequence at a time ("大模型推理 memory bandwidth bound (5) - Medusa", 二.1
medusa_generate(): batch size 1 only). Batching changes no sequence's result: each sequence of a batched
session must decode exactly as the oracle decodes it alone (greedy output identical to its own greedy
autoregressive stream, "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 2️⃣), up to the first position whose
oracle top-2 margin is below the bf16 tolerance; typical steps must match the oracle's single-sequence steps.
"""
import numpy as np
import pytest
import torch

import decision_check
import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import ar_greedy_decode, prefill as o_prefill, teacher_forced_logits, verify_step as o_verify_step
from oracle.model import Backbone
from oracle.posterior import GREEDY, TYPICAL
from oracle.tree import tree_buffers

pytestmark = pytest.mark.gpu
DIMS = synth.TINY
S_MAX = 256
MARGIN = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    yield
    st, code = mv.get_error()
    assert st == 0, f"device error word set: {code:#x}"


def _setup(B, choices, topk=10):
    w = synth.packed_weights(DIMS, 0, torch.bfloat16, "cuda")
    model = mv.Model(DIMS, mv.pack_model_weights(w))
    tree = mv.Tree(choices, topk)
    sess = mv.Session(model, tree, S_MAX, batch=B)
    om = Backbone(DIMS, synth.unpacked_getter(DIMS, w))
    return model, tree, sess, om, tree_buffers(choices, topk)


def _prompts(B, n=32):
    return [synth.prompt_tokens(100 + b, n + 3 * b, DIMS.vocab).numpy() for b in range(B)]  # different lengths


def _margin_first_close(gen, prompt, om):
    lg = teacher_forced_logits(om, prompt, gen, S_MAX)
    first_close = len(gen)
    for i, t in enumerate(gen):
        top = lg[i].max()
        assert top - lg[i, t] <= 1e-2 + 2e-2 * abs(top), (i, t, int(np.argmax(lg[i])))
        srt = np.sort(lg[i])
        if srt[-1] - srt[-2] < 1e-2 + 2e-2 * abs(top):
            first_close = min(first_close, i)
    return first_close


@pytest.mark.parametrize("B,tree", [(2, "dense"), (4, "dense"), (3, "synthetic")])
def test_batched_greedy_equals_each_sequence_ar(B, tree):
    choices = synth.dense_tree_choices([2, 3]) if tree == "dense" else synth.synthetic_tree_choices(64, 2, 10)
    _, _, sess, om, _ = _setup(B, choices)
    prompts = _prompts(B)
    for b, p in enumerate(prompts):
        sess.prefill_seq(b, torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    outs = [[] for _ in range(B)]
    while min(len(o) for o in outs) < 16:
        sess.step(mv.AcceptParams(GREEDY))
        for b in range(B):
            outs[b].extend(sess.read_result(b)["tokens"])
    for b in range(B):
        gen = np.asarray(outs[b][:16])
        first_close = _margin_first_close(gen, prompts[b], om)
        ar = ar_greedy_decode(om, prompts[b], 16, S_MAX)
        assert gen[:first_close + 1].tolist() == ar[:first_close + 1].tolist(), b
    lens = sess.cur_len.cpu().tolist()
    assert all(lens[b] >= len(prompts[b]) + 16 for b in range(B))


def test_batched_typical_steps_match_oracle():
    B = 3
    _, _, sess, om, ot = _setup(B, synth.dense_tree_choices([2, 3]))
    prompts = _prompts(B)
    states = []
    for b, p in enumerate(prompts):
        sess.prefill_seq(b, torch.as_tensor(p, dtype=torch.int32, device="cuda"))
        states.append(o_prefill(om, p, S_MAX, 10))
    prm = mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3)
    live = list(range(B))
    for _ in range(5):
        sess.step(prm)
        torch.cuda.synchronize()
        for b in list(live):
            toks, info = o_verify_step(om, states[b], ot, TYPICAL, 0.7, 0.09, 0.3)
            res, post = sess.read_result(b), info["post"]
            n = ot["n_nodes"]
            acc = decision_check.decisions_from_logits(sess.logits[64 * b: 64 * b + n].cpu().numpy(),
                                                       sess.tree_tokens[64 * b: 64 * b + n].cpu().numpy(),
                                                       TYPICAL, 0.7, 0.09, 0.3)
            if decision_check.check(res, acc, post, ot["retrieve"], TYPICAL):
                live.remove(b)  # this stream legitimately diverges after a near-threshold decision
                continue
            assert res["tokens"] == toks.tolist()
            assert int(sess.cur_len[b].item()) == states[b].cur_len
    assert live, "every sequence diverged at once"


def test_batched_graph_equals_eager_and_sampling_counters():
    B = 4
    prm = mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3)
    root = mv.RootParams(mv.ROOT_NUCLEUS, 0.7, top_p=0.8, key=9)
    outs = []
    for how in ("eager", "graph"):
        _, _, sess, _, _ = _setup(B, synth.dense_tree_choices([2, 3]))
        sess.set_root_sampling(root, 100)
        for b, p in enumerate(_prompts(B)):
            sess.prefill_seq(b, torch.as_tensor(p, dtype=torch.int32, device="cuda"))
        if how == "eager":
            for _ in range(4):
                sess.step(prm)
        else:
            sess.steps_graph(2, prm)
            sess.steps_graph(2, prm)
        torch.cuda.synchronize()
        outs.append(([sess.read_result(b) for b in range(B)], sess.cur_len.cpu().tolist(),
                     sess.head_topk.cpu().tolist(), sess.root_counter.cpu().tolist(), sess.kv.cpu()))
    assert outs[0][:4] == outs[1][:4]
    assert torch.equal(outs[0][4], outs[1][4])
    assert outs[0][3] == [100 + (b << 32) + 5 for b in range(B)]  # prefill + 4 steps per sequence


def test_batched_session_rejects_large_trees_and_single_sequence_calls():
    w = synth.packed_weights(DIMS, 0, torch.bfloat16, "cuda")
    model = mv.Model(DIMS, mv.pack_model_weights(w))
    big = mv.Tree(synth.synthetic_tree_choices(100, 2, 16), 16)
    with pytest.raises(mv.MVError):
        mv.Session(model, big, S_MAX, batch=2)
    with pytest.raises(mv.MVError):
        mv.Session(model, mv.Tree(synth.dense_tree_choices([2, 3]), 10), S_MAX, batch=5)
    sess = mv.Session(model, mv.Tree(synth.dense_tree_choices([2, 3]), 10), S_MAX, batch=2)
    with pytest.raises(mv.MVError):
        sess.prefill(torch.as_tensor(_prompts(1)[0], dtype=torch.int32, device="cuda"))


def test_batched_long_cache_runs_the_tcgen05_attention():
    """A batched session whose caches hold more than 4096 rows runs each layer's tree attention for all its
    sequences in one launch of the tcgen05 kernel (one query block and one set of cache planes per sequence, q
    copied by TMA from the sequence's 64 rows). Each sequence decodes as the oracle decodes it alone, up to its
    first position whose oracle top-2 margin is inside the bf16 tolerance."""
    dims, B, s_long, n_new = synth.SMALL64, 2, 4200, 8
    w = synth.packed_weights(dims, 0, torch.bfloat16, "cuda")
    model = mv.Model(dims, mv.pack_model_weights(w))
    om = Backbone(dims, synth.unpacked_getter(dims, w))
    sess = mv.Session(model, mv.Tree(synth.synthetic_tree_choices(48, 2, 10), 10), s_long, batch=B)
    prompts = [synth.prompt_tokens(200 + b, 24 + 5 * b, dims.vocab).numpy() for b in range(B)]
    for b, p in enumerate(prompts):
        sess.prefill_seq(b, torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    outs = [[] for _ in range(B)]
    while min(len(o) for o in outs) < n_new:
        sess.step(mv.AcceptParams(GREEDY))
        for b in range(B):
            outs[b].extend(sess.read_result(b)["tokens"])
    for b in range(B):
        gen = np.asarray(outs[b][:n_new])
        lg = teacher_forced_logits(om, prompts[b], gen, S_MAX)
        first_close = len(gen)
        for i, t in enumerate(gen):
            top = lg[i].max()
            assert top - lg[i, t] <= 1e-2 + 2e-2 * abs(top), (b, i, t, int(np.argmax(lg[i])))
            srt = np.sort(lg[i])
            if srt[-1] - srt[-2] < 1e-2 + 2e-2 * abs(top):
                first_close = min(first_close, i)
        ar = ar_greedy_decode(om, prompts[b], n_new, S_MAX)
        assert gen[:first_close + 1].tolist() == ar[:first_close + 1].tolist(), b
