"""GPU parity of the tcgen05 projection kernel and of the whole verify step, against the oracle.

The tiny decoder (d=64, 4 heads x 16, FFN 128, vocabulary 512, 2 layers, 2 Medusa heads, weights N(0, 0.02)
seed 0, rounded to bf16 for both sides) runs the dense head1 top-2 x head2 top-3 tree after a random 32-token
prompt. Token streams must match the oracle exactly except after a position where the oracle's own top-2
margin is below the bf16 tolerance; every GPU token is also checked by teacher forcing
("大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate(); greedy output identical to the base
model: "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 2️⃣).
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch

import decision_check
import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import (ar_greedy_decode, chain_mask, prefill as o_prefill, teacher_forced_logits,
                           verify_step as o_verify_step)
from oracle.model import Backbone, KVCache, medusa_heads, topk_ids
from oracle.posterior import GREEDY, TYPICAL
from oracle.tree import tree_buffers

pytestmark = pytest.mark.gpu
RTOL, ATOL, MARGIN = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    yield
    st, code = mv.get_error()
    assert st == 0, f"device error word set: {code:#x}"


# --------------------------------------------------------------------------------------------- projection kernel

@pytest.mark.parametrize("packed", [False, True])
@pytest.mark.parametrize("M,K,n", [(128, 64, 64), (300, 72, 9), (256, 4096, 64), (4096, 4096, 64),
                                   (12288, 4096, 1), (4096, 11008, 64), (32000, 4096, 64), (200, 8, 3),
                                   (300, 72, 65), (4096, 4096, 128), (4096, 11008, 130), (32000, 4096, 256),
                                   (200, 8, 255)])
def test_linear_bf16_vs_float64(M, K, n, packed):
    w = synth.normal(1, "w", (M, K), 1.0, dtype=torch.bfloat16, device="cuda")
    x = synth.normal(2, "x", (n, K), 1.0, dtype=torch.bfloat16, device="cuda")
    ld = M + 4
    out = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(mv.linear_bf16_workspace(), dtype=torch.uint8, device="cuda")
    if packed:
        wp = mv.pack_weight(w, 128)
        run = lambda: mv.linear_bf16_packed(wp, M, K, x, out, ws)
    else:
        run = lambda: mv.linear_bf16(w, x, out, ws)
    run()
    run()  # twice: the stream-K tickets must be back at zero
    got = out[:, :M].double().cpu().numpy()
    ref = x.double().cpu().numpy() @ w.double().cpu().numpy().T
    assert np.allclose(got, ref, rtol=1e-4, atol=1e-4 * math.sqrt(K))
    assert torch.isnan(out[:, M:]).all()          # nothing written past M


# --------------------------------------------------------------------------------------------- tiny decoder

DIMS = synth.TINY
S_MAX = 256


def _setup(tree_choices, topk=10, packed=True, dims=DIMS):
    w = synth.packed_weights(dims, 0, torch.bfloat16, "cuda")
    model = mv.Model(dims, mv.pack_model_weights(w) if packed else w)
    tree = mv.Tree(tree_choices, topk)
    sess = mv.Session(model, tree, S_MAX)
    om = Backbone(dims, synth.unpacked_getter(dims, w))
    return w, model, tree, sess, om, tree_buffers(tree_choices, topk)


def _prompt(n=32):
    return synth.prompt_tokens(0, n, DIMS.vocab)


def _check_topk_rows(gpu, z, k):
    for head in range(z.shape[0]):
        ref = topk_ids(z[head], k)
        for r in range(k):
            gi, ri = int(gpu[head, r]), int(ref[r])
            assert gi == ri or abs(z[head, gi] - z[head, ri]) < MARGIN, (head, r, gi, ri)


def test_prefill_matches_oracle():
    _, _, tree, sess, om, ot = _setup(synth.dense_tree_choices([2, 3]))
    p = _prompt()
    P = len(p)
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    st = o_prefill(om, p.numpy(), S_MAX, 10)
    assert int(sess.cur_len.item()) == P
    kv = sess.kv[:, :, :, :P].double().cpu().numpy()
    assert np.allclose(kv, st.cache.data[:, :, :, :P], rtol=RTOL, atol=ATOL)
    hs, lg = om.forward(p.numpy(), np.arange(P), KVCache(DIMS, S_MAX), 0, chain_mask(P))
    got = sess.logits[P - 1].double().cpu().numpy()        # one chunk of 32: its last row
    assert np.allclose(got, lg[-1], rtol=RTOL, atol=ATOL)
    root = sess.read_result()["next_root"]
    assert root == st.root or lg[-1].max() - lg[-1][root] < MARGIN
    _check_topk_rows(sess.head_topk.cpu().numpy(), medusa_heads(om.get, DIMS.n_medusa, hs[-1]), 10)


def test_three_heads_step_matches_oracle():
    """A decoder with 3 heads of 16 (48 q rows, not a power of two): the QKV epilogue takes a row's part, head and
    dimension by division instead of shifts. Prefill and one greedy verify step against the oracle, every node's
    logits and the prefill's cache rows element by element."""
    dims = dataclasses.replace(DIMS, n_heads=3)
    _, _, tree, sess, om, ot = _setup(synth.dense_tree_choices([2, 3]), dims=dims)
    p = synth.prompt_tokens(0, 32, dims.vocab)
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p.numpy(), S_MAX, 10)
    P = len(p)
    kv = sess.kv[:, :, :, :P].double().cpu().numpy()
    assert np.allclose(kv, st.cache.data[:, :, :, :P], rtol=RTOL, atol=ATOL)
    sess.step(mv.AcceptParams(GREEDY))
    torch.cuda.synchronize()
    _, info = o_verify_step(om, st, ot, GREEDY)
    got = sess.logits[:tree.n_nodes].double().cpu().numpy()
    assert np.allclose(got, info["logits"], rtol=RTOL, atol=ATOL)


@pytest.mark.parametrize("wide", [False, True])
def test_one_step_internals(wide):
    """One verify step against the oracle: candidates, every node's logits, the accepted path, the compacted
    cache and the next top-k. wide: a 200-node tree (four token groups, four query blocks, four mask words)."""
    choices, topk = (synth.synthetic_tree_choices(200, 2, 16), 16) if wide else (synth.dense_tree_choices([2, 3]), 10)
    _, _, tree, sess, om, ot = _setup(choices, topk=topk)
    p = _prompt()
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p.numpy(), S_MAX, topk)
    sess.step(mv.AcceptParams(GREEDY))
    torch.cuda.synchronize()
    toks, info = o_verify_step(om, st, ot, GREEDY)
    assert sess.tree_tokens.cpu().tolist() == info["tree_tokens"].tolist()
    assert sess.cart.cpu().tolist() == info["cart"].tolist()
    n = tree.n_nodes
    got = sess.logits[:n].double().cpu().numpy()
    assert np.allclose(got, info["logits"], rtol=RTOL, atol=ATOL)
    res, post = sess.read_result(), info["post"]
    # each retrieve row's first decision that differs from the oracle's must have an oracle margin below MARGIN
    dv = decision_check.check(res, decision_check.decisions_from_logits(got, sess.tree_tokens.cpu().numpy(), GREEDY),
                              post, ot["retrieve"], GREEDY)
    if not dv:
        L = st.cur_len
        assert int(sess.cur_len.item()) == L
        kv = sess.kv[:, :, :, :L].double().cpu().numpy()
        assert np.allclose(kv, st.cache.data[:, :, :, :L], rtol=RTOL, atol=ATOL)
        _check_topk_rows(sess.head_topk.cpu().numpy(), info["head_logits"], topk)
        assert res["next_root"] == st.root


def _gpu_decode(sess, prompt, n_new, params, force=None):
    sess.prefill(torch.as_tensor(prompt, dtype=torch.int32, device="cuda"))
    out, accs = [], []
    while len(out) < n_new:
        if force is not None:
            k = len(out)
            sess.head_topk[:, 0] = torch.as_tensor(force[k + 1: k + 1 + DIMS.n_medusa], dtype=torch.int32,
                                                   device="cuda")
        sess.step(params)
        r = sess.read_result()
        out.extend(r["tokens"])
        accs.append(r["acc"])
    return np.asarray(out[:n_new]), accs


def _margin_ok(gen, prompt, om):
    """Teacher forcing: every generated token is the oracle's argmax or within the bf16 tolerance of it."""
    lg = teacher_forced_logits(om, prompt, gen, S_MAX)
    first_close = len(gen)
    for i, t in enumerate(gen):
        top = lg[i].max()
        assert top - lg[i, t] <= 1e-2 + 2e-2 * abs(top), (i, t, int(np.argmax(lg[i])))
        srt = np.sort(lg[i])
        if srt[-1] - srt[-2] < 1e-2 + 2e-2 * abs(top):
            first_close = min(first_close, i)
    return first_close


@pytest.mark.parametrize("tree,packed", [("dense", True), ("synthetic", True), ("dense", False), ("page", True),
                                         ("wide200", True)])
def test_greedy_decode_equals_ar(tree, packed):
    dims = DIMS
    topk = 10
    if tree == "dense":
        choices = synth.dense_tree_choices([2, 3])
    elif tree == "wide200":  # 200 nodes: four token groups in the projections, four query blocks in the attention
        choices, topk = synth.synthetic_tree_choices(200, 2, 16), 16
    elif tree == "synthetic":
        choices = synth.synthetic_tree_choices(64, 2, 10)
    else:  # the page's own 63-choice tree ("大模型推理 memory bandwidth bound (5) - Medusa", 二.2): depth 4, 4 heads
        with open(os.path.join(os.path.dirname(__file__), "golden", "page4_tree.json")) as f:
            choices = [tuple(c) for c in json.load(f)["medusa_choices"]]
        dims = dataclasses.replace(DIMS, n_medusa=4)
    _, _, _, sess, om, ot = _setup(choices, topk=topk, packed=packed, dims=dims)
    p = _prompt().numpy()
    gen, accs = _gpu_decode(sess, p, 16, mv.AcceptParams(GREEDY))
    first_close = _margin_ok(gen, p, om)
    ar = ar_greedy_decode(om, p, 16, S_MAX)
    assert gen[:first_close + 1].tolist() == ar[:first_close + 1].tolist()


def test_forced_acceptance_tiny():
    _, _, _, sess, om, ot = _setup(synth.dense_tree_choices([2, 3]))
    p = _prompt().numpy()
    ar = ar_greedy_decode(om, p, 40, S_MAX)
    gen, accs = _gpu_decode(sess, p, 30, mv.AcceptParams(GREEDY), force=ar)
    first_close = _margin_ok(gen, p, om)
    assert gen[:first_close + 1].tolist() == ar[:first_close + 1].tolist()
    n_ok = sum(1 for a in accs if a == 2)
    assert n_ok >= len(accs) - 1 if first_close >= 30 else n_ok >= 1


def test_typical_steps_match_oracle():
    _, _, tree, sess, om, ot = _setup(synth.dense_tree_choices([2, 3]))
    p = _prompt()
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p.numpy(), S_MAX, 10)
    prm = mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3)
    for _ in range(6):
        sess.step(prm)
        torch.cuda.synchronize()
        toks, info = o_verify_step(om, st, ot, TYPICAL, 0.7, 0.09, 0.3)
        res, post = sess.read_result(), info["post"]
        acc = decision_check.decisions_from_logits(sess.logits[: tree.n_nodes].cpu().numpy(),
                                                   sess.tree_tokens.cpu().numpy(), TYPICAL, 0.7, 0.09, 0.3)
        if decision_check.check(res, acc, post, ot["retrieve"], TYPICAL):
            return  # the streams legitimately diverge after a near-threshold decision
        assert res["tokens"] == toks.tolist()
        assert int(sess.cur_len.item()) == st.cur_len


@pytest.mark.parametrize("buffers", ["pinned", "pageable", "pinned_alternating"])
def test_host_step_api_matches_device_step(buffers):
    """Pinned buffers run the host step as a replayed graph (re-captured when the buffers change), pageable ones
    launch by launch; both decode as the device-buffer step does."""
    _, _, tree, sess, om, ot = _setup(synth.dense_tree_choices([2, 3]))
    p = torch.as_tensor(_prompt(), dtype=torch.int32, device="cuda")
    sess.prefill(p)
    k = DIMS.n_medusa * 10

    def bufs():
        t = [torch.zeros(1 + k, dtype=torch.int32), torch.zeros(mv.RESULT_INTS, dtype=torch.int32),
             torch.zeros(1 + k, dtype=torch.int32)]
        return [x.pin_memory() for x in t] if buffers != "pageable" else t

    sets = [bufs(), bufs()] if buffers == "pinned_alternating" else [bufs()]
    seeds = sets[0][0]
    seeds[0] = int(sess.read_result()["next_root"])
    seeds[1:] = sess.head_topk.reshape(-1).cpu()
    toks_host = []
    for i in range(4):
        seeds, out, seeds_next = sets[i % len(sets)]
        sess.step_host(mv.AcceptParams(GREEDY), seeds, out, seeds_next)
        toks_host += mv.result_dict(out)["tokens"]
        sets[(i + 1) % len(sets)][0].copy_(seeds_next)
    _, _, _, sess2, _, _ = _setup(synth.dense_tree_choices([2, 3]))
    sess2.prefill(p)
    toks_dev = []
    for _ in range(4):
        sess2.step(mv.AcceptParams(GREEDY))
        toks_dev += sess2.read_result()["tokens"]
    assert toks_host == toks_dev


@pytest.mark.parametrize("mode", [GREEDY, TYPICAL])
def test_multi_step_graph_equals_eager(mode):
    """Several steps in one CUDA graph (consecutive launches overlap under programmatic launch) give the same
    decode as eager steps, and as one-step graphs."""
    prm = mv.AcceptParams(mode, 0.7, 0.09, 0.3)
    p = torch.as_tensor(_prompt(), dtype=torch.int32, device="cuda")
    outs = []
    for how in ("eager", "graph3", "graph1"):
        _, _, _, sess, _, _ = _setup(synth.dense_tree_choices([2, 3]))
        sess.prefill(p)
        if how == "eager":
            for _ in range(6):
                sess.step(prm)
        elif how == "graph3":
            sess.steps_graph(3, prm)
            sess.steps_graph(3, prm)
        else:
            for _ in range(6):
                sess.steps_graph(1, prm)
        torch.cuda.synchronize()
        outs.append((sess.read_result(), int(sess.cur_len.item()), sess.head_topk.cpu().tolist(),
                     sess.kv[:, :, :, : int(sess.cur_len.item())].cpu()))
    for o in outs[1:]:
        assert o[0] == outs[0][0] and o[1] == outs[0][1] and o[2] == outs[0][2]
        assert torch.equal(o[3], outs[0][3])


@pytest.mark.parametrize("fused", [True, False])
def test_small64_decoder_attention_inside_the_chain(fused, monkeypatch):
    """A decoder with 64-wide heads (d 256, 4 heads, 2 layers): its projection chains run each layer's attention
    first (cluster q = head q) unless MV_FUSE_ATTN=0. One step's logits match the oracle, and greedy Medusa decoding
    equals the oracle's greedy AR stream, either way."""
    monkeypatch.setenv("MV_FUSE_ATTN", "1" if fused else "0")
    dims = synth.SMALL64
    choices = synth.synthetic_tree_choices(48, 2, 10)
    _, _, tree, sess, om, ot = _setup(choices, dims=dims)
    p = synth.prompt_tokens(3, 40, dims.vocab)
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p.numpy(), S_MAX, 10)
    # the oracle's root and head top-k as the step's candidates (the tiny random heads have near ties)
    sess.result[3] = int(st.root)
    sess.head_topk.copy_(torch.as_tensor(st.head_topk, dtype=torch.int32, device="cuda"))
    sess.step(mv.AcceptParams(GREEDY))
    torch.cuda.synchronize()
    toks, info = o_verify_step(om, st, ot, GREEDY)
    assert sess.tree_tokens[: tree.n_nodes].cpu().tolist() == info["tree_tokens"].tolist()
    got = sess.logits[: tree.n_nodes].double().cpu().numpy()
    assert np.allclose(got, info["logits"], rtol=RTOL, atol=ATOL)
    _, _, _, sess2, _, _ = _setup(choices, dims=dims)
    gen, _ = _gpu_decode(sess2, p.numpy(), 12, mv.AcceptParams(GREEDY))
    lg = teacher_forced_logits(om, p.numpy(), gen, S_MAX)
    ar = ar_greedy_decode(om, p.numpy(), 12, S_MAX)
    first_close = len(gen)
    for i, tk in enumerate(gen):
        top = lg[i].max()
        assert top - lg[i, tk] <= 1e-2 + 2e-2 * abs(top)
        srt = np.sort(lg[i])
        if srt[-1] - srt[-2] < 1e-2 + 2e-2 * abs(top):
            first_close = min(first_close, i)
    assert gen[:first_close + 1].tolist() == ar[:first_close + 1].tolist()


@pytest.mark.parametrize("wide", [False, True])
def test_gate_up_layouts_bit_identical(wide):
    """pack_model_weights puts a layer's gate and up matrices in one allocation, up right after gate, and the
    projection kernel then loads both halves of a k-block with one copy; gate and up packed into separate
    allocations take one copy per matrix. Both fill shared memory with the same bytes, so prefill and steps give
    bit-identical logits, cache and decode state (one token group, and several: a wide tree)."""
    w = synth.packed_weights(DIMS, 0, torch.bfloat16, "cuda")
    joint = mv.pack_model_weights(w)
    gu = joint["w_up"][0].data_ptr() - joint["w_gate"][0].data_ptr()
    assert gu == joint["w_gate"][0].numel() * 2  # up right after gate
    apart = dict(joint)
    apart["w_gate"] = [mv.pack_weight(t, 64) for t in w["w_gate"]]
    apart["w_up"] = [mv.pack_weight(t, 64) for t in w["w_up"]]
    choices, topk = (synth.synthetic_tree_choices(200, 2, 16), 16) if wide else (synth.dense_tree_choices([2, 3]), 10)
    prm = mv.AcceptParams(GREEDY)
    p = torch.as_tensor(_prompt(), dtype=torch.int32, device="cuda")
    outs = []
    for ws in (joint, apart):
        sess = mv.Session(mv.Model(DIMS, ws), mv.Tree(choices, topk), S_MAX)
        sess.prefill(p)
        for _ in range(3):
            sess.step(prm)
        torch.cuda.synchronize()
        n = int(sess.cur_len.item())
        outs.append((sess.read_result(), n, sess.head_topk.cpu(), sess.kv[:, :, :, :n].cpu(), sess.logits.cpu()))
    a, b = outs
    assert a[0] == b[0] and a[1] == b[1]
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])


def test_long_cache_session_runs_the_tcgen05_attention():
    """A session whose cache holds more than 4096 rows runs each layer's tree attention on the tcgen05 kernel as its
    own launch (its projection chains carry no attention), every step. One step's logits match the oracle, and
    greedy Medusa decoding emits exactly the library's own greedy stream of a root-only tree in a session of the
    same cache length (random heads: nothing beyond the root is accepted, every token is a root row's argmax)."""
    dims = synth.SMALL64
    w = synth.packed_weights(dims, 0, torch.bfloat16, "cuda")
    model = mv.Model(dims, mv.pack_model_weights(w))
    om = Backbone(dims, synth.unpacked_getter(dims, w))
    choices = synth.synthetic_tree_choices(48, 2, 10)
    tree = mv.Tree(choices, 10)
    s_long = 4200
    p = synth.prompt_tokens(3, 40, dims.vocab)
    sess = mv.Session(model, tree, s_long)
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p.numpy(), s_long, 10)
    sess.result[3] = int(st.root)
    sess.head_topk.copy_(torch.as_tensor(st.head_topk, dtype=torch.int32, device="cuda"))
    sess.step(mv.AcceptParams(GREEDY))
    torch.cuda.synchronize()
    toks, info = o_verify_step(om, st, tree_buffers(choices, 10), GREEDY)
    assert sess.tree_tokens[: tree.n_nodes].cpu().tolist() == info["tree_tokens"].tolist()
    got = sess.logits[: tree.n_nodes].double().cpu().numpy()
    assert np.allclose(got, info["logits"], rtol=RTOL, atol=ATOL)
    streams = []
    for t in (tree, mv.Tree([], 10)):
        s2 = mv.Session(model, t, s_long)
        gen, accs = _gpu_decode(s2, p.numpy(), 16, mv.AcceptParams(GREEDY))
        streams.append((gen.tolist(), accs))
    assert sum(streams[0][1]) == 0 and sum(streams[1][1]) == 0
    assert streams[0][0] == streams[1][0]
