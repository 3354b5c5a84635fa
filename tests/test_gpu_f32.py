"""The fp32 model path on the small correctness configuration, and the library's weight generator (GPU).

Tiny decoder in fp32: d=64, 4 heads x 16, FFN 128, vocabulary 512, 2 layers, 2 Medusa heads, every weight
N(0, 0.02) seed 0 rounded once to fp32; the dense head-1 top-2 x head-2 top-3 tree (9 nodes, 6 paths); a random
32-token prompt; greedy acceptance; 16 verify steps. In fp32 the path must reproduce the float64 oracle step by
step -- every node's logits within 2e-2 relative / 1e-2 absolute (in practice about 1e-6), the same accepted
paths, the same head top-k -- and its emitted stream must be the oracle's plain greedy autoregressive stream token
for token ("大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate(), 二.5 tree_decoding();
greedy output identical to the base model: "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 2️⃣).
"""
import numpy as np
import pytest
import torch

import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import ar_greedy_decode, chain_mask, prefill as o_prefill, verify_step as o_verify_step
from oracle.model import Backbone, KVCache, medusa_heads, topk_ids
from oracle.posterior import GREEDY
from oracle.tree import tree_buffers

pytestmark = pytest.mark.gpu
DIMS = synth.TINY
S_MAX = 256
RTOL, ATOL = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    yield
    st, code = mv.get_error()
    assert st == 0, f"device error word set: {code:#x}"


def _model(kind):
    w = synth.packed_weights(DIMS, 0, torch.float32, "cuda")  # the oracle's weights (and the caller's)
    model = mv.Model(DIMS, w) if kind == "caller" else mv.Model.random(DIMS, 0, DIMS.std, mv.DTYPE_F32)
    assert model.dtype == mv.DTYPE_F32
    return w, model


def _same_topk(sess, z, k=10, tol=1e-5):
    """The session's head top-k equals the oracle's top-k of head logits z [K, V], except at a near tie (two
    values within tol, far below what fp32 arithmetic could be expected to separate); then the oracle's rows are
    copied into the session so that both sides go on from the same candidates."""
    gpu = sess.head_topk.cpu().numpy()
    ref = np.stack([topk_ids(z[h], k) for h in range(z.shape[0])])
    if (gpu == ref).all():
        return True
    for h, r in zip(*np.nonzero(gpu != ref)):
        assert abs(z[h, gpu[h, r]] - z[h, ref[h, r]]) < tol, (h, r, gpu[h, r], ref[h, r])
    sess.head_topk.copy_(torch.as_tensor(ref, dtype=torch.int32, device="cuda"))
    return False


def _decode(sess, prompt, n_steps, force=None):
    sess.prefill(torch.as_tensor(prompt, dtype=torch.int32, device="cuda"))
    out = []
    for _ in range(n_steps):
        if force is not None:
            k = len(out)
            sess.head_topk[:, 0] = torch.as_tensor(force[k + 1: k + 1 + DIMS.n_medusa], dtype=torch.int32,
                                                   device="cuda")
        sess.step(mv.AcceptParams(mv.GREEDY))
        out.extend(sess.read_result()["tokens"])
    return np.asarray(out)


@pytest.mark.parametrize("kind", ["caller", "random"])
def test_f32_tiny_steps_match_oracle(kind):
    """16 verify steps against the oracle's, step by step: logits of every node, accepted path, emitted tokens,
    cache length and head top-k."""
    w, model = _model(kind)
    choices = synth.dense_tree_choices([2, 3])
    tree, ot = mv.Tree(choices, 10), tree_buffers(choices, 10)
    sess = mv.Session(model, tree, S_MAX)
    om = Backbone(DIMS, synth.unpacked_getter(DIMS, w))
    p = synth.prompt_tokens(0, 32, DIMS.vocab).numpy()
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    st = o_prefill(om, p, S_MAX, 10)
    assert sess.read_result()["next_root"] == st.root
    h, _ = om.forward(p, np.arange(len(p)), KVCache(DIMS, S_MAX), 0, chain_mask(len(p)))
    _same_topk(sess, medusa_heads(om.get, DIMS.n_medusa, h[-1]))
    worst, gen = 0.0, []
    for _ in range(16):
        sess.step(mv.AcceptParams(mv.GREEDY))
        toks, info = o_verify_step(om, st, ot, GREEDY)
        got = sess.logits[: tree.n_nodes].double().cpu().numpy()
        assert np.allclose(got, info["logits"], rtol=RTOL, atol=ATOL)
        worst = max(worst, float(np.abs(got - info["logits"]).max()))
        r = sess.read_result()
        assert r["nodes"] == info["post"]["nodes"].tolist() and r["tokens"] == toks.tolist()
        assert int(sess.cur_len.item()) == st.cur_len
        assert r["next_root"] == st.root
        _same_topk(sess, info["head_logits"])
        gen += r["tokens"]
    print(f"fp32 tiny decoder ({kind} weights): 16 steps, {len(gen)} tokens, largest |logit - oracle| {worst:.3g}")
    assert worst < 1e-4
    assert gen == ar_greedy_decode(om, p, len(gen), S_MAX).tolist()


def test_f32_tiny_forced_acceptance_equals_oracle_ar():
    """Candidates forced to the greedy continuation: every step accepts the whole depth (2) and the stream is the
    oracle's plain greedy stream, token for token."""
    w, model = _model("caller")
    tree = mv.Tree(synth.dense_tree_choices([2, 3]), 10)
    sess = mv.Session(model, tree, S_MAX)
    om = Backbone(DIMS, synth.unpacked_getter(DIMS, w))
    p = synth.prompt_tokens(0, 32, DIMS.vocab).numpy()
    ar = ar_greedy_decode(om, p, 16 * 3 + 4, S_MAX)
    gen = _decode(sess, p, 16, force=ar)
    assert len(gen) == 16 * 3
    assert gen.tolist() == ar[: len(gen)].tolist()


def test_f32_graph_replay_equals_eager_and_host_step():
    _, model = _model("caller")
    tree = mv.Tree(synth.dense_tree_choices([2, 3]), 10)
    p = torch.as_tensor(synth.prompt_tokens(0, 32, DIMS.vocab), dtype=torch.int32, device="cuda")
    a, b = mv.Session(model, tree, S_MAX), mv.Session(model, tree, S_MAX)
    for s in (a, b):
        s.prefill(p)
    for _ in range(6):
        a.step(mv.AcceptParams(mv.GREEDY))
    b.steps_graph(3, mv.AcceptParams(mv.GREEDY))
    b.steps_graph(3, mv.AcceptParams(mv.GREEDY))
    torch.cuda.synchronize()
    assert a.read_result() == b.read_result()
    assert torch.equal(a.kv, b.kv) and torch.equal(a.head_topk, b.head_topk)
    assert int(a.cur_len.item()) == int(b.cur_len.item())


def test_f32_session_rejects_batches():
    _, model = _model("caller")
    with pytest.raises(mv.MVError) as e:
        mv.Session(model, mv.Tree(synth.dense_tree_choices([2, 3]), 10), S_MAX, batch=2)
    assert e.value.status == 7  # MV_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("name,count,std", [("embed", 32768, 0.02), ("layer3.w_down", 1000, 0.02),
                                            ("q", 4097, 1.0), ("medusa1.w2", 1, 0.02)])
def test_fill_normal_equals_synth(dtype, name, count, std):
    """The library's generator is the input generator the oracle side uses: bit for bit."""
    out = torch.full((count,), float("nan"), dtype=dtype, device="cuda")
    mv.fill_normal(out, 7, name, std)
    ref = synth.normal(7, name, (count,), std, dtype=dtype, device="cuda")
    assert torch.equal(out.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       ref.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))


def test_random_bf16_model_equals_synth_weights():
    """A bf16 model the library draws (projections generated straight into the packed layout) computes exactly
    what the model built from synth's weights computes: the same logits, bit for bit, and the same stream."""
    dims = synth.SMALL64
    tree = mv.Tree(synth.synthetic_tree_choices(48, 2, 10), 10)
    p = torch.as_tensor(synth.prompt_tokens(3, 40, dims.vocab), dtype=torch.int32, device="cuda")
    runs = []
    for kind in ("synth", "library"):
        if kind == "synth":
            model = mv.Model(dims, mv.pack_model_weights(synth.packed_weights(dims, 0, torch.bfloat16, "cuda")))
        else:
            model = mv.Model.random(dims, 0, dims.std, mv.DTYPE_BF16)
        sess = mv.Session(model, tree, 256)
        sess.prefill(p)
        toks = []
        for _ in range(4):
            sess.step(mv.AcceptParams(mv.GREEDY))
            toks += sess.read_result()["tokens"]
        runs.append((toks, sess.logits[: tree.n_nodes].clone(), sess.head_topk.clone()))
    assert runs[0][0] == runs[1][0]
    assert torch.equal(runs[0][1], runs[1][1]) and torch.equal(runs[0][2], runs[1][2])
