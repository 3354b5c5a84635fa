"""Full-size parity of the verify loop at Llama-7B shape (32 layers, d 4096, 32 x 128 heads, FFN 11008,
vocabulary 32000, 4 Medusa heads, the synthetic 64-node tree, a random 128-token prompt), in the launch
configuration bench.py times (packed weights, CUDA-graph replay of the steps).

Two kinds of check ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 2️⃣: greedy Medusa output equals the
base model's; "大模型推理 memory bandwidth bound (5) - Medusa", 二.1 medusa_generate(), 二.5 tree_decoding()):
* the library's greedy Medusa stream equals plain greedy decoding of the same bf16 model in the same library (a
  session whose tree is the root alone verifies nothing and emits the argmax of each position's logits), token
  for token, at 64 and at 512 new tokens, also with the heads' candidates forced to the right continuation so
  that every step accepts the full depth. No tolerance enters: a tree node's logits are computed with exactly
  the arithmetic of the same token decoded alone at the same position;
* the float64 oracle, which cannot decode 7B tokens one by one in reasonable time, checks the bf16 arithmetic
  itself by teacher forcing (one causal oracle forward over prompt + the 64 GPU tokens) and on the first verify
  step's logits at sampled tree nodes, against the bound stated once below (STORE_BOUND_FACTOR).
"""
import numpy as np
import pytest
import torch

import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import chain_mask
from oracle.model import Backbone, KVCache
from oracle.tree import tree_buffers

pytestmark = pytest.mark.gpu
DIMS = synth.LLAMA7B
P, N_NEW = 128, 64

# The bound of the oracle checks at full depth, in one place. The GPU path stores q, k, v (the cache), the
# attention output, the SiLU-gate product and the normalised projection operands in bf16. That storage alone
# (the oracle's own float64 arithmetic with exactly those intermediates rounded to bf16: Backbone(store=...))
# moves the 7B-shape logits by a few percent and changes about one argmax in ten of these random-model rows, so
# no bf16 path meets 2e-2 / 1e-2 per element or token-exact teacher forcing at full depth. The GPU may differ
# from the float64 oracle by at most STORE_BOUND_FACTOR times what the storage format alone causes, measured in
# the same test: normwise and per element (relative to the row RMS) on the logits, and on each teacher-forced
# token's margin (oracle top-1 minus the GPU token's logit), which must also stay within the larger of that and
# the per-element 1e-2 + 2e-2 |top-1|.
STORE_BOUND_FACTOR = 2.0


@pytest.fixture(scope="module")
def model7b():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = synth.packed_weights(DIMS, 0, torch.bfloat16, "cuda")
    wp = mv.pack_model_weights(w)
    return w, mv.Model(DIMS, wp)


def test_7b_greedy_stream_teacher_forced(model7b):
    w, model = model7b
    choices = synth.synthetic_tree_choices(64, 4, 10)
    tree = mv.Tree(choices, 10)
    sess = mv.Session(model, tree, 1024)
    prompt = synth.prompt_tokens(0, P, DIMS.vocab)
    sess.prefill(torch.as_tensor(prompt, dtype=torch.int32, device="cuda"))
    gen, first_logits = [], None
    while len(gen) < N_NEW:
        if first_logits is None:
            sess.step(mv.AcceptParams(mv.GREEDY))
            first_logits = sess.logits[: tree.n_nodes].double().cpu().numpy()
            first_tree_tokens = sess.tree_tokens.cpu().numpy().copy()
        else:
            sess.steps_graph(1, mv.AcceptParams(mv.GREEDY))
        gen += sess.read_result()["tokens"]
    gen = np.asarray(gen[:N_NEW])

    cache = {}

    def get(name):  # every logical weight converted once to float64 (about 63 GB of host memory)
        if name not in cache:
            cache[name] = synth.unpacked_getter(DIMS, w)(name)
        return cache[name]

    om = Backbone(DIMS, get)
    o = tree_buffers(choices, 10)
    kv = KVCache(DIMS, P + 64 + N_NEW)
    _, lg_prompt = om.forward(prompt.numpy(), np.arange(P), kv, 0, chain_mask(P))
    kv_tree = KVCache(DIMS, P + 64 + N_NEW, kv.data)
    _, tl = om.forward(first_tree_tokens, P + o["position_ids"], kv_tree, P, o["attn_mask"])
    _, lg_gen = om.forward(gen, P + np.arange(N_NEW), kv, P, chain_mask(N_NEW))
    bf16 = lambda name, v: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16).double().numpy()
    ob = Backbone(DIMS, get, bf16)  # the same oracle with bf16 storage of the intermediates
    kv_b = KVCache(DIMS, P + 64)
    ob.forward(prompt.numpy(), np.arange(P), kv_b, 0, chain_mask(P))
    _, tl_store = ob.forward(first_tree_tokens, P + o["position_ids"], kv_b, P, o["attn_mask"])
    # 1) teacher forcing: the logits that predict gen[i] are the prompt's last row (i = 0) or gen[i-1]'s row.
    # a GPU token is the oracle argmax, or its oracle margin (top-1 minus its logit) is within the bound above
    lg = np.concatenate([lg_prompt[-1:], lg_gen[:-1]])
    margins = lg.max(axis=1) - lg[np.arange(N_NEW), gen]
    d_store = np.abs(tl_store - tl).max()
    print(f"7B teacher forcing: {int((margins > 0).sum())} of {N_NEW} tokens differ from the oracle argmax, "
          f"largest margin {margins.max():.4f}, exact-match prefix {int(np.argmax(margins > 0)) if (margins > 0).any() else N_NEW}; "
          f"bf16 storage alone moves a tree-row logit by up to {d_store:.4f} and keeps "
          f"{float((tl_store.argmax(1) == tl.argmax(1)).mean()):.3f} of the argmaxes")
    for i, t in enumerate(gen):
        top = lg[i].max()
        bound = max(1e-2 + 2e-2 * abs(top), STORE_BOUND_FACTOR * d_store)
        assert top - lg[i, t] <= bound, (i, int(t), int(np.argmax(lg[i])), top - lg[i, t], bound)
    # 2) the first step's LM logits on sampled tree nodes against the oracle's tree forward at prefix P, within
    # STORE_BOUND_FACTOR times the storage-only movement (normwise and per element relative to the row RMS)
    rows = [0, 1, 7, 30, 63]
    ref = tl[rows]
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))

    def err(x):
        return np.linalg.norm(x - ref) / np.linalg.norm(ref), (np.abs(x - ref) / rms).max()

    rel, peak = err(first_logits[rows])
    rel_s, peak_s = err(tl_store[rows])
    elem = (np.abs(first_logits[rows] - ref) > 1e-2 + 2e-2 * np.abs(ref)).mean()
    print(f"7B logits: GPU normwise rel {rel:.5f}, max|diff|/row rms {peak:.4f}; bf16 storage alone: "
          f"{rel_s:.5f}, {peak_s:.4f}; GPU fraction outside 1e-2 + 2e-2|ref|: {elem:.5f}")
    assert rel <= STORE_BOUND_FACTOR * rel_s and peak <= STORE_BOUND_FACTOR * peak_s, (rel, rel_s, peak, peak_s)


S_MAX_AR = 768  # prompt 128 + 512 new tokens + one step's tree of 64 nodes and its accepted overshoot


def _library_decode(model, tree, prompt, n_new, force=None, rows=None):
    """Greedy decode of n_new tokens through verify steps. force: the heads' rank-0 candidates are set to
    force[k + 1 ..] before each step (k = tokens emitted so far). rows: a list that receives, for every emitted
    token, the GPU logits row it is the argmax of (the prompt's last row, a root row, or an accepted node's row)."""
    sess = mv.Session(model, tree, S_MAX_AR)
    sess.prefill(torch.as_tensor(prompt, dtype=torch.int32, device="cuda"))
    if rows is not None:
        rows.append(sess.logits[(len(prompt) - 1) % 64].clone())
    out, accs = [], []
    while len(out) < n_new:
        if force is not None:
            k = len(out)
            sess.head_topk[:, 0] = torch.as_tensor(force[k + 1: k + 1 + DIMS.n_medusa], dtype=torch.int32,
                                                   device="cuda")
        sess.step(mv.AcceptParams(mv.GREEDY))
        r = sess.read_result()
        if rows is not None:  # accepted token j + 1 is the argmax of node j's row; the next root of the last one's
            rows.extend(sess.logits[nd].clone() for nd in r["nodes"])
        out += r["tokens"]
        accs.append(r["acc"])
    return np.asarray(out[:n_new]), accs


@pytest.mark.parametrize("n_new", [64, 512])
def test_7b_medusa_equals_library_ar(model7b, n_new):
    """Greedy Medusa decoding with the 64-node tree against the library's plain greedy stream of the same model
    (a root-only tree).

    With the heads' own (random) candidates nothing beyond the root is accepted, every emitted token is the argmax
    of a root row, and a root row is computed bit for bit as the same position decoded alone (the attention sums
    each key tile on a split fixed by its position, whatever the tree): the streams must be identical, with no
    tolerance. With the candidates forced to the AR stream every step accepts the whole path; an accepted node's
    logits are then a second computation of the same row (its keys sit at other cache rows, so the attention sums
    them in another order), equal to the AR row up to rounding. The streams must agree until a position where
    that measured difference of the two rows covers the AR row's top-2 gap, and the two rows must agree within
    2e-2 normwise wherever they are compared."""
    _, model = model7b
    prompt = synth.prompt_tokens(0, P, DIMS.vocab).numpy()
    ar_rows = []
    ar, ar_acc = _library_decode(model, mv.Tree([], 10), prompt, n_new + 8, rows=ar_rows)
    assert set(ar_acc) == {0}
    A = torch.stack(ar_rows[: n_new])
    top2 = torch.topk(A, 2, dim=1).values
    gaps = (top2[:, 0] - top2[:, 1]).cpu().numpy()
    tree = mv.Tree(synth.synthetic_tree_choices(64, 4, 10), 10)
    med, accs = _library_decode(model, tree, prompt, n_new)
    first = lambda a: int(np.argmax(a != ar[:n_new])) if (a != ar[:n_new]).any() else n_new
    print(f"7B library greedy, {n_new} tokens: Medusa = AR for {first(med)} tokens ({len(accs)} steps, "
          f"{sum(accs)} candidates accepted); smallest AR top-2 gap {gaps.min():.3g} at token {int(gaps.argmin())}, "
          f"{int((gaps < 1e-3).sum())} gaps below 1e-3")
    if sum(accs) == 0:  # only root rows: bit-identical computations
        assert med.tolist() == ar[:n_new].tolist()
    f_rows = []
    forced, f_accs = _library_decode(model, tree, prompt, n_new, force=ar, rows=f_rows)
    m = first(forced)
    Fm = torch.stack(f_rows[: m + 1 if m < n_new else n_new])
    diff = (Fm - A[: len(Fm)]).abs()
    rel = (diff.norm(dim=1) / A[: len(Fm)].norm(dim=1)).cpu().numpy()
    print(f"7B forced candidates: = AR for {m} of {n_new} tokens over {len(f_accs)} steps (accept lengths "
          f"{sorted(set(f_accs))}); accepted-node rows against the AR rows: normwise {rel.max():.3g} at most, "
          f"max |diff| {float(diff.max()):.3g}" + (f"; first difference at token {m}: AR top-2 gap {gaps[m]:.3g}, "
                                                   f"the two rows differ there by up to {float(diff[m].max()):.3g}"
                                                   if m < n_new else ""))
    assert rel.max() <= 2e-2, rel.max()
    if m < n_new:
        # the flip needs the two computations to differ by at least half the gap on the two tokens involved
        t_ar, t_med = int(ar[m]), int(forced[m])
        assert gaps[m] <= float(diff[m, t_ar] + diff[m, t_med]), (m, gaps[m], float(diff[m, t_ar]),
                                                                  float(diff[m, t_med]))
    accepted_whole = sum(1 for a in f_accs if a == tree.depth)
    assert accepted_whole >= 1 and (m < n_new or accepted_whole == len(f_accs)), f_accs
