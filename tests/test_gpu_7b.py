"""Full-size parity of the verify loop at Llama-7B shape (32 layers, d 4096, 32 x 128 heads, FFN 11008,
vocabulary 32000, 4 Medusa heads, the synthetic 64-node tree, a random 128-token prompt), in the launch
configuration bench.py times (packed weights, CUDA-graph replay of the steps).

The float64 oracle cannot decode 64 tokens of a 7B model one by one in reasonable time, so it checks sampled
outputs and properties that hold at any size:
* teacher forcing: one causal oracle forward over prompt + the 64 GPU tokens; every GPU token must be the
  oracle argmax or within the margin that bf16 storage itself explains ("Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu", 2️⃣:
  greedy Medusa output equals the base model's; "大模型推理 memory bandwidth bound (5) - Medusa", 二.1);
* the first verify step's LM logits on sampled tree nodes against the oracle's tree forward (二.5).
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
    # Reading of the token check at full depth: a GPU token is the oracle argmax, or its oracle margin (top-1
    # minus its logit) is at most the larger of 1e-2 + 2e-2 |top-1| and twice the largest logit movement that bf16
    # storage alone causes on this step's 64 tree rows (same oracle, storage hook, no other change); and at least
    # 3/4 of the tokens are the exact argmax (bf16 storage alone keeps about 9 in 10 argmaxes of these rows).
    lg = np.concatenate([lg_prompt[-1:], lg_gen[:-1]])
    margins = lg.max(axis=1) - lg[np.arange(N_NEW), gen]
    d_store = np.abs(tl_store - tl).max()
    exact = float((margins == 0).mean())
    print(f"7B teacher forcing: {int((margins > 0).sum())} of {N_NEW} tokens differ from the oracle argmax, "
          f"largest margin {margins.max():.4f}, exact-match prefix {int(np.argmax(margins > 0)) if (margins > 0).any() else N_NEW}; "
          f"bf16 storage alone moves a tree-row logit by up to {d_store:.4f} and keeps "
          f"{float((tl_store.argmax(1) == tl.argmax(1)).mean()):.3f} of the argmaxes")
    for i, t in enumerate(gen):
        top = lg[i].max()
        assert top - lg[i, t] <= max(1e-2 + 2e-2 * abs(top), 2 * d_store), (i, int(t), int(np.argmax(lg[i])), top - lg[i, t])
    assert exact >= 0.75, exact
    # 2) the first step's LM logits on sampled tree nodes against the oracle's tree forward at prefix P.
    # Reading of the 2e-2 relative / 1e-2 absolute bound for an output composed through 32 layers: the path keeps
    # q, k, v (the cache), the attention output, the SiLU-gate product and the normalised operands in bf16, and
    # that storage alone moves the exact model's logits by a measurable amount that grows with depth (tl_store
    # above). The GPU logits must stay within twice that movement (normwise and per element relative to the row's
    # RMS), i.e. the kernels' own arithmetic may add at most as much error again as the storage format itself.
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
    assert rel <= 2 * rel_s and peak <= 2 * peak_s, (rel, rel_s, peak, peak_s)
