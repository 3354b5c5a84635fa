"""GPU parity of the standalone kernels against the oracle, through the C ABI.

Integer outputs (candidates, accepted paths, compacted KV bits) are compared bit-exactly. Floating-point
outputs must be within 2e-2 relative / 1e-2 absolute of the float64 oracle; an acceptance decision may differ
only where the oracle's margin is below 1e-3; a top-k index may differ only where the two values it separates
are within 1e-3 of each other (a near tie).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import decision_check
import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import generate_candidates
from oracle.kv import kv_compact as oracle_kv_compact
from oracle.model import medusa_heads, topk_ids, tree_attention as oracle_tree_attention
from oracle.posterior import GREEDY, TYPICAL, evaluate_posterior as oracle_posterior
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


def ws(nbytes):
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device="cuda")


def i32(a):
    return torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")


def page_tree_choices():
    """The 63 choices printed on "大模型推理 memory bandwidth bound (5) - Medusa", 二.2 (64 nodes, 42 paths, depth 4)."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "page4_tree.json")) as f:
        return [tuple(c) for c in json.load(f)["medusa_choices"]]


TREES = {
    "synthetic64": (lambda: synth.synthetic_tree_choices(64, 4, 10), 10),
    "page63": (page_tree_choices, 10),
    "dense1x2x3": (lambda: synth.dense_tree_choices([2, 3]), 10),
    "chain5": (lambda: [tuple([0] * k) for k in range(1, 6)], 10),
    "root": (lambda: [], 10),
    "synthetic100": (lambda: synth.synthetic_tree_choices(100, 4, 10), 10),   # two query blocks, two mask words
    "synthetic256": (lambda: synth.synthetic_tree_choices(256, 4, 10), 10),   # the largest tree: four of each
}


def both_trees(name):
    f, topk = TREES[name]
    ch = f()
    return mv.Tree(ch, topk), tree_buffers(ch, topk)


# --------------------------------------------------------------------------------------------- candidates

@pytest.mark.parametrize("name", ["synthetic64", "page63", "dense1x2x3", "chain5", "root", "synthetic256"])
def test_build_candidates_bit_exact(name):
    t, o = both_trees(name)
    K = max(1, o["depth"])
    head_topk = synth.randint(3, "topk", K * 12, 0, 32000).numpy().reshape(K, 12)
    root = 31999
    tt = torch.full((t.n_nodes,), -7, dtype=torch.int32, device="cuda")
    cart = torch.full((t.n_paths, t.depth + 1), -7, dtype=torch.int32, device="cuda")
    mv.build_candidates(i32([root]), i32(head_topk), t, tt, cart)
    ref_tt, ref_cart = generate_candidates(root, head_topk[:, :10], o)
    assert tt.cpu().tolist() == ref_tt.tolist()
    assert cart.cpu().tolist() == ref_cart.tolist()


# --------------------------------------------------------------------------------------------- posterior

def _run_posterior(logits, tokens, t, mode, T=0.7, eps=0.09, delta=0.3):
    n, V = logits.shape
    out = torch.zeros(mv.RESULT_INTS, dtype=torch.int32, device="cuda")
    stats = torch.zeros(n, 4, dtype=torch.float32, device="cuda")
    amax = torch.zeros(n, dtype=torch.int32, device="cuda")
    mv.evaluate_posterior(logits, tokens, t, mv.AcceptParams(mode, T, eps, delta), out,
                          ws(mv.evaluate_posterior_workspace(n)), stats, amax)
    return mv.result_dict(out), stats.cpu().numpy(), amax.cpu().numpy()


def _check_decisions(res, stats, amax, z, tokens, ref, retrieve, mode, T):
    """Each row's first decision that differs from the oracle's must have an oracle margin below MARGIN."""
    acc = decision_check.decisions_from_stats(z, tokens, mode, amax, stats, T)
    return decision_check.check(res, acc, ref, retrieve, mode)


@pytest.mark.parametrize("tree", ["synthetic64", "page63", "synthetic256"])
@pytest.mark.parametrize("mode", [GREEDY, TYPICAL])
@pytest.mark.parametrize("seed", range(10))
def test_posterior_planted_full_size(mode, seed, tree):
    """64 nodes x 32000 vocabulary, logits ~N(0, 3^2), an agreement planted along a random path."""
    t, o = both_trees(tree)
    r = o["retrieve"]
    p = int(synth.randint(seed, "plant_path", 1, 0, len(r))[0])
    path = [int(x) for x in r[p] if x >= 0]
    L = int(synth.randint(seed, "plant_len", 1, 1, len(path))[0])
    tokens, logits = synth.planted_tokens_and_logits(seed, o["n_nodes"], 32000, path, L)
    res, stats, amax = _run_posterior(logits.cuda(), i32(tokens.numpy()), t, mode)
    ref = oracle_posterior(logits.numpy(), tokens.numpy(), r, mode, 0.7, 0.09, 0.3)
    dv = _check_decisions(res, stats, amax, logits.numpy(), tokens.numpy(), ref, r, mode, 0.7)
    assert res["acc"] >= L or dv
    assert res["tokens"] == tokens.numpy()[res["nodes"]].tolist()
    assert res["n_tokens"] == res["acc"] + 1
    assert res["next_node"] == res["nodes"][-1]
    z = logits.numpy().astype(np.float64)
    assert res["next_root"] == int(np.argmax(z[res["next_node"]]))
    assert (amax == np.argmax(z, axis=1)).all()
    assert np.array_equal(stats[:, 0], z.max(axis=1).astype(np.float32))
    if mode == TYPICAL:
        st = ref["stats"]
        y = z / 0.7
        logZ = np.log(np.exp(y - y.max(1, keepdims=True)).sum(1))
        assert np.allclose(stats[:, 1], logZ, rtol=1e-5, atol=1e-5)
        assert np.allclose(stats[:, 2], st["entropy"], rtol=1e-4, atol=1e-5)
        assert np.allclose(stats[:, 3], st["tau"], rtol=1e-4, atol=1e-9)


@pytest.mark.parametrize("mode", [GREEDY, TYPICAL])
@pytest.mark.parametrize("V", [2, 7, 1001])
def test_posterior_small_ragged(mode, V):
    t, o = both_trees("dense1x2x3")
    rng = np.random.default_rng(V + mode)
    tokens = rng.permutation(max(V, 9))[:9] % V
    z = rng.normal(0, 2, size=(9, V)).astype(np.float32)
    # plant node 0 -> node 2 -> node 7
    z[0, tokens[2]] = z[0].max() + 3
    z[2, tokens[7]] = z[2].max() + 3
    ld = (V + 3) // 4 * 4                        # rows padded to a multiple of 4 floats (API contract)
    zp = torch.full((9, ld), float("nan"), dtype=torch.float32)
    zp[:, :V] = torch.tensor(z)
    res, stats, amax = _run_posterior(zp.cuda()[:, :V], i32(tokens), t, mode, T=1.0)
    ref = oracle_posterior(z, tokens, o["retrieve"], mode, 1.0)
    _check_decisions(res, stats, amax, z, tokens, ref, o["retrieve"], mode, 1.0)


def test_posterior_rejects_unaligned_rows():
    t, _ = both_trees("dense1x2x3")
    out = torch.zeros(mv.RESULT_INTS, dtype=torch.int32, device="cuda")
    with pytest.raises(mv.MVError) as e:
        mv.evaluate_posterior(torch.zeros(9, 7, device="cuda"), i32(np.zeros(9)), t, mv.AcceptParams(), out,
                              ws(mv.evaluate_posterior_workspace(9)))
    assert e.value.status == 2


def test_posterior_strided_rows_and_typical_tie_break():
    t, o = both_trees("dense1x2x3")
    V = 8
    tokens = np.array([0, 1, 2, 3, 4, 5, 3, 4, 5])
    z = np.full((9, 12), -20.0, dtype=np.float32)     # rows padded to 12 (ld = 12)
    z[0, [1, 2]] = 0.0
    z[1, [3, 4]] = 0.0
    z[2, [3, 4, 5]] = [1.0, 0.0, 0.0]
    res, _, _ = _run_posterior(torch.tensor(z).cuda()[:, :V], i32(tokens), t, TYPICAL, T=1.0)
    ref = oracle_posterior(z[:, :V], tokens, o["retrieve"], TYPICAL, 1.0)
    assert res["nodes"] == ref["nodes"].tolist() == [0, 2, 6]
    assert res["best"] == ref["best"]


# --------------------------------------------------------------------------------------------- KV compaction

def _kv_case(L, H, S, D, prefix, nodes, seed=0):
    kv = synth.kv_cache(seed, (L, 2, H, S, D), device="cuda")
    before = kv.view(torch.int16).cpu().numpy()
    res = mv.PosteriorResult()
    res.acc = len(nodes) - 1
    res.n_tokens = len(nodes)
    for j, nd in enumerate(nodes):
        res.nodes[j] = nd
    buf = torch.tensor(np.frombuffer(bytes(res), dtype=np.int32).copy(), device="cuda")
    cur = torch.zeros(1, dtype=torch.int32, device="cuda")
    mv.kv_compact(kv, prefix, buf, cur)
    after = kv.view(torch.int16).cpu().numpy()
    ref, new_len = oracle_kv_compact(before, prefix, nodes)
    assert int(cur.item()) == new_len
    assert np.array_equal(after, ref)


@pytest.mark.parametrize("nodes", [[0], [0, 1], [0, 3, 26, 56], [0, 1, 11, 34, 57]])
def test_kv_compact_full_size_bit_exact(nodes):
    """32 layers x 32 heads x 128 dims, prefix 1024 (S_max = 1088)."""
    _kv_case(32, 32, 1088, 128, 1024, nodes)


@pytest.mark.parametrize("D", [4, 16, 132, 256])
def test_kv_compact_small_dims(D):
    _kv_case(2, 3, 80, D, 5, [0, 2, 9, 40])


# --------------------------------------------------------------------------------------------- heads + top-k

def _check_topk(gpu_idx, gpu_val, z, k):
    """gpu top-k (ids, values) against the float64 head logits z."""
    ref = topk_ids(z, k)
    for r in range(k):
        gi, ri = int(gpu_idx[r]), int(ref[r])
        assert gi == ri or abs(z[gi] - z[ri]) < MARGIN, (r, gi, ri, z[gi], z[ri])
        if gpu_val is not None:
            assert abs(gpu_val[r] - z[gi]) <= ATOL + RTOL * abs(z[gi])
    assert len(set(int(i) for i in gpu_idx[:k])) == k


def _heads_case(B, d, K, V, topk, with_lm, seed=0):
    dims = synth.ModelDims(d=d, n_layers=0, n_heads=1, head_dim=d, ffn=d, vocab=V, n_medusa=K)
    w = synth.model_weights(dims, seed, torch.bfloat16, "cuda",
                            names=[f"medusa{k}.w{i}" for k in range(K) for i in (1, 2)] + ["lm_head"])
    w1 = torch.stack([w[f"medusa{k}.w1"] for k in range(K)])
    w2 = torch.stack([w[f"medusa{k}.w2"] for k in range(K)])
    h = synth.normal(seed, "h", (B, d), 1.0, dtype=torch.bfloat16, device="cuda")
    out_idx = torch.full((B, K, topk), -1, dtype=torch.int32, device="cuda")
    out_val = torch.zeros(B, K, topk, dtype=torch.float32, device="cuda")
    root = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    mv.medusa_heads_topk(h, w1, w2, topk, out_idx, out_val, w_lm=w["lm_head"] if with_lm else None,
                         out_root=root, workspace=ws(mv.medusa_heads_topk_workspace(B, d, K, V, topk)))
    torch.cuda.synchronize()
    cache = {}

    def get(name):
        if name not in cache:
            cache[name] = w[name].double().cpu().numpy()
        return cache[name]

    hh = h.double().cpu().numpy()
    gi, gv, gr = out_idx.cpu().numpy(), out_val.cpu().numpy(), root.cpu().numpy()
    for b in range(B):
        z = medusa_heads(get, K, hh[b])
        for k in range(K):
            _check_topk(gi[b, k], gv[b, k], z[k], topk)
        if with_lm:
            zl = get("lm_head") @ hh[b]
            ri = int(np.argmax(zl))
            assert gr[b] == ri or abs(zl[gr[b]] - zl[ri]) < MARGIN


@pytest.mark.parametrize("B", [1, 4, 16])
def test_heads_topk_full_size(B):
    """4 heads, d = 4096, V = 32000, top-10, plus the LM-head top-1."""
    _heads_case(B, 4096, 4, 32000, 10, True)


@pytest.mark.parametrize("B,d,K,V,topk", [(1, 64, 2, 512, 10), (3, 64, 2, 512, 10), (2, 8, 1, 16, 16),
                                          (5, 1024, 3, 1000, 7), (1, 8192, 1, 300, 1), (1, 8, 1, 16, 16),
                                          (1, 520, 3, 777, 5), (1, 2056, 2, 4099, 10), (1, 64, 8, 300, 16)])
def test_heads_topk_small(B, d, K, V, topk):
    _heads_case(B, d, K, V, topk, True)


def test_heads_topk_workspace_reused_across_calls():
    """One zero-filled workspace serves repeated calls, batch-1 and batched ones interleaved: each batch-1 pass
    leaves its tile counters and tickets at zero, and the batched path does not touch them."""
    d, K, V, topk = 520, 3, 777, 5
    dims = synth.ModelDims(d=d, n_layers=0, n_heads=1, head_dim=d, ffn=d, vocab=V, n_medusa=K)
    w = synth.model_weights(dims, 0, torch.bfloat16, "cuda",
                            names=[f"medusa{k}.w{i}" for k in range(K) for i in (1, 2)] + ["lm_head"])
    w1 = torch.stack([w[f"medusa{k}.w1"] for k in range(K)])
    w2 = torch.stack([w[f"medusa{k}.w2"] for k in range(K)])
    wk = ws(mv.medusa_heads_topk_workspace(4, d, K, V, topk))
    get = lambda name: w[name].double().cpu().numpy()
    for call, B in enumerate([1, 1, 4, 1, 2, 1]):
        h = synth.normal(call, "h", (B, d), 1.0, dtype=torch.bfloat16, device="cuda")
        out_idx = torch.full((B, K, topk), -1, dtype=torch.int32, device="cuda")
        out_val = torch.zeros(B, K, topk, dtype=torch.float32, device="cuda")
        root = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        mv.medusa_heads_topk(h, w1, w2, topk, out_idx, out_val, w_lm=w["lm_head"], out_root=root, workspace=wk)
        torch.cuda.synchronize()
        hh = h.double().cpu().numpy()
        gi, gv, gr = out_idx.cpu().numpy(), out_val.cpu().numpy(), root.cpu().numpy()
        for b in range(B):
            z = medusa_heads(get, K, hh[b])
            for k in range(K):
                _check_topk(gi[b, k], gv[b, k], z[k], topk)
            zl = get("lm_head") @ hh[b]
            ri = int(np.argmax(zl))
            assert gr[b] == ri or abs(zl[gr[b]] - zl[ri]) < MARGIN, (call, b)
        assert int(wk[:256].view(torch.int32).abs().sum().item()) == 0, call  # the control block is zero again


# --------------------------------------------------------------------------------------------- tree attention

def _attn_case(H, D, P, tree_name, S_max=None, seed=0):
    t, o = both_trees(tree_name)
    n = o["n_nodes"]
    S_max = S_max or P + n
    q = synth.normal(seed, "q", (n, H, D), dtype=torch.bfloat16, device="cuda")
    k = synth.normal(seed, "k", (H, S_max, D), dtype=torch.bfloat16, device="cuda")
    v = synth.normal(seed, "v", (H, S_max, D), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(n, H, D, dtype=torch.bfloat16, device="cuda")
    scale = 1.0 / math.sqrt(D)
    mv.tree_attention(q, k, v, P, t, scale, out, ws(mv.tree_attention_workspace(H, D, S_max, n)))
    got = out.double().cpu().numpy()
    ref = oracle_tree_attention(q.double().cpu().numpy(), k.double().cpu().numpy().transpose(1, 0, 2),
                                v.double().cpu().numpy().transpose(1, 0, 2), P, o["attn_mask"], scale)
    assert np.allclose(got, ref, rtol=RTOL, atol=ATOL)
    assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)


@pytest.mark.parametrize("P", [64, 512, 1024, 4096])
@pytest.mark.parametrize("tree", ["synthetic64", "page63", "synthetic100", "synthetic256"])
def test_tree_attention_full_size(P, tree):
    """32 heads x 128 dims, the synthetic 64-node tree or the page's own, q/k/v ~N(0,1)."""
    _attn_case(32, 128, P, tree)


@pytest.mark.parametrize("H,D,P,tree,S_max", [(3, 16, 0, "dense1x2x3", None), (2, 32, 5, "dense1x2x3", 40),
                                              (4, 64, 130, "chain5", None), (1, 128, 7, "root", None),
                                              (5, 128, 0, "synthetic64", 64), (2, 128, 200, "synthetic64", 300),
                                              (2, 64, 37, "synthetic100", None), (3, 128, 0, "synthetic256", 256),
                                              (1, 32, 70, "synthetic256", None)])
def test_tree_attention_small_ragged(H, D, P, tree, S_max):
    _attn_case(H, D, P, tree, S_max)


@pytest.mark.parametrize("H,D,P,tree,S_max", [(2, 128, 0, "synthetic64", 4200), (3, 64, 37, "synthetic100", 4400),
                                              (1, 128, 4100, "root", None), (2, 128, 1000, "synthetic256", 4300),
                                              (1, 64, 4200, "chain5", None), (4, 128, 4500, "page63", None),
                                              (2, 128, 131, "dense1x2x3", 4200), (3, 64, 0, "synthetic256", 4097)])
def test_tree_attention_long_cache(H, D, P, tree, S_max):
    """Caches longer than 4096 rows (head dim 64 or 128) run on the tcgen05 attention: 128-key tiles on the tensor
    memory accumulators, 64 query rows per CTA. Short and long prefixes, trees of 1 to 256 nodes (up to four blocks
    of 64 rows), ragged ends."""
    _attn_case(H, D, P, tree, S_max)


@pytest.mark.parametrize("S_max", [700, 4200])
def test_tree_attention_root_row_independent_of_the_tree(S_max):
    """Both attention kernels: the root row of a 64-node tree is bit for bit the row of the same token attending
    alone (a tree of the root only) at the same prefix, since key tiles go to splits by absolute position and
    fully masked tiles add exact zeros."""
    H, D, P = 8, 128, 600
    k = synth.normal(1, "k", (H, S_max, D), dtype=torch.bfloat16, device="cuda")
    v = synth.normal(1, "v", (H, S_max, D), dtype=torch.bfloat16, device="cuda")
    rows = []
    for name in ("root", "synthetic64"):
        t, o = both_trees(name)
        n = o["n_nodes"]
        q = synth.normal(1, "q", (n, H, D), dtype=torch.bfloat16, device="cuda")
        if name == "synthetic64":
            q[0] = rows_q0
        rows_q0 = q[0].clone()
        out = torch.zeros(n, H, D, dtype=torch.bfloat16, device="cuda")
        mv.tree_attention(q, k, v, P, t, 1.0 / math.sqrt(D), out, ws(mv.tree_attention_workspace(H, D, S_max, n)))
        torch.cuda.synchronize()
        rows.append(out[0].cpu())
    assert torch.equal(rows[0], rows[1])
