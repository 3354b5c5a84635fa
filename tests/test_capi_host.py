"""The C-ABI library on the host (no GPU needed): it loads, exports every declared entry point, and its
tree builder matches the oracle's on the page's example and on the synthetic and dense trees."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import synth
import medusa_tree_speculative_verify_gb300 as mv
from oracle.tree import tree_buffers

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            names += re.findall(r"^(?:mv_status|void|const char\s*\*)\s+(\w+)\s*\(", txt, re.M)
    return names


def test_library_exports_every_declared_symbol():
    L = mv.lib()
    names = _declared()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
    assert set(names) <= set(mv.EXPORTED_SYMBOLS) | set(getattr(mv, "EXTRA_SYMBOLS", ()))


def _compare(choices, topk):
    t = mv.Tree(choices, topk)
    o = tree_buffers(choices, topk)
    assert t.n_nodes == o["n_nodes"] and t.depth == o["depth"]
    assert t.tree_indices.tolist() == o["tree_indices"].tolist()
    assert t.position_ids.tolist() == o["position_ids"].tolist()
    assert t.retrieve.tolist() == o["retrieve"].tolist()
    assert t.parent.tolist() == o["parent"].tolist()
    assert (t.attn_mask() == o["attn_mask"]).all()


def test_tree_page_example():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "page4_tree.json")))
    _compare([tuple(c) for c in g["medusa_choices"]], 10)
    t = mv.Tree([tuple(c) for c in g["medusa_choices"]], 10)
    assert t.retrieve.tolist() == g["retrieve_indices"]


@pytest.mark.parametrize("kind", ["synthetic", "dense", "chain", "root_only", "synthetic130", "synthetic256"])
def test_tree_matches_oracle(kind):
    choices = {"synthetic": synth.synthetic_tree_choices(64, 4, 10),
               "synthetic130": synth.synthetic_tree_choices(130, 4, 10),   # masks of three words
               "synthetic256": synth.synthetic_tree_choices(256, 4, 10),
               "dense": synth.dense_tree_choices([2, 3]),
               "chain": [tuple([0] * k) for k in range(1, 9)],
               "root_only": []}[kind]
    if kind == "root_only":
        t = mv.Tree([], 10)
        assert t.n_nodes == 1 and t.retrieve.tolist() == [[0]]
        return
    _compare(choices, 10)


@pytest.mark.parametrize("choices,topk", [
    ([(0, 0)], 10),                      # not prefix-closed
    ([(0,), (0,)], 10),                  # duplicate
    ([(3,)], 3),                         # rank >= topk
    ([(0,) * 9], 10),                    # deeper than MAX_DEPTH (and not prefix-closed)
    ([(i,) for i in range(200)] + [(0, j) for j in range(56)], 200),   # 257 nodes > MAX_NODES
])
def test_tree_errors(choices, topk):
    with pytest.raises(mv.MVError) as e:
        mv.Tree(choices, topk)
    assert e.value.status == 3            # MV_ERR_TREE


def test_packed_weight_sizes():
    import ctypes
    n = ctypes.c_size_t()
    assert mv.lib().mv_packed_weight_bytes(300, 72, 128, ctypes.byref(n)) == 0
    assert n.value == 3 * 2 * 128 * 64 * 2            # 3 row tiles x 2 k-blocks, zero padded
    assert mv.lib().mv_packed_weight_bytes(300, 70, 128, ctypes.byref(n)) == 2   # K % 8 != 0


def test_workspace_queries_and_shape_errors():
    assert mv.evaluate_posterior_workspace(64) > 64 * 16
    assert mv.tree_attention_workspace(32, 128, 4160, 64) > 0
    assert mv.medusa_heads_topk_workspace(16, 4096, 4, 32000, 10) > 0
    with pytest.raises(mv.MVError):
        mv.tree_attention_workspace(32, 96, 4160, 64)        # unsupported head dim
    with pytest.raises(mv.MVError):
        mv.medusa_heads_topk_workspace(17, 4096, 4, 32000, 10)  # batch above 16


def test_root_sampling_argument_errors():
    """sample_root / mv_session_set_root_sampling reject bad arguments on the host, before any launch."""
    L = mv.lib()
    fake = ctypes.c_void_p(0x1000)                              # never dereferenced: validation fails first
    bad = [mv.RootParams(3), mv.RootParams(mv.ROOT_NUCLEUS, 0.0), mv.RootParams(mv.ROOT_NUCLEUS, -1.0),
           mv.RootParams(mv.ROOT_NUCLEUS, float("nan")), mv.RootParams(mv.ROOT_NUCLEUS, top_p=0.0),
           mv.RootParams(mv.ROOT_NUCLEUS, top_p=1.01), mv.RootParams(mv.ROOT_TYPICAL, eps=-0.1),
           mv.RootParams(mv.ROOT_TYPICAL, delta=-0.1)]
    for prm in bad:
        assert L.sample_root(fake, 100, prm, 0, fake, None) == 1, (prm.mode, prm.temperature, prm.top_p)
    good = mv.RootParams(mv.ROOT_NUCLEUS)
    assert L.sample_root(None, 100, good, 0, fake, None) == 1    # null logits
    assert L.sample_root(fake, 0, good, 0, fake, None) == 1      # empty row
    assert L.sample_root(fake, 100, good, 0, None, None) == 1    # null output
    assert L.mv_session_set_root_sampling(None, good, 0, None) == 1
    assert ctypes.sizeof(mv.RootParams) == 32
