"""The allocation-free posterior entry point against the workspace one (GPU).

evaluate_posterior_noalloc serves callers that cannot call cudaMalloc (code under another runtime's memory
manager, or a serving loop that must not touch the device allocator after start-up): it keeps its scratch in
a fixed array inside the library instead of a caller workspace. Its results must equal evaluate_posterior's
on the same inputs, on two calls in a row (the second call finds the array as the first one left it). This
file is collected last and is self-contained, so it passes alone in a fresh process or after the other tests.
"""
import numpy as np
import pytest
import torch

import medusa_tree_speculative_verify_gb300 as mv
import synth

pytestmark = pytest.mark.gpu
RTOL, ATOL = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    yield
    st, code = mv.get_error()
    assert st == 0, f"device error word set: {code:#x}"


def _case(seed, tree):
    path = [int(x) for x in tree.retrieve[seed % tree.n_paths] if x >= 0]
    tokens, logits = synth.planted_tokens_and_logits(seed, tree.n_nodes, 32000, path, len(path) - 1)
    return logits.cuda(), torch.as_tensor(tokens, dtype=torch.int32, device="cuda")


def _outputs(fn, logits, tokens, tree, prm, **kw):
    n = tree.n_nodes
    out = torch.full((mv.RESULT_INTS,), -5, dtype=torch.int32, device="cuda")
    stats = torch.zeros(n, 4, dtype=torch.float32, device="cuda")
    amax = torch.zeros(n, dtype=torch.int32, device="cuda")
    fn(logits, tokens, tree, prm, out, node_stats=stats, node_argmax=amax, **kw)
    torch.cuda.synchronize()
    return mv.result_dict(out), stats.cpu().numpy(), amax.cpu().numpy()


def test_noalloc_posterior_matches_workspace_posterior_twice():
    tree = mv.Tree(synth.synthetic_tree_choices(64, 4, 10), 10)
    ws = torch.zeros(mv.evaluate_posterior_workspace(tree.n_nodes), dtype=torch.uint8, device="cuda")
    calls = [(0, mv.AcceptParams(mv.GREEDY)), (1, mv.AcceptParams(mv.TYPICAL, 0.7, 0.09, 0.3))]
    for seed, prm in calls:  # two calls in a row on the shared scratch array
        logits, tokens = _case(seed, tree)
        ref = _outputs(lambda *a, **k: mv.evaluate_posterior(*a[:5], ws, **k), logits, tokens, tree, prm)
        got = _outputs(mv.evaluate_posterior_noalloc, logits, tokens, tree, prm)
        assert got[0] == ref[0]
        assert np.array_equal(got[2], ref[2])
        assert np.allclose(got[1], ref[1], rtol=RTOL, atol=ATOL)
        assert got[0]["acc"] >= 1            # the planted path is accepted


def test_noalloc_posterior_rejects_trees_past_its_limit():
    """A tree of more nodes than the fixed array holds is refused before anything is launched."""
    big = mv.Tree(synth.synthetic_tree_choices(65, 4, 10), 10)
    assert big.n_nodes == 65 > mv.NOALLOC_MAX_NODES
    logits, tokens = _case(0, big)
    out = torch.full((mv.RESULT_INTS,), -5, dtype=torch.int32, device="cuda")
    with pytest.raises(mv.MVError) as e:
        mv.evaluate_posterior_noalloc(logits, tokens, big, mv.AcceptParams(mv.GREEDY), out)
    assert e.value.status == 4  # MV_ERR_CAPACITY
    torch.cuda.synchronize()
    assert (out == -5).all()    # nothing ran
