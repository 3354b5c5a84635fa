"""GPU parity of the stochastic root (typical and nucleus one-token draws) against the oracle.

"大模型推理 memory bandwidth bound (5) - Medusa", 二.4 generate_candidates() (get_typical_one_token /
get_nucleus_one_token for temperature > 0), 一.3 Typical acceptance; nucleus sampling after Holtzman et al.

The kernel draws with its own SplitMix64 and fixed-point masses; the oracle draws in float64 with the uniform of
``synth``. A draw must equal the oracle's, unless the oracle's own decision lies within rounding of a boundary:
a token whose membership could flip (|ln p - ln tau| below the typical tolerance, or the mass before it within
the nucleus tolerance of top_p) or a uniform within the cumulative tolerance of a step of the CDF. Such a draw
must still be one the oracle can reach inside those tolerances, and at least 90% of the draws must match exactly.
"""
import numpy as np
import pytest
import torch

import decision_check
import medusa_tree_speculative_verify_gb300 as mv
import synth
from oracle.decode import chain_mask, prefill as o_prefill, verify_step as o_verify_step
from oracle.model import Backbone, KVCache
from oracle.posterior import TYPICAL
from oracle.sampling import (NUCLEUS, TYPICAL_ONE, RootSampler, inverse_cdf, nucleus_allow, softmax_t,
                             typical_allow, uniform)
from oracle.tree import tree_buffers

pytestmark = pytest.mark.gpu

TOL_LN = 1e-4     # typical: fp32 exp / log / entropy sums against float64, in ln(p / tau)
TOL_MASS = 5e-6   # nucleus mass before a token, and the uniform against the cumulative (fixed-point + fp32 exp)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    yield
    st, code = mv.get_error()
    assert st == 0, f"device error word set: {code:#x}"


class OracleRow:
    """The oracle's view of one row for many uniforms: p, the allow set and its tolerance bounds."""

    def __init__(self, z, mode, T, eps, delta, top_p, tol_ln=TOL_LN, tol_mass=TOL_MASS):
        self.p = softmax_t(z, T)
        if mode == TYPICAL_ONE:
            allow, margin = typical_allow(z, T, eps, delta)
            self.lo, self.hi = margin > tol_ln, margin > -tol_ln
        else:
            allow, before = nucleus_allow(z, T, top_p)
            self.lo, self.hi = before < top_p - tol_mass, before < top_p + tol_mass
        self.allow = allow
        self.tol_u = tol_mass

    def token(self, u):
        return inverse_cdf(self.p, self.allow, u)

    def reachable(self, g, u):
        """Whether some allow set between the strict and the loose one, and a uniform within tolerance, give g."""
        p, lo, hi = self.p, self.lo, self.hi
        if not (0 <= g < len(p)) or not hi[g]:
            return False
        b_min, b_max = p[:g][lo[:g]].sum(), p[:g][hi[:g]].sum()
        z_min = p[lo].sum() + (0.0 if lo[g] else p[g])
        z_max = p[hi].sum()
        return b_min / z_max <= u + self.tol_u and (b_max + p[g]) / z_min >= u - self.tol_u


def _draws(row, prm, counters, offset=0):
    """GPU tokens for each counter; row is placed `offset` floats into its buffer (alignment cases)."""
    V = row.numel()
    buf = torch.zeros(V + offset, dtype=torch.float32, device="cuda")
    buf[offset:] = row
    out = torch.empty(len(counters), dtype=torch.int32, device="cuda")
    for i, c in enumerate(counters):
        mv.sample_root(buf[offset:], prm, c, out[i:i + 1])
    torch.cuda.synchronize()
    return out.cpu().tolist()


def _check_row(z, mode, T, top_p, key, n_draws, offset=0, eps=0.09, delta=0.3):
    row = torch.as_tensor(z, dtype=torch.float32, device="cuda")
    zr = row.double().cpu().numpy()                     # the fp32 row both sides read
    mvmode = mv.ROOT_TYPICAL if mode == TYPICAL_ONE else mv.ROOT_NUCLEUS
    prm = mv.RootParams(mvmode, T, eps, delta, top_p, key)
    counters = list(range(5, 5 + n_draws))
    got = _draws(row, prm, counters, offset)
    orow = OracleRow(zr, mode, T, eps, delta, top_p)
    exact = 0
    for c, g in zip(counters, got):
        u = uniform(key, c)
        want = orow.token(u)
        if g == want:
            exact += 1
        else:
            assert orow.reachable(g, u), (mode, T, top_p, c, u, g, want)
    return exact, len(counters)


@pytest.mark.parametrize("mode", [TYPICAL_ONE, NUCLEUS])
@pytest.mark.parametrize("T,top_p,scale", [(0.7, 0.8, 2.0), (1.0, 0.5, 1.0), (0.3, 0.95, 3.0), (0.7, 1.0, 0.05),
                                           (2.0, 0.8, 4.0)])
def test_root_draw_matches_oracle_32000(mode, T, top_p, scale):
    z = synth.normal(int(T * 10) + int(scale * 100), "root_row", (32000,), scale, dtype=torch.float32)
    exact, n = _check_row(z, mode, T, top_p, key=0xABCDEF, n_draws=160)
    assert exact >= 0.9 * n


@pytest.mark.parametrize("mode", [TYPICAL_ONE, NUCLEUS])
@pytest.mark.parametrize("V,offset", [(1, 0), (7, 1), (513, 0), (1001, 3), (60000, 0), (128256, 0)])
def test_root_draw_shapes(mode, V, offset):
    """Tiny rows, rows not a multiple of 4 at unaligned addresses, and rows too long to stage in shared memory."""
    z = synth.normal(V, "root_shape", (V,), 2.0, dtype=torch.float32)
    exact, n = _check_row(z, mode, 0.7, 0.8, key=V, n_draws=60, offset=offset)
    assert exact >= 0.9 * n


@pytest.mark.parametrize("top_p", [0.3, 0.8, 0.999])
def test_nucleus_ties_quantised_logits(top_p):
    """Logits on a grid of 0.25: large groups of equal logits, kept by lower index first."""
    z = torch.round(synth.normal(3, "root_ties", (32000,), 1.5, dtype=torch.float32) * 4.0) / 4.0
    exact, n = _check_row(z, NUCLEUS, 0.7, top_p, key=99, n_draws=120)
    assert exact >= 0.9 * n


def test_nucleus_allow_set_exact_on_ties():
    """With top_p splitting a tie group, the kept members are the lowest indices: draws from a grid of
    counters reach exactly the oracle's kept set (no token outside it)."""
    V = 4096
    z = torch.zeros(V, dtype=torch.float32)
    z[100:110] = 3.0              # 10 tied leaders, then a flat tail
    row = z.cuda()
    p = softmax_t(z.double().numpy(), 1.0)
    top_p = 6.5 * p[100]          # 6.5 leaders' mass: the 7 lowest-index leaders are kept
    allow, _ = nucleus_allow(z.double().numpy(), 1.0, top_p)
    assert np.flatnonzero(allow).tolist() == list(range(100, 107))
    got = _draws(row, mv.RootParams(mv.ROOT_NUCLEUS, 1.0, top_p=float(top_p), key=5), list(range(400)))
    assert set(got) == set(range(100, 107))
    for c, g in zip(range(400), got):
        assert g == inverse_cdf(p, allow, uniform(5, c))


@pytest.mark.parametrize("top_p", [0.3, 0.8, 1.0])
def test_nucleus_cluster_equals_single_cta(top_p):
    """Rows up to 131072 logits are drawn by a cluster of CTAs, longer rows by one CTA. The masses are exact
    fixed-point sums, so both give the same token: a row, and the same row with one -inf logit appended
    (131072 -> 131073 logits, the other kernel), for the same counters."""
    V = 131072
    z = synth.normal(7, "root_long", (V,), 2.0, dtype=torch.float32)
    z2 = torch.cat([z, torch.tensor([-float("inf")], dtype=torch.float32)])
    prm = mv.RootParams(mv.ROOT_NUCLEUS, 0.7, top_p=top_p, key=3)
    counters = list(range(40))
    assert _draws(z.cuda(), prm, counters) == _draws(z2.cuda(), prm, counters)


@pytest.mark.parametrize("top_p", [0.5, 0.9])
def test_nucleus_dense_bin(top_p):
    """32000 distinct logits within 0.032 of each other: every token falls in the first bin of 1/16 nat, so the
    boundary is found among the sub-bins of that bin."""
    V = 32000
    order = torch.argsort(synth.normal(5, "root_perm", (V,), 1.0, dtype=torch.float32))
    z = order.to(torch.float32) * 1e-6
    exact, n = _check_row(z, NUCLEUS, 0.7, top_p, key=11, n_draws=120)
    assert exact >= 0.9 * n


def test_argmax_mode_and_bad_params():
    z = synth.normal(0, "root_row", (32000,), 1.0, dtype=torch.float32).cuda()
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    mv.sample_root(z, mv.RootParams(mv.ROOT_ARGMAX), 0, out)
    assert int(out.item()) == int(torch.argmax(z).item())
    for bad in [mv.RootParams(3), mv.RootParams(mv.ROOT_NUCLEUS, 0.0), mv.RootParams(mv.ROOT_NUCLEUS, top_p=0.0),
                mv.RootParams(mv.ROOT_NUCLEUS, top_p=1.5), mv.RootParams(mv.ROOT_TYPICAL, eps=-1.0)]:
        with pytest.raises(mv.MVError):
            mv.sample_root(z, bad, 0, out)


# --------------------------------------------------------------------------------------------- in the decode

DIMS = synth.TINY
S_MAX = 256


def _setup():
    w = synth.packed_weights(DIMS, 0, torch.bfloat16, "cuda")
    model = mv.Model(DIMS, mv.pack_model_weights(w))
    choices = synth.dense_tree_choices([2, 3])
    tree = mv.Tree(choices, 10)
    sess = mv.Session(model, tree, S_MAX)
    om = Backbone(DIMS, synth.unpacked_getter(DIMS, w))
    return model, tree, sess, om, tree_buffers(choices, 10)


@pytest.mark.parametrize("mode", [mv.ROOT_TYPICAL, mv.ROOT_NUCLEUS])
def test_session_root_uses_the_consumed_row_and_counter(mode):
    """After prefill and after each step the session's root is the standalone draw from the logits row of
    node retrieve[best][acc] (the prompt's last row after prefill) with counters c0, c0 + 1, ..."""
    _, tree, sess, _, _ = _setup()
    prm = mv.RootParams(mode, 0.7, 0.09, 0.3, 0.8, key=0x1234)
    c0 = 40
    sess.set_root_sampling(prm, c0)
    p = torch.as_tensor(synth.prompt_tokens(0, 32, DIMS.vocab), dtype=torch.int32, device="cuda")
    sess.prefill(p)
    one = torch.empty(1, dtype=torch.int32, device="cuda")
    row = sess.logits[31].contiguous()
    mv.sample_root(row, prm, c0, one)
    torch.cuda.synchronize()
    assert sess.read_result()["next_root"] == int(one.item())
    assert int(sess.root_counter.item()) == c0 + 1
    for i in range(5):
        sess.step(mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3))
        r = sess.read_result()
        mv.sample_root(sess.logits[r["next_node"]].contiguous(), prm, c0 + 1 + i, one)
        torch.cuda.synchronize()
        assert r["next_root"] == int(one.item())
        assert int(sess.root_counter.item()) == c0 + 2 + i


def test_sampled_decode_matches_oracle():
    """Typical acceptance with nucleus roots: the GPU stream equals the oracle's until a decision the bf16
    logits can legitimately flip (a near-threshold acceptance or a draw within tolerance of a CDF step)."""
    _, tree, sess, om, ot = _setup()
    key, c0 = 77, 0
    sess.set_root_sampling(mv.RootParams(mv.ROOT_NUCLEUS, 0.7, top_p=0.8, key=key), c0)
    p = synth.prompt_tokens(0, 32, DIMS.vocab)
    sess.prefill(torch.as_tensor(p, dtype=torch.int32, device="cuda"))
    rs = RootSampler(NUCLEUS, 0.7, top_p=0.8, key=key, counter=c0)
    st = o_prefill(om, p.numpy(), S_MAX, 10, root=rs)
    loose = dict(tol_ln=2e-2, tol_mass=2e-2)
    if sess.read_result()["next_root"] != st.root:     # the prefill root: explained by the oracle's last row
        _, lg = om.forward(p.numpy(), np.arange(len(p)), KVCache(DIMS, S_MAX), 0, chain_mask(len(p)))
        assert OracleRow(lg[-1], NUCLEUS, 0.7, 0.09, 0.3, 0.8, **loose).reachable(
            sess.read_result()["next_root"], rs.draws[0][1])
        return
    for _ in range(8):
        sess.step(mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3))
        toks, info = o_verify_step(om, st, ot, TYPICAL, 0.7, 0.09, 0.3, root=rs)
        res, post = sess.read_result(), info["post"]
        acc = decision_check.decisions_from_logits(sess.logits[: tree.n_nodes].cpu().numpy(),
                                                   sess.tree_tokens.cpu().numpy(), TYPICAL, 0.7, 0.09, 0.3)
        if decision_check.check(res, acc, post, ot["retrieve"], TYPICAL):
            return  # a near-threshold decision: the streams legitimately diverge from here
        assert res["tokens"] == toks.tolist()
        if res["next_root"] != st.root:
            c, u, _ = rs.draws[-1]
            orow = OracleRow(info["logits"][post["next_node"]], NUCLEUS, 0.7, 0.09, 0.3, 0.8, **loose)
            assert orow.reachable(res["next_root"], u)
            return



def test_graph_replay_with_sampled_roots_equals_eager():
    _, _, s1, _, _ = _setup()
    _, _, s2, _, _ = _setup()
    prm = mv.RootParams(mv.ROOT_TYPICAL, 0.7, 0.09, 0.3, key=3)
    p = torch.as_tensor(synth.prompt_tokens(0, 32, DIMS.vocab), dtype=torch.int32, device="cuda")
    acc = mv.AcceptParams(TYPICAL, 0.7, 0.09, 0.3)
    for s in (s1, s2):
        s.set_root_sampling(prm, 11)
        s.prefill(p)
    for _ in range(6):
        s1.step(acc)
    s2.steps_graph(3, acc)
    s2.steps_graph(3, acc)
    torch.cuda.synchronize()
    assert s1.read_result() == s2.read_result()
    assert int(s1.cur_len.item()) == int(s2.cur_len.item())
    assert int(s1.root_counter.item()) == int(s2.root_counter.item()) == 11 + 7
    assert torch.equal(s1.head_topk, s2.head_topk)
