"""Device-side failure detection, exercised without any GPU fault (GPU).

The kernels never trust an index read from device memory and never wait without a bound: a bad index is
rejected before it is used, and a wait gives up after its limit. Either way the kernel records a code in the
library's sticky device error word and returns, and the context stays usable. Both forms are made to happen
here on purpose:
* an index rejected before any access: KV compaction ("大模型推理 memory bandwidth bound (5) - Medusa", 二.7
  update_inference_inputs()) given an accepted path whose rows lie past the end of the cache;
* a bounded wait that runs out: the library's own counter and mbarrier waits, run with a 20 us limit on a
  counter and a barrier that nothing completes (mv_selftest_wait_timeout).
"""
import numpy as np
import pytest
import torch

import medusa_tree_speculative_verify_gb300 as mv
import synth

pytestmark = pytest.mark.gpu
MV_ERR_DEVICE = 6
DEVERR_TIMEOUT, DEVERR_INDEX = 1, 2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    mv.lib()
    st, _ = mv.get_error()
    assert st == 0
    yield


def _result(acc, nodes):
    r = mv.PosteriorResult()
    r.acc, r.n_tokens = acc, acc + 1
    for j, nd in enumerate(nodes):
        r.nodes[j] = nd
    return torch.tensor(np.frombuffer(bytes(r), dtype=np.int32).copy(), device="cuda")


@pytest.mark.parametrize("case", ["row_past_cache", "acc_out_of_range"])
def test_kv_compact_rejects_bad_indices_before_any_access(case):
    L, H, S, D = 2, 2, 64, 16
    kv = synth.kv_cache(0, (L, 2, H, S, D), device="cuda")
    before = kv.clone()
    prefix = S - 10
    cur = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    if case == "row_past_cache":  # node 20 of the path: row prefix + 20 = S + 10
        mv.kv_compact(kv, prefix, _result(1, [0, 20]), cur)
        site, detail = 6, (1 << 24) | (prefix + 20)
    else:  # an accept length past MV_MAX_DEPTH
        mv.kv_compact(kv, prefix, _result(9, [0]), cur)
        site, detail = 5, (9 << 24) | prefix
    st, code, det = mv.get_error(with_detail=True)
    assert st == MV_ERR_DEVICE and code == (site << 16) | DEVERR_INDEX and det == detail, (st, hex(code), hex(det))
    assert torch.equal(kv, before)          # rejected before any row was read or written
    assert int(cur.item()) == -7            # and before the length was touched
    # the context is usable and the word clear: a valid compaction right after works
    mv.kv_compact(kv, prefix, _result(1, [0, 3]), cur)
    assert mv.get_error() == (0, 0)
    assert int(cur.item()) == prefix + 2
    assert torch.equal(kv[:, :, :, prefix + 1], before[:, :, :, prefix + 3])


def test_bounded_waits_expire_report_and_return():
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    mv.selftest_wait_timeout(20_000, out)   # 20 us per wait
    torch.cuda.synchronize()
    got_counter, got_mbar, counter, us = out.cpu().tolist()
    assert got_counter == 0 and got_mbar == 0 and counter == 0
    assert 40 <= us < 100_000, us            # each wait ran to its limit, and no wait ran unbounded
    st, code, det = mv.get_error(with_detail=True)
    assert st == MV_ERR_DEVICE and code == (20 << 16) | DEVERR_TIMEOUT and det == 3, (st, hex(code), det)
    assert mv.get_error() == (0, 0)          # read once, cleared
    # the context is still usable
    x = torch.arange(8, device="cuda")
    assert int(x.sum().item()) == 28


def test_selftest_rejects_unbounded_limits():
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    for bad in (0, 999, 10_000_001):
        with pytest.raises(mv.MVError) as e:
            mv.selftest_wait_timeout(bad, out)
        assert e.value.status == 1
