"""Failure path of the kernels' bounded device waits, without faulting or hanging the GPU:
octo_wait_selftest runs the same bounded mbarrier wait the tensor-core and decode kernels
use on a barrier phase nothing completes; the wait gives up after the given number of
polls, the status word reads OCTO_ETIMEOUT at the next octo_sync (which clears it), and
the next decode on the same plan and stream runs normally and gives the same result."""
import math

import numpy as np
import pytest

import synth
from helpers import pool_pages_needed, replay_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def test_expired_wait_reports_timeout_and_the_context_stays_usable(lib):
    ep = synth.random_dag(21, page_size=64, max_segments=10, max_len=300)
    Hq, Hkv, d, P = 8, 2, 128, 64
    t = synth.make_tensors(ep, Hq, Hkv, d, "bf16", 0.5, 2, with_do=False)
    npages = pool_pages_needed(ep)
    kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
    replay_device(pool, ep, torch.from_numpy(t.K).cuda().bfloat16(), torch.from_numpy(t.V).cuda().bfloat16())
    curs = [s for s in range(ep.n_segments) if ep.length[s] > 0]
    plan = pool.decode_plan(curs)
    q = torch.from_numpy(synth.make_decode_q(len(curs), Hq, d, "bf16", 0.5, 4)).cuda().bfloat16()
    wsn = plan.decode_workspace_size(Hq)
    ws = torch.empty(max(wsn, 1), dtype=torch.uint8, device="cuda")

    def decode():
        o = torch.empty_like(q)
        lse = torch.empty((len(curs), Hq), dtype=torch.float32, device="cuda")
        plan.decode(Hq, q, o, lse, 1.0 / math.sqrt(d), ws, wsn)
        return o, lse

    o1, l1 = decode()
    plan.sync()
    for polls in (1, 1000):
        plan.wait_selftest(polls)
        with pytest.raises(lib.OctoError) as e:
            plan.sync()
        assert e.value.code == lib.ETIMEOUT
        plan.sync()                        # cleared by the sync that reported it
        o2, l2 = decode()
        plan.sync()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(lib.OctoError) as e:
        plan.wait_selftest(0)
    assert e.value.code == lib.EINVAL
