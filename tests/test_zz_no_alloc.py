"""octo_decode_noalloc: the decode for callers that cannot allocate device memory (their
device memory all belongs to their own allocator, or allocation is not allowed where
they run).  It uses the library's static device scratch instead of a caller workspace.

Checked through the C ABI against octo_decode (the workspace entry point) on the same
inputs, on two calls in a row (the scratch is shared and reused), within the bf16 parity
tolerance.  This file is named to be collected last."""
import math

import numpy as np
import pytest

import synth
from helpers import assert_close, replay_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _episode_pool(lib, seed):
    ep = synth.random_dag(seed, page_size=64, max_segments=16, max_len=900, n_roots=2)
    Hq, Hkv, d, P = 16, 4, 128, 64
    t = synth.make_tensors(ep, Hq, Hkv, d, "bf16", 0.5, seed, with_do=False)
    npages = sum((L + P - 1) // P for L in ep.length) + 2
    kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
    replay_device(pool, ep, torch.from_numpy(t.K).cuda().bfloat16(), torch.from_numpy(t.V).cuda().bfloat16())
    curs = [s for s in range(ep.n_segments) if ep.length[s] > 0]
    return pool, curs, Hq, d


def test_noalloc_matches_workspace_decode_twice(lib):
    pool, curs, Hq, d = _episode_pool(lib, 4242)
    scale = 1.0 / math.sqrt(d)
    plan = pool.decode_plan(curs)
    wsn = plan.decode_workspace_size(Hq)
    assert 0 < wsn <= lib.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(wsn, dtype=torch.uint8, device="cuda")
    for call in range(2):
        q = torch.from_numpy(synth.make_decode_q(len(curs), Hq, d, "bf16", 0.5, 100 + call)).cuda().bfloat16()
        ref = torch.empty_like(q)
        ref_lse = torch.empty((len(curs), Hq), dtype=torch.float32, device="cuda")
        plan.decode(Hq, q, ref, ref_lse, scale, ws, wsn)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((len(curs), Hq), float("nan"), dtype=torch.float32, device="cuda")
        plan.decode_noalloc(Hq, q, out, lse, scale)
        plan.sync()
        assert_close(out.float().cpu().numpy(), ref.float().cpu().numpy(), "bf16", "noalloc out, call %d" % call)
        assert_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), "bf16", "noalloc lse, call %d" % call)


def test_noalloc_rejects_oversized_request(lib):
    """A request larger than the static scratch fails with OCTO_ESCRATCH before launching."""
    Hq, Hkv, d, P = 64, 8, 128, 64
    n_cur, pages_per = 32, 1024
    pool = lib.Pool(n_cur * pages_per + 64, P, Hkv, d, lib.DTYPE_BF16)   # metadata only
    r = pool.root()
    pool.append(r, 1)
    kids = pool.fork(r, n_cur)
    for k in kids:
        pool.append(k, pages_per * P - 64)
    plan = pool.decode_plan(kids)
    assert plan.decode_workspace_size(Hq) > lib.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((n_cur, Hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(lib.OctoError) as e:
        plan.decode_noalloc(Hq, q, out, None, 0.1)
    assert e.value.code == lib.ESCRATCH
