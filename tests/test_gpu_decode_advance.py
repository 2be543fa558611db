"""octo_decode_plan_advance: a decode plan moved on by one token per cursor equals a
fresh octo_decode_plan on the same cursors, array for array and bit for bit."""
import numpy as np
import pytest

import synth
from helpers import pool_pages_needed

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _replay(pool, ep):
    for op in ep.ops:
        k = op[0]
        if k == "root":
            pool.root()
        elif k == "append":
            pool.append(op[1], op[2])
        elif k == "fork":
            pool.fork(op[1], op[2])
        elif k == "mount":
            pool.mount(*op[1:])
        elif k == "rewind":
            pool.rewind(op[1], op[2])
        elif k == "done":
            pool.done(op[1])


def _same(a, b):
    ia, ib = a.info, b.info
    assert ia == ib, (ia, ib)
    ca, cb = a.copy_out(), b.copy_out()
    assert ca.keys() == cb.keys()
    for k in ca:
        assert np.array_equal(ca[k], cb[k]), k


@pytest.mark.parametrize("seed", [2, 7, 13, 31])
def test_advance_equals_fresh_plan(lib, seed):
    ep = synth.random_dag(seed, page_size=16, max_segments=14, max_len=90)
    pool = lib.Pool(pool_pages_needed(ep) + 64, 16, 1, 64, lib.DTYPE_BF16)
    _replay(pool, ep)
    curs = [s for s in range(ep.n_segments) if ep.appendable[s] and ep.length[s] > 0]
    assert curs
    plan = pool.decode_plan(curs)
    for step in range(20):              # every cursor crosses a page boundary at least once
        for c in curs:
            pool.append(c, 1)
        plan.advance()
        _same(plan, pool.decode_plan(curs))


def test_mount_at_the_new_point_needs_a_fresh_plan(lib):
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 40)
    x, y = ep.fork(r, 2)
    ep.append(x, 30)
    ep.append(y, 50)
    pool = lib.Pool(64, 16, 1, 64, lib.DTYPE_BF16)
    _replay(pool, ep)
    curs = [x, y]
    plan = pool.decode_plan(curs)
    for c in curs:
        pool.append(c, 1)
    plan.advance()
    _same(plan, pool.decode_plan(curs))
    before = plan.copy_out()
    pool.mount(x, y, 0, 20)             # at x's current length: the next token of x sees it
    for c in curs:
        pool.append(c, 1)
    assert plan.advance(check=False) == lib.ESTATE
    after = plan.copy_out()             # refused before any change
    for k in before:
        assert np.array_equal(before[k], after[k]), k
    plan = pool.decode_plan(curs)       # a fresh plan moves on again
    for c in curs:
        pool.append(c, 1)
    plan.advance()
    _same(plan, pool.decode_plan(curs))
    # two tokens since the last plan: refused
    for c in curs:
        pool.append(c, 2)
    assert plan.advance(check=False) == lib.ESTATE


def test_advanced_plan_decodes_like_a_fresh_one(lib):
    """bf16, 16 query / 4 kv heads, d 128, page 64: the split-KV kernels give identical
    outputs through an advanced plan and a fresh plan of the same cursors."""
    ep = synth.random_dag(5, page_size=64, max_segments=12, max_len=400)
    Hq, Hkv, d, P = 16, 4, 128, 64
    npages = pool_pages_needed(ep) + 32
    kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
    T = ep.n_tokens
    K = synth.hash_fill(synth.STREAM_Q + 7, (T, Hkv, d), torch.bfloat16, "cuda", 0.5)
    V = synth.hash_fill(synth.STREAM_Q + 8, (T, Hkv, d), torch.bfloat16, "cuda", 0.5)
    t = 0
    for op in ep.ops:
        if op[0] == "append":
            pool.append(op[1], op[2], K[t:t + op[2]], V[t:t + op[2]])
            t += op[2]
        elif op[0] == "root":
            pool.root()
        elif op[0] == "fork":
            pool.fork(op[1], op[2])
        elif op[0] == "mount":
            pool.mount(*op[1:])
        elif op[0] == "rewind":
            pool.rewind(op[1], op[2])
        elif op[0] == "done":
            pool.done(op[1])
    curs = [s for s in range(ep.n_segments) if ep.appendable[s] and ep.length[s] > 0]
    plan = pool.decode_plan(curs)
    n = len(curs)
    for step in range(3):
        kn = synth.hash_fill(synth.STREAM_Q + 9 + step, (n, Hkv, d), torch.bfloat16, "cuda", 0.5)
        vn = synth.hash_fill(synth.STREAM_Q + 12 + step, (n, Hkv, d), torch.bfloat16, "cuda", 0.5)
        for i, c in enumerate(curs):
            pool.append(c, 1, kn[i:i + 1], vn[i:i + 1])
        plan.advance()
        fresh = pool.decode_plan(curs)
        q = synth.hash_fill(synth.STREAM_Q + 20 + step, (n, Hq, d), torch.bfloat16, "cuda", 0.5)
        outs = []
        for p in (plan, fresh):
            o = torch.empty_like(q)
            lse = torch.empty((n, Hq), dtype=torch.float32, device="cuda")
            wsn = p.decode_workspace_size(Hq)
            ws = torch.empty(max(wsn, 1), dtype=torch.uint8, device="cuda")
            p.decode(Hq, q, o, lse, 1.0 / np.sqrt(d), ws, wsn)
            p.sync()
            outs.append((o.cpu(), lse.cpu()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
