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


# ------------------------------------------------------------------ against the oracle
def _oracle_rows(orc, roots, curs):
    """The oracle's one-row tiles (bm = 1) of each cursor's last token: entries (q_tile
    cleared), position, and the pairs of those rows."""
    from helpers import oracle_entries
    opl = orc.pack(roots, 1)
    base = {int(s): int(b) for s, b in zip(opl.seg_order, opl.seg_row_base)}
    oe = oracle_entries(opl)
    out = []
    for c in curs:
        t = base[c] + orc.seg_info(c)["len"] - 1
        e = oe[opl.tile_off[t]:opl.tile_off[t + 1]].copy()
        e[:, 0] = 0
        out.append((e, int(opl.row_pos[t])))
    return out


def _check_against_oracle(plan, orc, roots, curs):
    from helpers import product_entries
    gp = plan.copy_out()
    pe = product_entries(gp["entries"])
    want = _oracle_rows(orc, roots, curs)
    pairs = 0
    for i, (e, pos) in enumerate(want):
        mine = pe[gp["tile_off"][i]:gp["tile_off"][i + 1]].copy()
        mine[:, 0] = 0
        assert np.array_equal(mine, e), (i, curs[i])
        assert gp["row_pos"][i] == pos, i
        pairs += int((e[:, 3] - e[:, 2]).sum())
    assert plan.info["pairs"] == pairs
    # CSC: each page's entries in increasing entry order, page offsets from the entries
    perm, poff = gp["csc_perm"], gp["page_off"]
    assert np.array_equal(np.sort(perm), np.arange(len(perm)))
    pages = pe[perm, 1]
    assert np.all(np.diff(pages) >= 0)
    same = pages[1:] == pages[:-1]
    assert np.all(np.diff(perm)[same] > 0)
    assert np.array_equal(np.bincount(pe[:, 1], minlength=len(poff) - 1), np.diff(poff))
    assert plan.info["n_touched_pages"] == int((np.diff(poff) > 0).sum())


@pytest.mark.parametrize("seed", [3, 11, 29])
def test_advance_matches_oracle_tiles(lib, oracle_mod, seed):
    """After every advance, each cursor's entries, position and the plan's pair count equal
    the oracle's brute-force one-row tile of the cursor's newest token (page size 8, so
    cursors open pages often and the general path runs with several fresh pages at once)."""
    ep = synth.random_dag(seed, page_size=8, max_segments=14, max_len=60)
    npages = pool_pages_needed(ep) + 200
    pool = lib.Pool(npages, 8, 1, 64, lib.DTYPE_BF16)
    _replay(pool, ep)
    orc = oracle_mod.Oracle(8, npages, 1, 64)
    orc.replay(ep)
    curs = [s for s in range(ep.n_segments) if ep.appendable[s] and ep.length[s] > 0]
    assert curs
    plan = pool.decode_plan(curs)
    _check_against_oracle(plan, orc, ep.roots, curs)
    for step in range(17):
        for c in curs:
            pool.append(c, 1)
            orc.append(c, 1)
        plan.advance()
        _check_against_oracle(plan, orc, ep.roots, curs)


def test_advance_fast_path_matches_oracle(lib, oracle_mod):
    """Page size 64 and three cursors: most steps open no page (the in-place update) and a
    few open one (the rebuilt part); both are checked against the oracle."""
    ep = synth.Episode(64)
    r = ep.root()
    ep.append(r, 100)
    x, y, z = ep.fork(r, 3)
    ep.append(x, 10)
    ep.append(y, 62)
    ep.append(z, 20)
    ep.mount(z, x, 2, 9)
    ep.append(z, 5)
    npages = 64
    pool = lib.Pool(npages, 64, 1, 64, lib.DTYPE_BF16)
    _replay(pool, ep)
    orc = oracle_mod.Oracle(64, npages, 1, 64)
    orc.replay(ep)
    curs = [x, y, z]
    plan = pool.decode_plan(curs)
    for step in range(70):
        for c in curs:
            pool.append(c, 1)
            orc.append(c, 1)
        plan.advance()
        if step % 7 == 0 or step in (1, 2, 3, 38, 39, 40, 54, 55):
            _check_against_oracle(plan, orc, ep.roots, curs)
    _check_against_oracle(plan, orc, ep.roots, curs)
    _same(plan, pool.decode_plan(curs))


def test_advanced_decode_matches_oracle_across_streams(lib, oracle_mod):
    """bf16 split-KV decode (8 query / 2 kv heads, d 128, page 64) through a plan advanced
    70 times, each cursor one new K/V row per step; decodes alternate between two streams
    and the advance runs on the other one.  Outputs against the oracle's decode."""
    import math
    ep = synth.random_dag(41, page_size=64, max_segments=12, max_len=300)
    Hq, Hkv, d, P = 8, 2, 128, 64
    curs = [s for s in range(ep.n_segments) if ep.appendable[s] and ep.length[s] > 0]
    n = len(curs)
    steps = 70
    npages = pool_pages_needed(ep) + n * (steps // P + 2)
    t = synth.make_tensors(ep, Hq, Hkv, d, "bf16", 0.5, 4)
    kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
    from helpers import replay_device
    replay_device(pool, ep, torch.from_numpy(t.K).cuda().to(torch.bfloat16),
                  torch.from_numpy(t.V).cuda().to(torch.bfloat16))
    orc = oracle_mod.Oracle(P, npages, Hkv, d)
    orc.replay(ep, t.K.astype(np.float64), t.V.astype(np.float64))
    rng = np.random.default_rng(8)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    plan = pool.decode_plan(curs)
    scale = 1.0 / math.sqrt(d)
    for step in range(steps):
        kn = synth.round_bf16(rng.normal(0, 0.5, (n, Hkv, d)))
        vn = synth.round_bf16(rng.normal(0, 0.5, (n, Hkv, d)))
        kd = torch.from_numpy(kn).float().cuda().to(torch.bfloat16)
        vd = torch.from_numpy(vn).float().cuda().to(torch.bfloat16)
        torch.cuda.synchronize()
        for i, c in enumerate(curs):
            pool.append(c, 1, kd[i:i + 1], vd[i:i + 1])
            orc.append(c, 1, kn[i:i + 1].astype(np.float64), vn[i:i + 1].astype(np.float64))
        torch.cuda.synchronize()
        sa, sb = streams[step % 2], streams[(step + 1) % 2]
        plan.advance(stream=sb)
        if step % 10 != 9:
            continue
        q = synth.round_bf16(rng.normal(0, 0.5, (n, Hq, d)))
        qd = torch.from_numpy(q).float().cuda().to(torch.bfloat16)
        o = torch.empty_like(qd)
        lse = torch.empty((n, Hq), dtype=torch.float32, device="cuda")
        wsn = plan.decode_workspace_size(Hq)
        ws = torch.empty(max(wsn, 1), dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        plan.decode(Hq, qd, o, lse, scale, ws, wsn, stream=sa)
        plan.sync(stream=sa)
        want, wl = orc.decode(curs, q.astype(np.float64), scale)
        from helpers import assert_close
        assert_close(o.float().cpu().numpy(), want, "bf16", "decode out step %d" % step)
        assert_close(lse.cpu().numpy(), wl, "bf16", "decode lse step %d" % step)
