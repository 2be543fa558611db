"""Host-side tests (no GPU): the C-ABI library loads and exports every symbol the
header declares, and its pool metadata (pages, refcounts, positions, cursor states,
error codes) matches the oracle's independent model bit for bit."""
import numpy as np
import pytest

import synth
from helpers import compare_pools, header_param_counts, header_symbols, replay_host


@pytest.fixture(scope="module")
def lib():
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def test_exports_every_header_symbol(lib):
    L = lib.load()
    syms = header_symbols()
    assert len(syms) >= 20
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) == set(lib.SYMBOLS)


def test_binding_argument_counts_match_header(lib):
    """Every ctypes signature of the binding has as many arguments as the declaration."""
    L = lib.load()
    counts = header_param_counts()
    assert set(counts) == set(lib.SYMBOLS)
    for name, n in counts.items():
        argtypes = getattr(L, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes)


def test_tensor_arguments_must_be_dense(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros((4, 6))
    assert lib._ptr(x) == x.data_ptr()
    assert lib._ptr(x[1:3]) == x[1:3].data_ptr()          # leading-row slices stay dense
    for bad in (x.t(), x[:, :5], x[::2]):
        with pytest.raises(ValueError):
            lib._ptr(bad)


def test_strerror(lib):
    L = lib.load()
    for code in range(7):
        assert L.octo_strerror(code)


@pytest.mark.parametrize("seed", range(25))
def test_pool_matches_oracle(lib, oracle_mod, seed):
    ep = synth.random_dag(seed, page_size=[4, 8, 16][seed % 3], max_segments=12, max_len=60,
                          n_roots=1 + seed % 2)
    npages = sum((L + ep.page_size - 1) // ep.page_size for L in ep.length) + 3
    pool = lib.Pool(npages, ep.page_size, 2, 64, lib.DTYPE_F32)
    orc = oracle_mod.Oracle(ep.page_size, npages, 2, 64)
    replay_host(pool, ep)
    orc.replay(ep)
    compare_pools(pool, orc)
    # now release everything in a seeded order, comparing after each step
    rng = np.random.default_rng(seed)
    live = [s for s in range(orc.n_segments) if orc.seg_info(s)["flags"] & 1]
    rng.shuffle(live)
    for c in live:
        assert pool.release(c, check=False) == orc.release(c, check=False)
        compare_pools(pool, orc)
    pinned = [s for s in range(orc.n_segments) if orc.seg_info(s)["flags"] & 2]
    for c in pinned:
        assert pool.unpin(c, check=False) == orc.unpin(c, check=False)
        compare_pools(pool, orc)
    assert pool.info()["free_pages"] == npages


def test_presets_match_oracle(lib, oracle_mod):
    for name in ("tiny", "tree_fwd", "episode", "decode"):
        ep = synth.make_preset(name, seed=1)
        npages = sum((L + ep.page_size - 1) // ep.page_size for L in ep.length) + 1
        pool = lib.Pool(npages, ep.page_size, 1, 64, lib.DTYPE_F32)
        orc = oracle_mod.Oracle(ep.page_size, npages, 1, 64)
        replay_host(pool, ep)
        orc.replay(ep)
        compare_pools(pool, orc)


def test_error_codes_match_oracle(lib, oracle_mod):
    """Invalid operations give the same status on both sides and change nothing."""
    rng = np.random.default_rng(0)
    for trial in range(40):
        ep = synth.random_dag(1000 + trial, page_size=4, max_segments=8, max_len=20)
        npages = sum((L + 3) // 4 for L in ep.length) + 2
        pool = lib.Pool(npages, 4, 1, 64, lib.DTYPE_F32)
        orc = oracle_mod.Oracle(4, npages, 1, 64)
        replay_host(pool, ep)
        orc.replay(ep)
        n = orc.n_segments
        for _ in range(30):
            kind = rng.integers(0, 6)
            c = int(rng.integers(-1, n + 1))
            if kind == 0:
                p = int(rng.integers(-1, n + 1))
                a = int(rng.integers(-2, 25)); b = int(rng.integers(-2, 25))
                r1 = pool.mount(c, p, a, b, check=False)
                r2 = orc.mount(c, p, a, b, check=False)
            elif kind == 1:
                k = int(rng.integers(-2, 25))
                r1 = pool.rewind(c, k, check=False)
                r2 = orc.rewind(c, k, check=False)
            elif kind == 2:
                nn = int(rng.integers(0, 12))
                r1 = pool.append(c, nn, check=False)
                r2 = orc.append(c, nn, check=False)
            elif kind == 3:
                r1 = pool.done(c, check=False); r2 = orc.done(c, check=False)
            elif kind == 4:
                r1 = pool.release(c, check=False); r2 = orc.release(c, check=False)
            else:
                r1 = pool.unpin(c, check=False); r2 = orc.unpin(c, check=False)
            assert r1 == r2, (kind, c, r1, r2)
            compare_pools(pool, orc)


def test_append_all_or_nothing(lib, oracle_mod):
    pool = lib.Pool(3, 4, 1, 64, lib.DTYPE_F32)
    orc = oracle_mod.Oracle(4, 3, 1, 64)
    for x in (pool, orc):
        r = x.root()
        x.append(r, 10)
    assert pool.append(0, 3, check=False) == lib.ENOMEM
    assert orc.append(0, 3, check=False) == oracle_mod.ENOMEM
    compare_pools(pool, orc)
    assert pool.append(0, 2, check=False) == lib.OK
    orc.append(0, 2)
    compare_pools(pool, orc)



@pytest.mark.parametrize("seed", range(8))
def test_pool_query_matches_oracle(lib, oracle_mod, seed):
    """octo_pool_query: every segment's refcount and page count and every page's owner
    against the oracle's allocator model, on episodes with releases and pins."""
    from helpers import oracle_checked_dag
    ep = oracle_checked_dag(oracle_mod, 700 + seed, page_size=8, max_segments=12, max_len=50)
    # release a few cursors at the end (their segments free once nothing reaches them)
    for c in range(ep.n_segments):
        if seed % 2 and c % 3 == 1:
            ep.ops.append(("release", c))
    npages = sum((L + 7) // 8 for L in ep.length) + 5
    pool = lib.Pool(npages, 8, 1, 64, lib.DTYPE_F32)
    orc = oracle_mod.Oracle(8, npages, 1, 64)
    for op in ep.ops:
        st_l = _apply(pool, op)
        st_o = _apply_oracle(orc, op)
        assert st_l == st_o, op
    q = pool.query()
    assert q["n_segments"] == orc.n_segments and q["free_pages"] == orc.free_pages()
    assert q["n_mounts"] == orc.n_mounts and q["num_pages"] == npages
    owner = np.full(npages, -1)
    for s in range(orc.n_segments):
        info = orc.seg_info(s)
        assert q["refcount"][s] == info["refcount"], s
        assert q["n_pages"][s] == info["n_pages"], s
        if not info["flags"] & 16:
            owner[orc.seg_pages(s)] = s
    assert np.array_equal(q["page_owner"], owner)
    assert int((owner < 0).sum()) == q["free_pages"]


def _apply(pool, op):
    k = op[0]
    if k == "root":
        pool.root()
        return 0
    if k == "append":
        return pool.append(op[1], op[2], check=False)
    if k == "fork":
        return pool.fork(op[1], op[2], check=False)
    if k == "mount":
        return pool.mount(*op[1:], check=False)
    if k == "rewind":
        return pool.rewind(op[1], op[2], check=False)
    if k == "done":
        return pool.done(op[1], check=False)
    if k == "release":
        return pool.release(op[1], check=False)
    raise ValueError(k)


def _apply_oracle(orc, op):
    k = op[0]
    if k == "root":
        orc.root()
        return 0
    if k == "append":
        return orc.append(op[1], op[2], check=False)
    if k == "fork":
        return orc.fork(op[1], op[2], check=False)
    if k == "mount":
        return orc.mount(*op[1:], check=False)
    if k == "rewind":
        return orc.rewind(op[1], op[2], check=False)
    if k == "done":
        return orc.done(op[1], check=False)
    if k == "release":
        return orc.release(op[1], check=False)
    raise ValueError(k)


@pytest.mark.parametrize("seed", range(4))
def test_append_step_matches_oracle(lib, oracle_mod, seed):
    """octo_append_step (one token for each of several cursors) leaves the pool as the
    oracle's one-token appends do, step after step, cursors opening pages included; refused
    calls (a cursor twice, a frozen cursor, too few pages) change nothing."""
    ep = synth.random_dag(900 + seed, page_size=4, max_segments=10, max_len=30)
    npages = sum((L + 3) // 4 for L in ep.length) + 40
    pool = lib.Pool(npages, 4, 1, 64, lib.DTYPE_F32)
    orc = oracle_mod.Oracle(4, npages, 1, 64)
    replay_host(pool, ep)
    orc.replay(ep)
    curs = [s for s in range(ep.n_segments) if ep.appendable[s]]
    assert curs
    for step in range(9):
        pos = pool.append_step(curs)
        want = [int(orc.append(c, 1)[0]) for c in curs]
        assert pos.tolist() == want
        compare_pools(pool, orc)
    before = pool.query()
    assert pool.append_step(curs + curs[:1], check=False) == lib.EINVAL
    if len(ep.roots) and not ep.appendable[ep.roots[0]]:
        assert pool.append_step([ep.roots[0]] + curs, check=False) == lib.ESTATE
    big = lib.Pool(3, 4, 1, 64, lib.DTYPE_F32)
    r = big.root()
    kids = big.fork(r, 4)
    assert big.append_step(kids, check=False) == lib.ENOMEM      # 4 pages needed, 3 free
    assert big.info()["free_pages"] == 3 and all(big.seg_info(k)["len"] == 0 for k in kids)
    after = pool.query()
    for key in ("n_segments", "free_pages", "n_mounts"):
        assert before[key] == after[key]
    assert np.array_equal(before["page_owner"], after["page_owner"])
