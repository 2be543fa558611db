"""GPU parity: the library's plans, forward, backward and decode against the fp64 oracle
on the same seeded inputs, through the C ABI.  Plans and pool tables are compared bit for
bit; values within |err| <= 1e-5 + 1e-5|ref| (fp32 pools) or 2e-2 + 2e-2|ref| (bf16)."""
import math

import numpy as np
import pytest

import synth
from helpers import (assert_close, compare_plans, compare_pools, packed, pool_pages_needed, product_entries,
                     replay_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


class Run:
    """An episode replayed into both the oracle and the library, with its tensors."""

    def __init__(self, lib, oracle_mod, ep, Hq, Hkv, d, dtype, seed, bm=None, npages=None, with_kv=True,
                 pool_fill=0.0):
        self.ep, self.Hq, self.Hkv, self.d, self.dtype = ep, Hq, Hkv, d, dtype
        P = ep.page_size
        self.P = P
        self.npages = npages or pool_pages_needed(ep)
        self.t = synth.make_tensors(ep, Hq, Hkv, d, dtype, 1.0 if dtype == "f32" else 0.5, seed)
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        self.tdt = tdt
        dev = "cuda"
        # pool_fill: initial content of the pool arrays (NaN checks that pages a segment is
        # given are cleared before slots past its end can reach a kernel)
        self.kpool = torch.full((self.npages, Hkv, P, d), pool_fill, dtype=tdt, device=dev)
        self.vpool = torch.full_like(self.kpool, pool_fill)
        self.pool = lib.Pool(self.npages, P, Hkv, d, lib.DTYPE_F32 if dtype == "f32" else lib.DTYPE_BF16,
                             self.kpool, self.vpool)
        K = torch.from_numpy(self.t.K).to(dev).to(tdt)
        V = torch.from_numpy(self.t.V).to(dev).to(tdt)
        replay_device(self.pool, ep, K, V)
        torch.cuda.synchronize()
        self.orc = oracle_mod.Oracle(P, self.npages, Hkv, d)
        self.orc.replay(ep, self.t.K.astype(np.float64), self.t.V.astype(np.float64))
        self.scale = 1.0 / math.sqrt(d)

    def pack(self, bm, tile_stride=1):
        self.bm = bm
        self.plan = self.pool.pack_tree(self.ep.roots, bm)
        self.opl = self.orc.pack(self.ep.roots, bm, tile_stride)
        self.Q = packed(self.t, self.opl.seg_order, self.t.Q)
        self.dO = packed(self.t, self.opl.seg_order, self.t.dO)
        return self.plan, self.opl

    def dev(self, a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda().to(self.tdt)

    def fwd(self):
        N = self.plan.info["n_rows"]
        q = self.dev(self.Q)
        o = torch.empty((N, self.Hq, self.d), dtype=self.tdt, device="cuda")
        lse = torch.empty((self.Hq, N), dtype=torch.float32, device="cuda")
        self.plan.attn_fwd(self.Hq, q, o, lse, self.scale)
        self.plan.sync()
        self.q_dev, self.o_dev, self.lse_dev = q, o, lse
        return o.float().cpu().numpy(), lse.cpu().numpy()

    def bwd(self):
        N = self.plan.info["n_rows"]
        do = self.dev(self.dO)
        dq = torch.empty((N, self.Hq, self.d), dtype=torch.float32, device="cuda")
        dk = torch.full((self.npages, self.Hkv, self.P, self.d), float("nan"), device="cuda")
        dv = torch.full_like(dk, float("nan"))
        ws = torch.empty(max(1, self.plan.attn_bwd_workspace_size(self.Hq)), dtype=torch.uint8, device="cuda")
        self.plan.attn_bwd(self.Hq, self.q_dev, self.o_dev, self.lse_dev, do, dq, dk, dv, self.scale, ws)
        self.plan.sync()
        return dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy()

    def token_slots(self):
        seg, idx = self.orc.token_owner()
        pages = {s: self.orc.seg_pages(s) for s in set(seg.tolist())}
        page = np.array([pages[s][i // self.P] for s, i in zip(seg.tolist(), idx.tolist())], dtype=np.int64)
        return page, idx % self.P


# ------------------------------------------------------------------ plans, bit-exact
@pytest.mark.parametrize("seed", range(12))
def test_plan_random(lib, oracle_mod, seed):
    P = [4, 8, 16, 64][seed % 4]
    bm = [16, 32, 64, 128, 1, 48][seed % 6]
    ep = synth.random_dag(300 + seed, page_size=P, max_segments=14, max_len=[40, 90, 200][seed % 3],
                          n_roots=1 + seed % 3)
    r = Run(lib, oracle_mod, ep, 2, 1, 64, "f32", seed)
    compare_pools(r.pool, r.orc)
    plan, opl = r.pack(bm)
    compare_plans(plan.copy_out(), opl)
    assert plan.info["pairs"] == opl.pairs == opl.total_pairs()


@pytest.mark.parametrize("bm", [32, 128])
def test_plan_tiny(lib, oracle_mod, bm):
    ep = synth.make_preset("tiny")
    r = Run(lib, oracle_mod, ep, 1, 1, 64, "f32", 0)
    plan, opl = r.pack(bm)
    compare_plans(plan.copy_out(), opl)
    assert plan.info["pairs"] == 7488


def test_plan_tree_fwd_full(lib, oracle_mod):
    ep = synth.make_preset("tree_fwd")
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", 0)
    plan, opl = r.pack(128)
    compare_plans(plan.copy_out(), opl)
    assert plan.info["pairs"] == opl.pairs


@pytest.mark.parametrize("name,stride", [("episode", 7), ("decode", 97)])
def test_plan_full_size_sampled(lib, oracle_mod, name, stride):
    """Full-size episodes: every tile's layout, positions and the total pair count are
    compared; entries on a sample of tiles the oracle derives one by one."""
    ep = synth.make_preset(name, seed=0)
    r = Run(lib, oracle_mod, ep, 1, 1, 64, "f32", 0)   # K/V values do not matter for plans
    plan, opl = r.pack(128, tile_stride=stride)
    gp = plan.copy_out()
    for k in ("seg_order", "seg_row_base", "row_pos", "tile_seg", "tile_t0", "tile_rows"):
        assert np.array_equal(gp[k], getattr(opl, k)), k
    assert plan.info["pairs"] == opl.total_pairs()
    pe = product_entries(gp["entries"])
    ot = opl.tile_off
    oe = opl.entries.astype(np.int64)
    for t in range(0, len(gp["tile_rows"]), stride):
        mine = pe[gp["tile_off"][t]:gp["tile_off"][t + 1]]
        want = oe[ot[t]:ot[t + 1]]
        assert np.array_equal(mine, want), t
    # CSC: every page's list is its entries in increasing entry order
    perm, poff = gp["csc_perm"], gp["page_off"]
    assert np.array_equal(np.sort(perm), np.arange(len(perm)))
    pages = pe[perm, 1]
    assert np.all(np.diff(pages) >= 0)
    same = pages[1:] == pages[:-1]
    assert np.all(np.diff(perm)[same] > 0)
    assert np.array_equal(np.bincount(pe[:, 1], minlength=r.npages), np.diff(poff))


def test_decode_plan(lib, oracle_mod):
    ep = synth.random_dag(77, page_size=16, max_segments=14, max_len=70)
    r = Run(lib, oracle_mod, ep, 4, 2, 64, "f32", 1)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    dp = r.pool.decode_plan(curs)
    gp = dp.copy_out()
    # a decode row is the last row of its segment: its context is that row's context,
    # so its entries are the oracle's entries of a one-row tile -- compare by pairs
    opl = r.orc.pack(ep.roots, 1)
    rows = {int(s): int(b) + r.orc.seg_info(int(s))["len"] - 1 for s, b in zip(opl.seg_order, opl.seg_row_base)}
    oe = opl.entries.astype(np.int64)
    pe = product_entries(gp["entries"])
    for i, c in enumerate(curs):
        t = rows[c]           # bm = 1: tile index == packed row
        want = oe[opl.tile_off[t]:opl.tile_off[t + 1]].copy()
        mine = pe[gp["tile_off"][i]:gp["tile_off"][i + 1]].copy()
        want[:, 0] = 0
        mine[:, 0] = 0
        assert np.array_equal(mine, want), c
        assert gp["row_pos"][i] == opl.row_pos[t]


# ------------------------------------------------------------------ values
def _check_fwd_bwd(r, do_bwd=True):
    O, LSE = r.fwd()
    Oo, Lo = r.opl.fwd(r.Q.astype(np.float64), r.scale, nthreads=8)
    assert_close(O, Oo, r.dtype, "O")
    assert_close(LSE, Lo, r.dtype, "LSE")
    if not do_bwd:
        return
    dq, dk, dv = r.bwd()
    dQo, dKo, dVo = r.opl.bwd(r.Q.astype(np.float64), r.dO.astype(np.float64), r.scale, nthreads=8)
    assert_close(dq, dQo, r.dtype, "dQ")
    page, slot = r.token_slots()
    assert_close(dk[page, :, slot, :], dKo, r.dtype, "dK")
    assert_close(dv[page, :, slot, :], dVo, r.dtype, "dV")
    # slots of touched pages that hold no token read by any row are zero
    gp = r.plan.copy_out()
    touched = np.nonzero(np.diff(gp["page_off"]))[0]
    mask = np.zeros((r.npages, r.P), dtype=bool)
    mask[page, slot] = True
    for p in touched:
        for j in np.nonzero(~mask[p])[0]:
            assert np.all(dk[p, :, j] == 0) and np.all(dv[p, :, j] == 0)


def test_tiny_fp32(lib, oracle_mod):
    r = Run(lib, oracle_mod, synth.make_preset("tiny"), 1, 1, 64, "f32", 0)
    r.pack(32)
    _check_fwd_bwd(r)


@pytest.mark.parametrize("seed", range(6))
def test_random_fp32(lib, oracle_mod, seed):
    P = [8, 16][seed % 2]
    ep = synth.random_dag(400 + seed, page_size=P, max_segments=12, max_len=90, n_roots=1 + seed % 2)
    r = Run(lib, oracle_mod, ep, [2, 4][seed % 2], [1, 2][seed % 2], [64, 128][seed % 2], "f32", seed)
    r.pack([32, 16, 128][seed % 3])
    _check_fwd_bwd(r)


@pytest.mark.parametrize("seed", range(6))
def test_random_bf16_gqa(lib, oracle_mod, seed):
    """bf16, 16 q heads over 4 kv heads, head_dim 128, page 64, q-tile 128: several tiles
    per segment, ragged tails, partial pages, mounts, rewinds.  Odd seeds start from pool
    arrays full of NaN."""
    ep = synth.random_dag(500 + seed, page_size=64, max_segments=10, max_len=400, n_roots=1 + seed % 2)
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", seed, pool_fill=float("nan") if seed % 2 else 0.0)
    r.pack(128)
    _check_fwd_bwd(r)


def test_tree_fwd_sampled_rows(lib, oracle_mod):
    """The full-size bf16 tree (fwd only): all outputs computed; the oracle checks a
    seeded sample of rows, covering every segment's first, last and mounted rows."""
    ep = synth.make_preset("tree_fwd")
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", 0)
    r.pack(128)
    O, LSE = r.fwd()
    rng = np.random.default_rng(0)
    rows = set(rng.integers(0, r.plan.info["n_rows"], 48).tolist())
    for s, b in zip(r.opl.seg_order, r.opl.seg_row_base):
        L = r.orc.seg_info(int(s))["len"]
        rows.update([int(b), int(b) + L - 1, int(b) + min(L - 1, 4096)])
    rows = np.array(sorted(rows), dtype=np.int32)
    Oo, Lo = r.opl.fwd(r.Q.astype(np.float64), r.scale, rows=rows, nthreads=8)
    assert_close(O[rows], Oo[rows], "bf16", "O")
    assert_close(LSE[:, rows], Lo[:, rows], "bf16", "LSE")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_values(lib, oracle_mod, dtype):
    ep = synth.random_dag(91, page_size=16 if dtype == "f32" else 64, max_segments=14, max_len=300)
    Hq, Hkv, d = (4, 2, 64) if dtype == "f32" else (16, 4, 128)
    r = Run(lib, oracle_mod, ep, Hq, Hkv, d, dtype, 3)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    q = synth.make_decode_q(len(curs), Hq, d, dtype, 0.5, 9)
    dp = r.pool.decode_plan(curs)
    out = torch.empty((len(curs), Hq, d), dtype=r.tdt, device="cuda")
    lse = torch.empty((len(curs), Hq), dtype=torch.float32, device="cuda")
    ws_n = dp.decode_workspace_size(Hq)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    dp.decode(Hq, r.dev(q), out, lse, r.scale, ws, ws_n)
    dp.sync()
    want, wl = r.orc.decode(curs, q.astype(np.float64), r.scale)
    assert_close(out.float().cpu().numpy(), want, dtype, "decode out")
    assert_close(lse.cpu().numpy(), wl, dtype, "decode lse")


@pytest.mark.gpu
@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 4), (6, 2), (8, 2), (12, 2), (16, 2)])
def test_decode_group_sizes(lib, oracle_mod, Hq, Hkv):
    """bf16 decode for query groups of 1, 2, 3, 4, 6 and 8 heads per kv head: every head of
    a group is computed in one pass over the K/V rows, groups that are not a power of two
    padded with zero queries whose results are dropped."""
    ep = synth.random_dag(17 + Hq + Hkv, page_size=64, max_segments=12, max_len=400)
    r = Run(lib, oracle_mod, ep, Hq, Hkv, 128, "bf16", 5)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    q = synth.make_decode_q(len(curs), Hq, 128, "bf16", 0.5, 11)
    dp = r.pool.decode_plan(curs)
    assert dp.kernel_path(Hq, 2) == 2
    out = torch.empty((len(curs), Hq, 128), dtype=r.tdt, device="cuda")
    lse = torch.empty((len(curs), Hq), dtype=torch.float32, device="cuda")
    ws_n = dp.decode_workspace_size(Hq)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    dp.decode(Hq, r.dev(q), out, lse, r.scale, ws, ws_n)
    dp.sync()
    want, wl = r.orc.decode(curs, q.astype(np.float64), r.scale)
    assert_close(out.float().cpu().numpy(), want, "bf16", "decode out")
    assert_close(lse.cpu().numpy(), wl, "bf16", "decode lse")


# ------------------------------------------------------------------ mounts the episode generators never make
def _checked_dag(oracle_mod, seed, **kw):
    from helpers import mount_kinds, oracle_checked_dag
    ep = oracle_checked_dag(oracle_mod, seed, **kw)
    return ep, mount_kinds(ep)


@pytest.mark.parametrize("seed", range(600, 612))
def test_plan_checked_mounts(lib, oracle_mod, seed):
    """Plans bit-exact with the oracle on episodes with every kind of legal mount."""
    P = [4, 8, 16, 64][seed % 4]
    ep, _ = _checked_dag(oracle_mod, seed, page_size=P, max_segments=12, max_len=[40, 80, 150][seed % 3])
    r = Run(lib, oracle_mod, ep, 2, 1, 64, "f32", seed)
    compare_pools(r.pool, r.orc)
    plan, opl = r.pack([16, 32, 128, 1][seed % 4])
    compare_plans(plan.copy_out(), opl)
    assert plan.info["pairs"] == opl.total_pairs()


@pytest.mark.parametrize("seed", [602, 603, 605, 606, 607, 609])
def test_values_checked_mounts(lib, oracle_mod, seed):
    """fp32 (CUDA-core kernels) and bf16 (tensor-core kernels, 16 q / 4 kv heads, d 128,
    page 64) forward and backward against the oracle on those episodes."""
    ep, _ = _checked_dag(oracle_mod, seed, page_size=16, max_segments=12, max_len=80)
    r = Run(lib, oracle_mod, ep, 4, 2, 64, "f32", seed)
    r.pack(32)
    _check_fwd_bwd(r)
    ep, _ = _checked_dag(oracle_mod, seed, page_size=64, max_segments=12, max_len=300)
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", seed)
    r.pack(128)
    assert r.plan.kernel_path(16, 0) == 1 and r.plan.kernel_path(16, 1) == 1
    _check_fwd_bwd(r)


def test_decode_checked_mounts(lib, oracle_mod):
    ep, _ = _checked_dag(oracle_mod, 607, page_size=64, max_segments=12, max_len=300)
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", 2)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    q = synth.make_decode_q(len(curs), 16, 128, "bf16", 0.5, 3)
    dp = r.pool.decode_plan(curs)
    out = torch.empty((len(curs), 16, 128), dtype=r.tdt, device="cuda")
    lse = torch.empty((len(curs), 16), dtype=torch.float32, device="cuda")
    ws_n = dp.decode_workspace_size(16)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    dp.decode(16, r.dev(q), out, lse, r.scale, ws, ws_n)
    dp.sync()
    want, wl = r.orc.decode(curs, q.astype(np.float64), r.scale)
    assert_close(out.float().cpu().numpy(), want, "bf16", "decode out")
    assert_close(lse.cpu().numpy(), wl, "bf16", "decode lse")


# ------------------------------------------------------------------ heavily shared prefix pages
def _shared_prefix_episode(seed, prefix=1024, branches=7):
    """A prefix forked into 7 branches of 1.5-2K tokens that mount spans of each other:
    the prefix pages are read by every query tile of every branch (over 100 reader tiles
    each), the mounted pages by their owner's tiles and the readers'."""
    rng = np.random.default_rng(seed)
    ep = synth.Episode(64)
    r = ep.root()
    ep.append(r, prefix)
    kids = ep.fork(r, branches)
    want = {k: int(rng.integers(1536, 2049)) for k in kids}
    for rnd in range(8):
        for k in kids:
            ep.append(k, want[k] // 8)
        if rnd in (3, 5):
            for k in kids[:4]:
                p = kids[(kids.index(k) + 1 + rnd) % branches]
                if ep.can_mount(k, p) and ep.length[p] >= 256:
                    a = int(rng.integers(0, ep.length[p] - 192))
                    ep.mount(k, p, a, a + int(rng.integers(64, min(640, ep.length[p] - a) + 1)))
    return ep


def test_shared_prefix_every_dk_dv(lib, oracle_mod):
    """Tensor-core path, 2 query heads over 1 kv head, d 128, page 64, q-tile 128: every
    element of O, LSE, dQ, dK and dV against the oracle, where each prefix page's dK/dV is
    an ordered sum over more than 100 reader tiles."""
    ep = _shared_prefix_episode(5)
    r = Run(lib, oracle_mod, ep, 2, 1, 128, "bf16", 6)
    plan, _ = r.pack(128)
    assert plan.kernel_path(2, 0) == 1 and plan.kernel_path(2, 1) == 1
    gp = plan.copy_out()
    readers = np.diff(gp["page_off"])
    prefix_pages = r.orc.seg_pages(0)
    assert readers[prefix_pages].min() >= 100, readers[prefix_pages]
    assert any(e[7] >= 0 for e in product_entries(gp["entries"]))   # mounted spans are read
    _check_fwd_bwd(r)


def test_decode_cursors_one_call(lib, oracle_mod):
    """octo_decode_cursors (plan, decode and release in one call; with and without a caller
    workspace) equals the plan-based decode bit for bit and the oracle within tolerance."""
    ep = synth.random_dag(93, page_size=64, max_segments=14, max_len=300)
    r = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", 3)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    q = r.dev(synth.make_decode_q(len(curs), 16, 128, "bf16", 0.5, 12))
    dp = r.pool.decode_plan(curs)
    ref = torch.empty_like(q)
    ref_lse = torch.empty((len(curs), 16), dtype=torch.float32, device="cuda")
    ws_n = dp.decode_workspace_size(16)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    dp.decode(16, q, ref, ref_lse, r.scale, ws, ws_n)
    for w in (ws, None):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((len(curs), 16), float("nan"), dtype=torch.float32, device="cuda")
        r.pool.decode_cursors(curs, 16, q, out, lse, r.scale, w, ws_n if w is not None else 0)
        torch.cuda.synchronize()
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    want, wl = r.orc.decode(curs, q.float().cpu().numpy().astype(np.float64), r.scale)
    assert_close(out.float().cpu().numpy(), want, "bf16", "decode out")
    assert_close(lse.cpu().numpy(), wl, "bf16", "decode lse")


@pytest.mark.parametrize("rope", [0.0, 10000.0])
def test_append_step_writes_like_single_appends(lib, oracle_mod, rope):
    """octo_append_step with K/V rows (bf16, plain and rotated) writes the pool arrays bit
    for bit as one-token octo_append / octo_append_rope calls on a twin pool do."""
    ep = synth.random_dag(33, page_size=16, max_segments=10, max_len=60)
    Hkv, d, P = 2, 64, 16
    npages = pool_pages_needed(ep) + 40
    pools = []
    for _ in range(2):
        kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
        vp = torch.zeros_like(kp)
        pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
        from helpers import replay_host
        replay_host(pool, ep)
        pools.append((pool, kp, vp))
    curs = [s for s in range(ep.n_segments) if ep.appendable[s]]
    rng = np.random.default_rng(4)
    for step in range(20):
        k = torch.from_numpy(rng.normal(0, 1, (len(curs), Hkv, d)).astype(np.float32)).cuda().bfloat16()
        v = torch.from_numpy(rng.normal(0, 1, (len(curs), Hkv, d)).astype(np.float32)).cuda().bfloat16()
        a = pools[0][0].append_step(curs, k, v, rope_base=rope)
        b = []
        for i, c in enumerate(curs):
            if rope:
                b.append(int(pools[1][0].append_rope(c, 1, k[i:i + 1], v[i:i + 1], rope)[0]))
            else:
                b.append(int(pools[1][0].append(c, 1, k[i:i + 1], v[i:i + 1])[0]))
        assert a.tolist() == b
    torch.cuda.synchronize()
    assert torch.equal(pools[0][1], pools[1][1]) and torch.equal(pools[0][2], pools[1][2])
    for s in range(ep.n_segments):
        assert np.array_equal(pools[0][0].seg_pages(s), pools[1][0].seg_pages(s))


@pytest.mark.parametrize("dtype,Hq,Hkv,d,P", [("bf16", 4, 2, 128, 64), ("f32", 2, 1, 64, 16)])
def test_backward_repeat_over_a_dirty_workspace_is_bit_exact(lib, oracle_mod, dtype, Hq, Hkv, d, P):
    """A second backward over a workspace whose every byte was set to 0xFF (a NaN pattern)
    gives the first one's dQ, dK, dV bit for bit: the readers of shared pages are summed in
    a fixed order (no atomics) and no kernel reads workspace it has not written in the call.
    bf16 with d 128 and pages of 64 runs the tensor-core kernels, fp32 the CUDA-core ones."""
    ep = synth.random_dag(905, page_size=P, max_segments=12, max_len=300, n_roots=2)
    r = Run(lib, oracle_mod, ep, Hq, Hkv, d, dtype, 9)
    plan, _ = r.pack(128)
    assert plan.kernel_path(Hq, 1) == (1 if dtype == "bf16" else 0)
    r.fwd()
    N = plan.info["n_rows"]
    do = r.dev(r.dO)
    ws = torch.empty(max(1, plan.attn_bwd_workspace_size(Hq)), dtype=torch.uint8, device="cuda")
    outs = []
    for fill in (0, 255):
        ws.fill_(fill)
        dq = torch.empty((N, Hq, d), dtype=torch.float32, device="cuda")
        dk = torch.zeros((r.npages, Hkv, r.P, d), device="cuda")
        dv = torch.zeros_like(dk)
        plan.attn_bwd(Hq, r.q_dev, r.o_dev, r.lse_dev, do, dq, dk, dv, r.scale, ws)
        plan.sync()
        outs.append((dq, dk, dv))
    for name, x, y in zip(("dQ", "dK", "dV"), outs[0], outs[1]):
        assert torch.isfinite(x).all(), name
        assert torch.equal(x, y), name


def test_decode_repeat_over_a_dirty_workspace_is_bit_exact(lib, oracle_mod):
    """Split-KV decode twice, the second time over a workspace whose every byte was set to
    0xFF: the same output and LSE bit for bit (every split's partial is written before the
    combine reads it, and the combine merges them in split order)."""
    ep = synth.random_dag(933, page_size=64, max_segments=14, max_len=500, n_roots=2)
    r = Run(lib, oracle_mod, ep, 8, 2, 128, "bf16", 4)
    curs = [s for s in range(r.orc.n_segments) if r.orc.seg_info(s)["len"] > 0]
    q = r.dev(synth.make_decode_q(len(curs), 8, 128, "bf16", 0.5, 13))
    dp = r.pool.decode_plan(curs)
    assert dp.kernel_path(8, 2) == 2
    ws_n = dp.decode_workspace_size(8)
    ws = torch.empty(max(ws_n, 1), dtype=torch.uint8, device="cuda")
    outs = []
    for fill in (0, 255):
        ws.fill_(fill)
        out = torch.empty((len(curs), 8, 128), dtype=r.tdt, device="cuda")
        lse = torch.empty((len(curs), 8), dtype=torch.float32, device="cuda")
        dp.decode(8, q, out, lse, r.scale, ws, ws_n)
        dp.sync()
        outs.append((out, lse))
    assert torch.isfinite(outs[0][0].float()).all() and torch.isfinite(outs[0][1]).all()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
