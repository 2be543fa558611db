"""GPU parity of the tree-packed recurrent layer (octo_recurrent_fwd / octo_recurrent_bwd,
the gated delta rule over the packed DAG) against the fp64 reference in
oracle/recurrent.py, through the C ABI.

Inputs follow the recipe of the oracle's pins: q, v ~ N(0, 1), unit-norm keys, alpha
U[0.6, 1], beta U[0, 1], dO ~ N(0, 1), fp32.  The kernels compute in fp32 (chunks of 64
rows, products of length <= 128 accumulated in fp32, the chunk's triangular inverse by
substitution); the tolerance |err| <= 2e-4 + 2e-4 |ref| allows about 3,000 fp32 roundings
(2^-24 each) of O(1) terms per output, the products' lengths times a margin for the
state carried across chunks, whose gates (alpha <= 1) do not amplify it."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import recurrent
from oracle.token_logprob import path_predecessors
from helpers import oracle_checked_dag, pool_pages_needed, replay_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = RTOL = 2e-4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), "%s: %d of %d outside tolerance; worst err %g at ref %g (max |ref| %g)" % (
        what, int(bad.sum()), bad.size, float(err.max()), float(ref.flat[np.argmax(err - bound)]),
        float(np.abs(ref).max()))


def _inputs(N, H, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.normal(0, 1, (N, H, D)).astype(np.float32)
    k = rng.normal(0, 1, (N, H, D))
    k = (k / np.linalg.norm(k, axis=2, keepdims=True)).astype(np.float32)
    v = rng.normal(0, 1, (N, H, D)).astype(np.float32)
    a = rng.uniform(0.6, 1.0, (N, H)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, (N, H)).astype(np.float32)
    do = rng.normal(0, 1, (N, H, D)).astype(np.float32)
    return q, k, v, a, b, do


def _setup(lib, ep):
    pool = lib.Pool(pool_pages_needed(ep), ep.page_size, 1, 64, lib.DTYPE_F32)
    replay_host(pool, ep)
    plan = pool.pack_tree(ep.roots, 128)
    orc = oracle.Oracle(ep.page_size, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, 128, tile_stride=1 << 30)
    mine = plan.copy_out()
    assert np.array_equal(mine["seg_order"], opl.seg_order)
    assert np.array_equal(mine["seg_row_base"], opl.seg_row_base)
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, opl.n_rows)
    return pool, plan, pred


def _run(lib, plan, H, D, q, k, v, a, b, do):
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    N = q.shape[0]
    tq, tk, tv, ta, tb, tdo = (dev(x) for x in (q, k, v, a, b, do))
    o = torch.full((N, H, D), float("nan"), device="cuda")
    ws = torch.empty(plan.recurrent_workspace_size(H, D), dtype=torch.uint8, device="cuda")
    plan.recurrent_fwd(H, D, tq, tk, tv, ta, tb, o, ws)
    g = [torch.full((N, H, D), float("nan"), device="cuda") for _ in range(3)]
    g += [torch.full((N, H), float("nan"), device="cuda") for _ in range(2)]
    plan.recurrent_bwd(H, D, tq, tk, tv, ta, tb, tdo, *g, ws)
    plan.sync()
    return o.cpu().numpy(), [x.cpu().numpy() for x in g]


def _check(lib, ep, H, D, seed):
    pool, plan, pred = _setup(lib, ep)
    N = plan.info["n_rows"]
    q, k, v, a, b, do = _inputs(N, H, D, seed)
    o, grads = _run(lib, plan, H, D, q, k, v, a, b, do)
    f64 = lambda x: x.astype(np.float64)
    o_ref, _ = recurrent.forward(f64(q), f64(k), f64(v), f64(a), f64(b), pred)
    _close(o, o_ref, "o")
    ref = recurrent.backward(f64(q), f64(k), f64(v), f64(a), f64(b), pred, f64(do))
    for name, got, want in zip(("dq", "dk", "dv", "dalpha", "dbeta"), grads, ref):
        _close(got, want, name)
    return plan


@pytest.mark.parametrize("seed", range(6))
def test_random_dags(lib, seed):
    """Forks, rewinds (continuations at any point, dead-end tails kept), mounts (which the
    recurrence skips), zero-length segments, runs of several chunks with ragged tails."""
    ep = synth.random_dag(800 + seed, page_size=16, max_segments=14, max_len=[90, 200, 400][seed % 3],
                          n_roots=1 + seed % 2)
    D = [64, 128][seed % 2]
    plan = _check(lib, ep, 2, D, seed)
    assert plan.info["n_rows"] > 0


@pytest.mark.parametrize("seed", [603, 607])
def test_checked_mount_dags(lib, oracle_mod, seed):
    """Episodes with an ancestor's post-fork span and repeated producers mounted: mounts
    never enter the recurrence, whatever their kind."""
    ep = oracle_checked_dag(oracle_mod, seed, page_size=16, max_segments=12, max_len=150)
    _check(lib, ep, 3, 64, seed)


def test_fork_and_rewind_on_chunk_boundaries(lib):
    """A 256-row prefix (four whole chunks) forked at its end and at row 128 (a chunk
    boundary inside a run), a rewind to row 64 of a child, and forks at point 0."""
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 128)
    a, = ep.fork(r, 1)                 # continues from row 127 of the root
    ep.append(r, 128)
    b, c = ep.fork(r, 2)               # from the root's last row
    ep.append(a, 100)
    ep.append(b, 192)
    d = ep.rewind(b, 64)               # continuation from row 63 of b
    ep.append(d, 70)
    e, = ep.fork(c, 1)                 # c has no own rows yet: e continues from the root
    ep.append(e, 65)
    ep.append(c, 1)
    _check(lib, ep, 2, 128, 3)


def test_single_sequence_matches_flat_recurrence(lib):
    """One segment of 300 rows: the plain gated delta rule, row by row."""
    ep = synth.Episode(64)
    r = ep.root()
    ep.append(r, 300)
    _check(lib, ep, 4, 64, 11)


def test_episode_sampled_rows(lib):
    """The bench's shape: the episode DAG (245,760 rows), 16 heads, head_dim 128.  The whole
    forward runs; the oracle's recurrence replays the paths of sampled rows (segment starts
    and ends, rows right after a fork or rewind point) for one head each."""
    ep = synth.make_preset("episode", seed=0)
    pool = lib.Pool(pool_pages_needed(ep), 64, 1, 64, lib.DTYPE_F32)
    replay_host(pool, ep)
    plan = pool.pack_tree(ep.roots, 128)
    orc = oracle.Oracle(64, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, 128, tile_stride=1 << 30)
    N, H, D = opl.n_rows, 16, 128
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, N)
    gen = lambda s, shape, sc: synth.hash_fill(s, shape, torch.float32, "cuda", sc)
    q = gen(201, (N, H, D), 1.0)
    k = gen(202, (N, H, D), 1.0)
    k = k / k.norm(dim=2, keepdim=True)
    v = gen(203, (N, H, D), 1.0)
    a = 0.6 + 0.4 * torch.rand((N, H), generator=torch.Generator("cuda").manual_seed(5), device="cuda")
    b = torch.rand((N, H), generator=torch.Generator("cuda").manual_seed(6), device="cuda")
    o = torch.empty_like(q)
    ws = torch.empty(plan.recurrent_workspace_size(H, D), dtype=torch.uint8, device="cuda")
    plan.recurrent_fwd(H, D, q, k, v, a, b, o, ws)
    plan.sync()
    rows = set()
    for s_, b0 in zip(opl.seg_order.tolist(), opl.seg_row_base.tolist()):
        L = orc.seg_info(s_)["len"]
        if L:
            rows.update([b0, b0 + L - 1, b0 + min(L - 1, 100)])
    rng = np.random.default_rng(0)
    rows = sorted(rng.choice(sorted(rows), size=6, replace=False).tolist())
    for i, r in enumerate(rows):
        h = i % H
        path = []
        x = r
        while x >= 0:
            path.append(x)
            x = int(pred[x])
        path = np.array(path[::-1])
        idx = torch.from_numpy(path).cuda()
        qs, ks, vs = (t[idx, h].double().cpu().numpy() for t in (q, k, v))
        as_, bs = (t[idx, h].double().cpu().numpy() for t in (a, b))
        S = np.zeros((D, D))
        for t in range(len(path)):
            S = as_[t] * (S - bs[t] * np.outer(S @ ks[t], ks[t])) + bs[t] * np.outer(vs[t], ks[t])
        _close(o[r, h].cpu().numpy(), S @ qs[-1], "o row %d head %d (path of %d rows)" % (r, h, len(path)))


@pytest.mark.parametrize("D", [64, 128])
def test_repeat_over_a_dirty_workspace_is_bit_exact(lib, D):
    """Deterministic and independent of what the workspace held: a second forward +
    backward, after every workspace byte is set to 0xFF (a NaN pattern), gives the same
    outputs bit for bit.  Runs ending at a fork point sum the start gradients of their
    continuations in run order, never by atomics, and no kernel reads a workspace entry
    that the call has not written."""
    ep = synth.random_dag(811 + D, page_size=16, max_segments=14, max_len=200, n_roots=2)
    pool, plan, _ = _setup(lib, ep)
    N, H = plan.info["n_rows"], 3
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    tq, tk, tv, ta, tb, tdo = (dev(x) for x in _inputs(N, H, D, 5))
    ws = torch.zeros(plan.recurrent_workspace_size(H, D), dtype=torch.uint8, device="cuda")
    outs = []
    for fill in (0, 255):
        ws.fill_(fill)
        o = torch.empty((N, H, D), device="cuda")
        g = [torch.empty((N, H, D), device="cuda") for _ in range(3)] + [torch.empty((N, H), device="cuda") for _ in range(2)]
        plan.recurrent_fwd(H, D, tq, tk, tv, ta, tb, o, ws)
        plan.recurrent_bwd(H, D, tq, tk, tv, ta, tb, tdo, *g, ws)
        plan.sync()
        outs.append([o] + g)
    for name, x, y in zip(("o", "dq", "dk", "dv", "dalpha", "dbeta"), outs[0], outs[1]):
        assert torch.isfinite(x).all(), name
        assert torch.equal(x, y), name
