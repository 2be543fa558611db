"""GPU parity of octo_token_logprob (per-token log-probability, loss and gradient over
the packed rows) against the fp64 reference in oracle/token_logprob.py."""
import numpy as np
import pytest

import synth
import oracle
from oracle.token_logprob import path_predecessors, token_logprob
from helpers import assert_close, pool_pages_needed

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _plans(lib, ep, bm=128):
    """The library's pack plan of ep (a pool holding layout only) and the oracle's rows and
    predecessors, from the oracle's own replay and pack."""
    pool = lib.Pool(pool_pages_needed(ep), ep.page_size, 1, 64, lib.DTYPE_BF16)
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
    plan = pool.pack_tree(ep.roots, bm)
    orc = oracle.Oracle(ep.page_size, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, bm, tile_stride=1 << 30)    # rows only: no tile derivation
    mine = plan.copy_out()
    assert np.array_equal(mine["seg_order"], opl.seg_order)
    assert np.array_equal(mine["seg_row_base"], opl.seg_row_base)
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, opl.n_rows)
    return pool, plan, pred


def _inputs(N, V, ld, dtype, seed):
    rng = np.random.default_rng(seed)
    x = np.full((N, ld), np.nan, dtype=np.float32)          # padding columns must not be read
    x[:, :V] = rng.normal(0, 3.0, (N, V))
    ids = rng.integers(0, V, N).astype(np.int32)
    w = rng.uniform(-1, 1, N).astype(np.float32)
    w[rng.random(N) < 0.2] = 0.0                              # untrainable tokens (mask 0)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    xt = torch.from_numpy(x).to(tdt).cuda()
    xr = xt.float().cpu().numpy()[:, :V].astype(np.float64)   # the logits as the kernel sees them
    return xt, xr, ids, w


def _run(lib, plan, xt, V, ids, w, row0=0, n=None, dlogits="sep", stream=None):
    n = plan.info["n_rows"] - row0 if n is None else n
    N = plan.info["n_rows"]
    ids_d = torch.from_numpy(ids).cuda()
    w_d = None if w is None else torch.from_numpy(w).cuda()
    logp = torch.full((N,), -7.0, dtype=torch.float32, device="cuda")
    lse = torch.empty(max(n, 1), dtype=torch.float32, device="cuda")
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.token_logprob_workspace_size(n), 1), dtype=torch.uint8, device="cuda")
    g = None if dlogits is None else (xt if dlogits == "inplace" else torch.full_like(xt, float("nan")))
    plan.token_logprob(row0, n, xt, V, ids_d, w_d, logp, ws, row_lse=lse, dlogits=g, grad_scale=1.0, loss=loss)
    plan.sync()
    return logp.cpu().numpy(), lse.cpu().numpy()[:n], loss.item(), None if g is None else g.float().cpu().numpy()


@pytest.mark.parametrize("dtype,V,ld", [("f32", 997, 1000), ("bf16", 1037, 1040), ("bf16", 4096, 4096)])
@pytest.mark.parametrize("seed", [5, 19])
def test_parity_random_dags(lib, dtype, V, ld, seed):
    ep = synth.random_dag(seed, page_size=16, max_segments=16, max_len=300)
    pool, plan, pred = _plans(lib, ep)
    N = plan.info["n_rows"]
    xt, xr, ids, w = _inputs(N, V, ld, dtype, seed)
    logp, lse, loss, g = _run(lib, plan, xt, V, ids, w)
    rlogp, rlse, rloss, rg = token_logprob(xr, ids, w, pred)
    assert_close(logp, rlogp, dtype, "logp")
    assert_close(lse, rlse, dtype, "row lse")
    assert_close([loss], [rloss], dtype, "loss")
    assert_close(g[:, :V], rg, dtype, "dlogits")
    assert np.isnan(g[:, V:]).all()                             # padding columns untouched
    assert np.all(logp[pred < 0] == 0.0)


def test_fork_and_rewind_rows(lib):
    """Rows with several successors: the last prefix row feeds three children, a rewound
    child's row feeds its continuation and its dead-end tail; a mount changes nothing."""
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 150)
    a, b, c = ep.fork(r, 3)
    ep.append(a, 40)
    ep.append(b, 70)
    a2 = ep.rewind(a, 17)
    ep.append(a2, 33)
    ep.append(c, 20)
    ep.mount(c, b, 10, 60)
    ep.append(c, 45)
    pool, plan, pred = _plans(lib, ep, bm=64)
    N, V = plan.info["n_rows"], 2048
    xt, xr, ids, w = _inputs(N, V, V, "f32", 3)
    logp, lse, loss, g = _run(lib, plan, xt, V, ids, w)
    rlogp, rlse, rloss, rg = token_logprob(xr, ids, w, pred)
    assert np.bincount(pred[pred >= 0]).max() == 3
    assert_close(logp, rlogp, "f32", "logp")
    assert_close(g, rg, "f32", "dlogits")
    assert_close([loss], [rloss], "f32", "loss")


def test_chunks_and_in_place(lib):
    ep = synth.random_dag(23, page_size=16, max_segments=14, max_len=200)
    pool, plan, pred = _plans(lib, ep)
    N, V = plan.info["n_rows"], 1200
    xt, xr, ids, w = _inputs(N, V, V, "bf16", 8)
    logp, lse, loss, g = _run(lib, plan, xt.clone(), V, ids, w)
    # three ragged chunks, each with its own logits slice, give the same values
    cuts = [0, N // 3 + 1, (2 * N) // 3 + 5, N]
    lp = np.full(N, np.nan, dtype=np.float32)
    gl = np.zeros((N, V), dtype=np.float32)
    tot = 0.0
    for a, b in zip(cuts[:-1], cuts[1:]):
        lpc, _, lc, gc = _run(lib, plan, xt[a:b].contiguous(), V, ids, w, row0=a, n=b - a)
        for t in range(N):
            if (pred[t] >= a and pred[t] < b) or (pred[t] < 0 and a <= t < b):
                lp[t] = lpc[t]
        gl[a:b] = gc
        tot += lc
    assert np.array_equal(lp, logp)
    assert np.array_equal(gl, g)
    assert abs(tot - loss) <= 1e-5 * max(1.0, abs(loss))
    # the gradient written over the logits equals the one written elsewhere
    xin = xt.clone()
    logp2, _, loss2, g2 = _run(lib, plan, xin, V, ids, w, dlogits="inplace")
    assert np.array_equal(logp2, logp) and np.array_equal(g2, g) and loss2 == loss
    # no weights, no gradient: the terms alone
    logp3, _, loss3, _ = _run(lib, plan, xt, V, ids, None, dlogits=None)
    rlogp, _, rloss, _ = token_logprob(xr, ids, None, pred)
    assert_close(logp3, rlogp, "bf16", "logp (no weights)")
    assert_close([loss3], [rloss], "bf16", "loss (no weights)")


def test_bad_id_is_reported(lib):
    ep = synth.random_dag(4, page_size=16, max_segments=6, max_len=100)
    pool, plan, pred = _plans(lib, ep)
    N, V = plan.info["n_rows"], 256
    xt, xr, ids, w = _inputs(N, V, V, "f32", 1)
    t = int(np.nonzero(pred >= 0)[0][0])
    ids[t] = V                                          # out of range: checked, never read
    ids_d = torch.from_numpy(ids).cuda()
    logp = torch.zeros(N, dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.token_logprob_workspace_size(N), dtype=torch.uint8, device="cuda")
    plan.token_logprob(0, N, xt, V, ids_d, None, logp, ws)
    with pytest.raises(lib.OctoError) as e:
        plan.sync()
    assert e.value.code == lib.EINVAL
    plan.sync()                                         # the status word was cleared
    got = logp.cpu().numpy()
    assert np.isnan(got[t])
    ok = np.arange(N) != t
    rlogp, _, _, _ = token_logprob(xr, np.where(ids < V, ids, 0), None, pred)
    assert_close(got[ok], rlogp[ok], "f32", "logp of the other rows")


def test_episode_chunk_full_vocabulary(lib):
    """The bench's configuration: episode rows at a vocabulary of 151,936 (bf16), a chunk
    of 2048 rows around the end of the shared prefix (a row with 7 successors), checked on
    a sample of rows."""
    ep = synth.make_preset("episode", seed=0)
    pool, plan, pred = _plans(lib, ep)
    N, V = plan.info["n_rows"], 151936
    fork_row = int(np.argmax(np.bincount(pred[pred >= 0], minlength=N)))
    row0 = max(0, fork_row - 1024)
    n = 2048
    xt = synth.hash_fill(synth.STREAM_Q + 101, (n, V), torch.bfloat16, "cuda", 3.0, chunk_rows=512)
    rng = np.random.default_rng(0)
    ids = rng.integers(0, V, N).astype(np.int32)
    w = rng.uniform(0, 1, N).astype(np.float32)
    logp, lse, loss, g = _run(lib, plan, xt, V, ids, w, row0=row0, n=n)
    sample = sorted(set(rng.integers(0, n, 40).tolist()) | {fork_row - row0, 0, n - 1})
    xs = xt[sample].float().cpu().numpy().astype(np.float64)
    # the oracle on a sub-problem: the sampled rows as logits rows, followed by the tokens
    # they predict (as rows of their own whose logits feed nothing here)
    rows = [row0 + rl for rl in sample]
    kids = [np.nonzero(pred == r)[0] for r in rows]
    toks = np.concatenate(kids)
    k = len(rows)
    x_sub = np.zeros((k + len(toks), V))
    x_sub[:k] = xs
    pred_sub = np.full(k + len(toks), -1)
    pred_sub[k:] = np.repeat(np.arange(k), [len(c) for c in kids])
    ids_sub = np.concatenate([np.zeros(k, dtype=np.int64), ids[toks]])
    w_sub = np.concatenate([np.zeros(k), w[toks].astype(np.float64)])
    rlogp, rlse, _, rdx = token_logprob(x_sub, ids_sub, w_sub, pred_sub)
    assert_close(lse[sample], rlse[:k], "bf16", "row lse")
    assert_close(logp[toks], rlogp[k:], "bf16", "logp")
    assert_close(g[sample], rdx[:k], "bf16", "dlogits")
    assert np.bincount(pred[pred >= 0]).max() >= 7
