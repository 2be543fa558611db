"""Edge cases of the GPU path against the oracle: empty plans on every call, a single
token, the largest page size, the deepest ancestor chain the compiler walks (and one
deeper, refused), segments ending exactly on tile and page boundaries, one-token
segments, and the degenerate gates of the recurrent layer."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import recurrent
from oracle.token_logprob import path_predecessors
from helpers import compare_plans, pool_pages_needed, replay_host
from test_gpu_parity import Run, _check_fwd_bwd

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def test_empty_plans_run_no_work(lib):
    """A root without tokens packs to an empty plan; every call on it succeeds and writes
    nothing; a decode plan over no cursors likewise."""
    kp = torch.zeros((4, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    pool = lib.Pool(4, 64, 1, 128, lib.DTYPE_BF16, kp, torch.zeros_like(kp))
    r = pool.root()
    plan = pool.pack_tree([r], 128)
    info = plan.info
    assert info["n_rows"] == info["n_tiles"] == info["n_entries"] == info["pairs"] == 0
    assert info["n_rec_runs"] == info["n_rec_chunks"] == 0
    x = torch.full((1, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((2, 1), 7.0, device="cuda")
    plan.attn_fwd(2, x, x, lse, 0.1)
    ws = torch.empty(max(plan.attn_bwd_workspace_size(2), 1), dtype=torch.uint8, device="cuda")
    dq = torch.full((1, 2, 128), 7.0, device="cuda")
    dk = torch.full((4, 1, 64, 128), 7.0, device="cuda")
    plan.attn_bwd(2, x, x, lse, x, dq, dk, dk.clone(), 0.1, ws)
    f = torch.full((1, 2, 128), 7.0, device="cuda")
    g = torch.full((1, 2), 0.5, device="cuda")
    rws = torch.empty(max(plan.recurrent_workspace_size(2, 128), 1), dtype=torch.uint8, device="cuda")
    plan.recurrent_fwd(2, 128, f, f, f, g, g, f.clone(), rws)
    plan.recurrent_bwd(2, 128, f, f, f, g, g, f, f.clone(), f.clone(), f.clone(), g.clone(), g.clone(), rws)
    plan.sync()
    assert torch.all(x == 7.0) and torch.all(lse == 7.0) and torch.all(dq == 7.0) and torch.all(dk == 7.0)
    dp = pool.decode_plan([])
    assert dp.info["n_rows"] == 0
    dp.decode(2, x[:0], x[:0], lse[:0], 0.1)
    dp.sync()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_token(lib, oracle_mod, dtype):
    """One token: its only key is itself (probability 1, O = V, dQ = dK = 0, dV = dO)."""
    ep = synth.Episode(16 if dtype == "f32" else 64)
    r = ep.root()
    ep.append(r, 1)
    H = (2, 1, 64) if dtype == "f32" else (16, 4, 128)
    run = Run(lib, oracle_mod, ep, H[0], H[1], H[2], dtype, 3)
    run.pack(128 if dtype == "bf16" else 16)
    if dtype == "bf16":
        assert run.plan.kernel_path(16, 0) == 1 and run.plan.kernel_path(16, 1) == 1
    _check_fwd_bwd(run)


def test_largest_page_size(lib, oracle_mod):
    """Page size 128 (the largest a pool takes) on the CUDA-core kernels, fp32."""
    ep = synth.random_dag(71, page_size=128, max_segments=10, max_len=300)
    run = Run(lib, oracle_mod, ep, 4, 2, 64, "f32", 7)
    plan, opl = run.pack(64)
    from helpers import compare_pools
    compare_pools(run.pool, run.orc)
    compare_plans(plan.copy_out(), opl)
    _check_fwd_bwd(run)


def _chain(depth, P=16, n=3):
    ep = synth.Episode(P)
    c = ep.root()
    ep.append(c, n)
    for _ in range(depth - 1):
        c, = ep.fork(c, 1)
        ep.append(c, n)
    return ep


def test_deepest_chain_and_one_deeper(lib, oracle_mod):
    """64 segments on one path (the deepest the compiler walks) match the oracle; one more
    makes the pack return OCTO_ENOTSUP instead of a wrong plan."""
    ep = _chain(64)
    run = Run(lib, oracle_mod, ep, 2, 1, 64, "f32", 1)
    plan, opl = run.pack(16)
    compare_plans(plan.copy_out(), opl)
    _check_fwd_bwd(run)
    ep = _chain(65)
    pool = lib.Pool(pool_pages_needed(ep), 16, 1, 64, lib.DTYPE_F32)
    replay_host(pool, ep)
    with pytest.raises(lib.OctoError) as e:
        pool.pack_tree(ep.roots, 16)
    assert e.value.code == lib.ENOTSUP


def test_tile_and_page_boundaries(lib, oracle_mod):
    """bf16 tensor-core path with every length on a tile (128) or page (64) boundary, or one
    past it: forks at the end of full tiles, mounts of whole pages, one-row tiles."""
    ep = synth.Episode(64)
    r = ep.root()
    ep.append(r, 256)
    a, b, c = ep.fork(r, 3)
    ep.append(a, 128)
    ep.append(b, 64)
    ep.mount(b, a, 0, 64)
    ep.append(b, 65)
    ep.append(c, 1)
    ep.mount(c, a, 64, 128)
    ep.append(c, 127)
    d, = ep.fork(c, 1)
    ep.append(d, 129)
    run = Run(lib, oracle_mod, ep, 16, 4, 128, "bf16", 9)
    plan, opl = run.pack(128)
    compare_plans(plan.copy_out(), opl)
    _check_fwd_bwd(run)


def test_recurrent_degenerate_gates(lib):
    """alpha = 1, beta = 0 everywhere: the state never leaves 0, so every output and every
    gradient but dbeta is exactly 0; dbeta_t = (G_t k_t) . v_t with G the state gradient,
    here from the oracle.  One-token segments and forks at point 0 included."""
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 70)
    kids = ep.fork(r, 3)
    for i, k in enumerate(kids):
        ep.append(k, [1, 0, 65][i])
    e, = ep.fork(kids[1], 1)
    ep.append(e, 2)
    pool = lib.Pool(pool_pages_needed(ep), 16, 1, 64, lib.DTYPE_F32)
    replay_host(pool, ep)
    plan = pool.pack_tree(ep.roots, 128)
    orc = oracle.Oracle(16, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, 128, tile_stride=1 << 30)
    N, H, D = opl.n_rows, 2, 64
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, N)
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.normal(0, 1, (N, H, D)).astype(np.float32) for _ in range(4))
    a = np.ones((N, H), np.float32)
    b = np.zeros((N, H), np.float32)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    o = torch.full((N, H, D), float("nan"), device="cuda")
    ws = torch.empty(plan.recurrent_workspace_size(H, D), dtype=torch.uint8, device="cuda")
    plan.recurrent_fwd(H, D, dev(q), dev(k), dev(v), dev(a), dev(b), o, ws)
    grads = [torch.full((N, H, D), float("nan"), device="cuda") for _ in range(3)] + \
        [torch.full((N, H), float("nan"), device="cuda") for _ in range(2)]
    plan.recurrent_bwd(H, D, dev(q), dev(k), dev(v), dev(a), dev(b), dev(do), *grads, ws)
    plan.sync()
    assert torch.all(o == 0)
    for g in grads[:4]:
        assert torch.all(g == 0)
    ref = recurrent.backward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                             a.astype(np.float64), b.astype(np.float64), pred, do.astype(np.float64))
    assert np.all(ref[3] == 0)
    got, want = grads[4].cpu().numpy().astype(np.float64), ref[4]
    assert np.all(np.abs(got - want) <= 2e-4 + 2e-4 * np.abs(want)), np.abs(got - want).max()
