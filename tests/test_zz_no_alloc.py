"""octo_decode_noalloc: the decode for callers that cannot allocate device memory (their
device memory all belongs to their own allocator, or allocation is not allowed where
they run).  It uses the library's static device scratch instead of a caller workspace.

Checked through the C ABI against octo_decode (the workspace entry point) and against the
oracle's decode on the same inputs, on two calls in a row (the scratch is shared and
reused), within the bf16 parity tolerance; for query groups of 1, 3, 4 and 8 heads per kv
head; at the 256-cursor decode workload, whose split partials come close to the scratch
size; and a call is seen to allocate nothing (device free memory and the stream-ordered
pool's used bytes unchanged).  This file is named to be collected last."""
import ctypes
import math

import numpy as np
import pytest

import synth
from helpers import assert_close, pool_pages_needed, replay_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _episode_pool(lib, oracle_mod, seed, Hq=16, Hkv=4, max_len=900):
    ep = synth.random_dag(seed, page_size=64, max_segments=16, max_len=max_len, n_roots=2)
    d, P = 128, 64
    t = synth.make_tensors(ep, Hq, Hkv, d, "bf16", 0.5, seed, with_do=False)
    npages = pool_pages_needed(ep)
    kp = torch.zeros((npages, Hkv, P, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pool = lib.Pool(npages, P, Hkv, d, lib.DTYPE_BF16, kp, vp)
    replay_device(pool, ep, torch.from_numpy(t.K).cuda().bfloat16(), torch.from_numpy(t.V).cuda().bfloat16())
    orc = oracle_mod.Oracle(P, npages, Hkv, d)
    orc.replay(ep, t.K.astype(np.float64), t.V.astype(np.float64))
    curs = [s for s in range(ep.n_segments) if ep.length[s] > 0]
    return pool, orc, curs, (kp, vp)


def _pool_used_bytes():
    """Bytes in use in the device's default stream-ordered memory pool (cudaMallocAsync),
    read through the driver API."""
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuCtxGetDevice(ctypes.byref(dev)) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    used = ctypes.c_uint64()
    assert cu.cuMemPoolGetAttribute(pool, 7, ctypes.byref(used)) == 0   # CU_MEMPOOL_ATTR_USED_MEM_CURRENT
    return used.value


def _decode_both(lib, plan, Hq, q, scale, ws, wsn):
    n = q.shape[0]
    ref = torch.empty_like(q)
    ref_lse = torch.empty((n, Hq), dtype=torch.float32, device="cuda")
    plan.decode(Hq, q, ref, ref_lse, scale, ws, wsn)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((n, Hq), float("nan"), dtype=torch.float32, device="cuda")
    plan.decode_noalloc(Hq, q, out, lse, scale)
    plan.sync()
    return ref, ref_lse, out, lse


def test_noalloc_matches_workspace_decode_twice(lib, oracle_mod):
    pool, orc, curs, _ = _episode_pool(lib, oracle_mod, 4242)
    Hq, d = 16, 128
    scale = 1.0 / math.sqrt(d)
    plan = pool.decode_plan(curs)
    wsn = plan.decode_workspace_size(Hq)
    assert 0 < wsn <= lib.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(wsn, dtype=torch.uint8, device="cuda")
    for call in range(2):
        qn = synth.make_decode_q(len(curs), Hq, d, "bf16", 0.5, 100 + call)
        q = torch.from_numpy(qn).cuda().bfloat16()
        ref, ref_lse, out, lse = _decode_both(lib, plan, Hq, q, scale, ws, wsn)
        assert_close(out.float().cpu().numpy(), ref.float().cpu().numpy(), "bf16", "noalloc out, call %d" % call)
        assert_close(lse.cpu().numpy(), ref_lse.cpu().numpy(), "bf16", "noalloc lse, call %d" % call)
        want, wl = orc.decode(curs, qn.astype(np.float64), scale)
        assert_close(out.float().cpu().numpy(), want, "bf16", "noalloc out vs oracle, call %d" % call)
        assert_close(lse.cpu().numpy(), wl, "bf16", "noalloc lse vs oracle, call %d" % call)


def test_noalloc_allocates_nothing(lib, oracle_mod):
    """After a first call (which looks up the scratch address), further calls leave the
    device's free memory, torch's allocator and the stream-ordered pool as they were."""
    pool, orc, curs, _ = _episode_pool(lib, oracle_mod, 77)
    Hq, d = 16, 128
    plan = pool.decode_plan(curs)
    q = torch.from_numpy(synth.make_decode_q(len(curs), Hq, d, "bf16", 0.5, 5)).cuda().bfloat16()
    out = torch.empty_like(q)
    lse = torch.empty((len(curs), Hq), dtype=torch.float32, device="cuda")
    plan.decode_noalloc(Hq, q, out, lse, 0.1)
    plan.sync()
    torch.cuda.synchronize()
    before = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(), _pool_used_bytes())
    for _ in range(3):
        plan.decode_noalloc(Hq, q, out, lse, 0.1)
    plan.sync()
    torch.cuda.synchronize()
    after = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(), _pool_used_bytes())
    assert before == after, (before, after)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (12, 4), (16, 2), (8, 2)])
def test_noalloc_group_sizes(lib, oracle_mod, Hq, Hkv):
    """Groups of 1, 3, 8 and 4 query heads per kv head (3 runs padded to 4) through the
    static scratch, against the oracle and the workspace decode."""
    pool, orc, curs, _ = _episode_pool(lib, oracle_mod, 900 + Hq + Hkv, Hq=Hq, Hkv=Hkv, max_len=400)
    d = 128
    scale = 1.0 / math.sqrt(d)
    plan = pool.decode_plan(curs)
    wsn = plan.decode_workspace_size(Hq)
    ws = torch.empty(max(wsn, 1), dtype=torch.uint8, device="cuda")
    qn = synth.make_decode_q(len(curs), Hq, d, "bf16", 0.5, 3)
    ref, ref_lse, out, lse = _decode_both(lib, plan, Hq, torch.from_numpy(qn).cuda().bfloat16(), scale, ws, wsn)
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    want, wl = orc.decode(curs, qn.astype(np.float64), scale)
    assert_close(out.float().cpu().numpy(), want, "bf16", "noalloc out vs oracle")
    assert_close(lse.cpu().numpy(), wl, "bf16", "noalloc lse vs oracle")


def test_noalloc_decode_workload(lib, oracle_mod):
    """The 256-cursor decode workload (32 episodes x 8 cursors, paths of 8-32K tokens):
    the same results as the workspace decode, bit for bit, and the oracle's on sampled
    cursors."""
    import bench
    ep, pool, kp, vp, cfg = bench.build_episode(lib, torch, "decode", 0, "cuda")
    Hq, Hkv, d, P = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["P"]
    scale = 1.0 / math.sqrt(d)
    curs = ep.cursors
    n = len(curs)
    plan = pool.decode_plan(curs)
    wsn = plan.decode_workspace_size(Hq)
    assert 0 < wsn <= lib.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(wsn, dtype=torch.uint8, device="cuda")
    q = synth.hash_fill(synth.STREAM_DECODE_Q, (n, Hq, d), torch.bfloat16, "cuda", 0.5)
    for call in range(2):
        ref, ref_lse, out, lse = _decode_both(lib, plan, Hq, q, scale, ws, wsn)
        assert torch.equal(out, ref) and torch.equal(lse, ref_lse), call
    # oracle: the op log without values, K/V set for the sampled cursors' contexts only
    orc = oracle_mod.Oracle(P, pool.num_pages, Hkv, d)
    orc.replay(ep)
    opl = orc.pack(ep.roots, 128, tile_stride=1 << 30)
    pick = sorted(np.random.default_rng(1).choice(n, size=6, replace=False).tolist())
    toks = []
    for i in pick:
        c = curs[i]
        sb = int(opl.seg_row_base[np.nonzero(opl.seg_order == c)[0][0]])
        toks.append(opl.row_context(sb + orc.seg_info(c)["len"] - 1)[0])
    toks = np.unique(np.concatenate(toks))
    K = synth.hash_rows(synth.STREAM_K, toks, Hkv * d, torch.bfloat16, 0.5)
    V = synth.hash_rows(synth.STREAM_V, toks, Hkv * d, torch.bfloat16, 0.5)
    orc.set_kv(toks, K.reshape(-1, Hkv, d), V.reshape(-1, Hkv, d))
    qs = synth.hash_rows(synth.STREAM_DECODE_Q, np.array(pick), Hq * d, torch.bfloat16, 0.5)
    want, wl = orc.decode([curs[i] for i in pick], qs.reshape(-1, Hq, d), scale)
    assert_close(out[pick].float().cpu().numpy(), want, "bf16", "noalloc out (sampled cursors)")
    assert_close(lse[pick].cpu().numpy(), wl, "bf16", "noalloc lse (sampled cursors)")


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
