"""GPU parity of the rotary embedding at the packed positions against the fp64 oracle,
through the C ABI: rows of a plan (forward and inverse, bf16 and fp32), keys rotated at
append, key gradients turned back in the pool layout, and a forward + backward over an
episode with mounts whose queries and keys carry the rotation."""
import math

import numpy as np
import pytest

import synth
from helpers import assert_close, packed, pool_pages_needed, replay_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BASE = 10000.0


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _setup(lib, oracle_mod, seed, Hq=16, Hkv=4, d=128, rope_keys=True):
    ep = synth.random_dag(700 + seed, page_size=64, max_segments=10, max_len=400, n_roots=1 + seed % 2)
    t = synth.make_tensors(ep, Hq, Hkv, d, "bf16", 0.5, seed)
    npages = pool_pages_needed(ep)
    kpool = torch.zeros((npages, Hkv, 64, d), dtype=torch.bfloat16, device="cuda")
    vpool = torch.zeros_like(kpool)
    pool = lib.Pool(npages, 64, Hkv, d, lib.DTYPE_BF16, kpool, vpool)
    K = torch.from_numpy(t.K).cuda().to(torch.bfloat16)
    V = torch.from_numpy(t.V).cuda().to(torch.bfloat16)
    pos = replay_device(pool, ep, K, V, rope_base=BASE if rope_keys else None)
    torch.cuda.synchronize()
    orc = oracle_mod.Oracle(64, npages, Hkv, d)
    opos = orc.replay(ep)
    assert np.array_equal(pos, opos)
    return ep, t, pool, kpool, vpool, pos, orc


def _close(got, want, rel, abs_):
    err = np.abs(got - want)
    bad = err > abs_ + rel * np.abs(want)
    assert not bad.any(), "%d of %d outside; worst %g" % (bad.sum(), bad.size, err.max())


@pytest.mark.parametrize("seed", [0, 1])
def test_append_rope_rotates_keys_at_their_positions(lib, oracle_mod, seed):
    ep, t, pool, kpool, vpool, pos, orc = _setup(lib, oracle_mod, seed)
    seg, idx = orc.token_owner()
    pages = {s: orc.seg_pages(s) for s in set(seg.tolist())}
    page = np.array([pages[s][i // 64] for s, i in zip(seg.tolist(), idx.tolist())])
    slot = idx % 64
    kp = kpool.float().cpu().numpy()
    vp = vpool.float().cpu().numpy()
    # token order of the oracle = append order
    Kb = t.K.astype(np.float32).astype(np.float64)
    want = oracle_mod.rope(torch.from_numpy(t.K).to(torch.bfloat16).float().numpy(), pos, BASE)
    got = kp[page, :, slot, :]
    _close(got, want, 2.0 ** -8, 1e-6)
    Vb = torch.from_numpy(t.V).to(torch.bfloat16).float().numpy()
    assert np.array_equal(vp[page, :, slot, :], Vb)
    del Kb


@pytest.mark.parametrize("dtype,inverse", [("bf16", False), ("f32", False), ("f32", True)])
def test_rope_rows_matches_oracle(lib, oracle_mod, dtype, inverse):
    ep, t, pool, kpool, vpool, pos, orc = _setup(lib, oracle_mod, 3, rope_keys=False)
    plan = pool.pack_tree(ep.roots, 128)
    opl = orc.pack(ep.roots, 128)
    N, Hq = plan.info["n_rows"], 16
    rng = np.random.default_rng(4)
    x = rng.standard_normal((N, Hq, 128)).astype(np.float32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    xd = torch.from_numpy(x).cuda().to(tdt)
    x_in = xd.float().cpu().numpy()
    plan.rope_rows(Hq, xd, BASE, inverse=inverse)
    torch.cuda.synchronize()
    want = oracle_mod.rope(x_in, opl.row_pos, BASE, inverse=inverse)
    got = xd.float().cpu().numpy()
    if dtype == "bf16":
        _close(got, want, 2.0 ** -8, 1e-6)
    else:
        _close(got, want, 1e-5, 1e-5)


def test_rope_pool_grad_turns_slots_back(lib, oracle_mod):
    ep, t, pool, kpool, vpool, pos, orc = _setup(lib, oracle_mod, 4)
    plan = pool.pack_tree(ep.roots, 128)
    rng = np.random.default_rng(5)
    dk = torch.from_numpy(rng.standard_normal(tuple(kpool.shape)).astype(np.float32)).cuda()
    before = dk.cpu().numpy()
    plan.rope_pool_grad(dk, BASE)
    got = dk.cpu().numpy()
    touched = set(np.nonzero(np.diff(plan.copy_out()["page_off"]))[0].tolist())
    seg, idx = orc.token_owner()
    pages = {s: orc.seg_pages(s) for s in set(seg.tolist())}
    page = np.array([pages[s][i // 64] for s, i in zip(seg.tolist(), idx.tolist())])
    slot = idx % 64
    sel = np.array([p in touched for p in page])
    want = oracle_mod.rope(before[page[sel], :, slot[sel], :], pos[sel], BASE, inverse=True)
    _close(got[page[sel], :, slot[sel], :], want, 1e-5, 1e-5)
    # pages the plan does not read and slots holding no token are untouched
    mask = np.ones(got.shape[:1] + got.shape[2:3], dtype=bool)   # [page, slot]
    mask[page[sel], slot[sel]] = False
    pg, sl = np.nonzero(mask)
    assert np.array_equal(got[pg, :, sl, :], before[pg, :, sl, :])


def test_fwd_bwd_with_rope_matches_oracle(lib, oracle_mod):
    """Queries rotated at their rows' positions, keys at their tokens' positions (read as
    stored through the mounts); the backward's dq and dk turned back."""
    Hq, Hkv, d = 16, 4, 128
    ep, t, pool, kpool, vpool, pos, orc = _setup(lib, oracle_mod, 6, Hq, Hkv, d)
    plan = pool.pack_tree(ep.roots, 128)
    opl = orc.pack(ep.roots, 128)
    N = plan.info["n_rows"]
    Q = packed(t, opl.seg_order, t.Q)
    dO = packed(t, opl.seg_order, t.dO)
    qd = torch.from_numpy(np.ascontiguousarray(Q)).cuda().to(torch.bfloat16)
    q_in = qd.float().cpu().numpy()
    plan.rope_rows(Hq, qd, BASE)
    o = torch.empty((N, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Hq, N), dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    plan.attn_fwd(Hq, qd, o, lse, scale)
    dod = torch.from_numpy(np.ascontiguousarray(dO)).cuda().to(torch.bfloat16)
    dq = torch.empty((N, Hq, d), dtype=torch.float32, device="cuda")
    dk = torch.zeros(tuple(kpool.shape), dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(max(1, plan.attn_bwd_workspace_size(Hq)), dtype=torch.uint8, device="cuda")
    plan.attn_bwd(Hq, qd, o, lse, dod, dq, dk, dv, scale, ws)
    plan.rope_rows(Hq, dq, BASE, inverse=True)
    plan.rope_pool_grad(dk, BASE)
    plan.sync()
    # the oracle on rotated inputs: keys as the pool stores them (bf16), queries rotated
    Kin = torch.from_numpy(t.K).to(torch.bfloat16).float().numpy()
    Krot = oracle_mod.rope(Kin, pos, BASE)
    Vin = torch.from_numpy(t.V).to(torch.bfloat16).float().numpy().astype(np.float64)
    orc2 = oracle_mod.Oracle(64, pool.num_pages, Hkv, d)
    orc2.replay(ep, Krot, Vin)
    opl2 = orc2.pack(ep.roots, 128)
    Qrot = oracle_mod.rope(q_in, opl2.row_pos, BASE)
    Oo, Lo = opl2.fwd(Qrot, scale)
    assert_close(o.float().cpu().numpy(), Oo, "bf16", "O")
    dQo, dKo, dVo = opl2.bwd(Qrot, dod.float().cpu().numpy().astype(np.float64), scale)
    dQo = oracle_mod.rope(dQo, opl2.row_pos, BASE, inverse=True)
    dKo = oracle_mod.rope(dKo, pos, BASE, inverse=True)
    assert_close(dq.cpu().numpy(), dQo, "bf16", "dQ")
    seg, idx = orc.token_owner()
    pages = {s: orc.seg_pages(s) for s in set(seg.tolist())}
    page = np.array([pages[s][i // 64] for s, i in zip(seg.tolist(), idx.tolist())])
    slot = idx % 64
    assert_close(dk.cpu().numpy()[page, :, slot, :], dKo, "bf16", "dK")
    assert_close(dv.cpu().numpy()[page, :, slot, :], dVo, "bf16", "dV")
