"""Parity at the full workload sizes, in the launch configuration the benchmark times
(bf16, 16 q / 4 kv heads, d 128, page 64, q-tile 128; inputs from the same counter-based
generator).  The oracle checks sampled outputs one by one -- rows it recomputes over
their whole context, and every key of a few pages through all of their readers -- and
whole-output invariants (sum over all keys of dK is 0; of dV, the sum of dO)."""
import math

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = (2e-2, 2e-2)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import packed_tree_attention_gb300 as pta
    pta.load()
    return pta


def _close(got, ref, what):
    atol, rtol = TOL
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), "%s: %d of %d outside tolerance, worst err %g (ref %g)" % (
        what, bad.sum(), bad.size, err.max(), ref.flat[np.argmax(err)])


class Workload:
    def __init__(self, lib, oracle_mod, name, seed=0, oracle_trees=None):
        import bench
        self.cfg = synth.CONFIGS[name]
        self.Hq, self.Hkv, self.d, self.P = (self.cfg[k] for k in ("Hq", "Hkv", "d", "P"))
        self.seed = seed
        self.ep, self.pool, self.kp, self.vp, _ = bench.build_episode(lib, torch, name, seed, "cuda")
        torch.cuda.synchronize()
        # the oracle replays the op log without values; only sampled tokens get K/V
        ops = self.ep.ops
        if oracle_trees is not None:
            # independent trees: replay the first `oracle_trees` trees only (their
            # segments and tokens come first in creation order)
            roots = [i for i, op in enumerate(ops) if op[0] == "root"]
            ops = ops[:roots[oracle_trees]] if oracle_trees < len(roots) else ops
        sub = synth.Episode(self.P)
        sub.ops = ops
        self.orc = oracle_mod.Oracle(self.P, self.pool.num_pages, self.Hkv, self.d)
        self.orc.replay(sub)
        self.oroots = [s for s in self.ep.roots if s < self.orc.n_segments]
        self.kv_set = np.zeros(self.orc.n_tokens, dtype=bool)
        self.scale = 1.0 / math.sqrt(self.d)

    def need_kv(self, tokens):
        tokens = np.unique(np.asarray(tokens, dtype=np.int64))
        tokens = tokens[~self.kv_set[tokens]]
        if len(tokens) == 0:
            return
        rs = self.Hkv * self.d
        K = synth.hash_rows(synth.STREAM_K + 16 * self.seed, tokens, rs, torch.bfloat16, 0.5)
        V = synth.hash_rows(synth.STREAM_V + 16 * self.seed, tokens, rs, torch.bfloat16, 0.5)
        self.orc.set_kv(tokens, K.reshape(-1, self.Hkv, self.d), V.reshape(-1, self.Hkv, self.d))
        self.kv_set[tokens] = True

    def run(self, with_bwd=True):
        lib_plan = self.pool.pack_tree(self.ep.roots, 128)
        N = lib_plan.info["n_rows"]
        Hq, d = self.Hq, self.d
        self.q = synth.hash_fill(synth.STREAM_Q + 16 * self.seed, (N, Hq, d), torch.bfloat16, "cuda", 0.5)
        self.do = synth.hash_fill(synth.STREAM_DO + 16 * self.seed, (N, Hq, d), torch.bfloat16, "cuda", 1.0)
        o = torch.empty_like(self.q)
        lse = torch.empty((Hq, N), dtype=torch.float32, device="cuda")
        lib_plan.attn_fwd(Hq, self.q, o, lse, self.scale)
        out = {"plan": lib_plan, "o": o, "lse": lse, "N": N}
        if with_bwd:
            dq = torch.empty((N, Hq, d), dtype=torch.float32, device="cuda")
            dk = torch.full((self.pool.num_pages, self.Hkv, self.P, d), float("nan"), device="cuda")
            dv = torch.full_like(dk, float("nan"))
            ws = torch.empty(lib_plan.attn_bwd_workspace_size(Hq), dtype=torch.uint8, device="cuda")
            lib_plan.attn_bwd(Hq, self.q, o, lse, self.do, dq, dk, dv, self.scale, ws)
            out.update(dq=dq, dk=dk, dv=dv)
        lib_plan.sync()
        return out

    def oracle_rows(self, opl, rows):
        """Q and dO arrays with only the given rows filled (the oracle reads only those)."""
        N, Hq, d = opl.n_rows, self.Hq, self.d
        Q = np.zeros((N, Hq, d))
        dO = np.zeros((N, Hq, d))
        Q[rows] = synth.hash_rows(synth.STREAM_Q + 16 * self.seed, rows, Hq * d, torch.bfloat16, 0.5).reshape(-1, Hq, d)
        dO[rows] = synth.hash_rows(synth.STREAM_DO + 16 * self.seed, rows, Hq * d, torch.bfloat16, 1.0).reshape(-1, Hq, d)
        return Q, dO


def _sample_rows(W, opl, k, seed):
    """Seeded rows plus each segment's first and last row and the row at each mount point."""
    rng = np.random.default_rng(seed)
    rows = set(rng.integers(0, opl.n_rows, k).tolist())
    for s, b in zip(opl.seg_order.tolist(), opl.seg_row_base.tolist()):
        L = W.orc.seg_info(s)["len"]
        if L:
            rows.update([b, b + L - 1])
    for i in range(W.orc.n_mounts):
        r, m, *_ = W.orc.mount_info(i)
        idx = np.nonzero(opl.seg_order == r)[0]
        if len(idx) and m < W.orc.seg_info(r)["len"]:
            rows.add(int(opl.seg_row_base[idx[0]]) + m)
    return np.array(sorted(rows), dtype=np.int32)


def _check_values(W, out, n_sample_rows=24, n_pages=2):
    opl = W.orc.pack(W.oroots, 128, tile_stride=1 << 30)
    rows = _sample_rows(W, opl, n_sample_rows, W.seed)
    ctx = [opl.row_context(int(r))[0] for r in rows]
    W.need_kv(np.concatenate(ctx))
    Q, dO = W.oracle_rows(opl, rows)
    Oo, Lo = opl.fwd(Q, W.scale, rows=rows, nthreads=16)
    O = out["o"][:opl.n_rows][torch.from_numpy(rows).long().cuda()].float().cpu().numpy()
    L = out["lse"][:, torch.from_numpy(rows).long().cuda()].cpu().numpy()
    _close(O, Oo[rows], "O (sampled rows)")
    _close(L, Lo[:, rows], "LSE (sampled rows)")
    if "dq" not in out:
        return
    need = np.zeros(opl.n_rows, dtype=np.uint8)
    need[rows] = 1
    dQo, _, _ = opl.bwd(Q, dO, W.scale, need_dq=need, need_dkdv=np.zeros(W.orc.n_tokens, np.uint8),
                        nthreads=16, partial=True)
    dq = out["dq"][torch.from_numpy(rows).long().cuda()].cpu().numpy()
    _close(dq, dQo[rows], "dQ (sampled rows)")
    # dK/dV of every slot of a few pages with few readers, summed by the oracle over all
    # of their reader rows
    gp = out["plan"].copy_out()
    cnt = np.diff(gp["page_off"])
    seg, idx = W.orc.token_owner()
    tok_page = np.array([W.orc.seg_pages(int(s))[int(i) // W.P] for s, i in zip(seg, idx)])
    ent = gp["entries"]
    seg_base = {int(s): int(b) for s, b in zip(opl.seg_order, opl.seg_row_base)}

    def readers(pg):
        rr = []
        for c in gp["csc_perm"][gp["page_off"][pg]:gp["page_off"][pg + 1]]:
            t = int(ent["q_tile"][c])
            b = seg_base[int(gp["tile_seg"][t])] + int(gp["tile_t0"][t])
            rr.extend(range(b, b + int(gp["tile_rows"][t])))
        return rr

    # pages of the oracle's trees read by one or two tiles; the cheapest to recompute
    # (rows x context length of their readers) are checked
    owned = np.zeros(len(cnt), dtype=bool)
    owned[np.unique(tok_page)] = True
    cand = np.nonzero((cnt > 0) & (cnt <= 2) & owned)[0]
    rng = np.random.default_rng(W.seed + 1)
    cand = rng.choice(cand, size=min(40, len(cand)), replace=False)
    cost = []
    for pg in cand:
        rr = readers(pg)
        cost.append(len(rr) * len(opl.row_context(int(rr[-1]))[0]))
    pages = [int(cand[i]) for i in np.argsort(cost)[:n_pages]]
    tok = np.nonzero(np.isin(tok_page, pages))[0]
    need_tok = np.zeros(W.orc.n_tokens, dtype=np.uint8)
    need_tok[tok] = 1
    reader_rows = [r for pg in pages for r in readers(pg)]
    reader_rows = np.array(sorted(set(reader_rows)), dtype=np.int32)
    W.need_kv(np.concatenate([opl.row_context(int(r))[0] for r in reader_rows]))
    Q2, dO2 = W.oracle_rows(opl, reader_rows)
    _, dKo, dVo = opl.bwd(Q2, dO2, W.scale, need_dq=np.zeros(opl.n_rows, np.uint8), need_dkdv=need_tok,
                          nthreads=16)
    slot = idx[tok] % W.P
    dk = out["dk"].cpu().numpy()[tok_page[tok], :, slot]
    dv = out["dv"].cpu().numpy()[tok_page[tok], :, slot]
    _close(dk, dKo[tok], "dK (pages %s)" % pages)
    _close(dv, dVo[tok], "dV (pages %s)" % pages)


def _check_invariants(W, out):
    gp = out["plan"].copy_out()
    touched = np.nonzero(np.diff(gp["page_off"]))[0]
    dk = out["dk"][torch.from_numpy(touched).long().cuda()].double()
    dv = out["dv"][torch.from_numpy(touched).long().cuda()].double()
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all()
    o = out["o"].float()
    assert torch.isfinite(o).all() and torch.isfinite(out["dq"]).all()
    G = W.Hq // W.Hkv
    N = out["N"]
    sk = dk.sum(dim=(0, 2))                                  # [Hkv, d]
    print("invariants: |sum dK| %.4g (scale %.4g)" % (float(sk.abs().max()), float(dk.abs().sum(dim=(0, 2)).max())))
    assert float(sk.abs().max()) <= 1e-2 * float(dk.abs().sum(dim=(0, 2)).max()) + 1e-3
    want = W.do.double().view(N, W.Hkv, G, W.d).sum(dim=(0, 2))  # [Hkv, d]
    sv = dv.sum(dim=(0, 2))
    print("invariants: |sum dV - sum dO| %.4g (max |sum dO| %.4g)" % (float((sv - want).abs().max()),
                                                                     float(want.abs().max())))
    # measured ~1e-3 of max|want|; a lost or half-read reader contribution shows as percents
    assert float((sv - want).abs().max()) <= 5e-3 * float(want.abs().max()) + 1e-2 * math.sqrt(N)


def test_episode_fwd_bwd_full(lib, oracle_mod):
    W = Workload(lib, oracle_mod, "episode", seed=0)
    out = W.run()
    assert out["plan"].kernel_path(W.Hq, 0) == 1 and out["plan"].kernel_path(W.Hq, 1) == 1
    assert out["plan"].info["pairs"] == W.orc.pack(W.oroots, 128, tile_stride=1 << 30).total_pairs()
    _check_invariants(W, out)
    _check_values(W, out)


def test_tree_fwd_full(lib, oracle_mod):
    W = Workload(lib, oracle_mod, "tree_fwd", seed=0)
    out = W.run(with_bwd=False)
    _check_values(W, out, n_sample_rows=32)


def test_train_step_full(lib, oracle_mod):
    """8 trees, ~1.12M packed rows: the library runs the whole step; the oracle checks the
    first tree (trees are independent, and the first tree's rows come first)."""
    W = Workload(lib, oracle_mod, "train_step", seed=0, oracle_trees=1)
    out = W.run()
    assert out["N"] > 1_000_000
    _check_invariants(W, out)
    _check_values(W, out, n_sample_rows=16, n_pages=1)


def test_decode_full(lib, oracle_mod):
    W = Workload(lib, oracle_mod, "decode", seed=0)
    curs = W.ep.cursors
    dp = W.pool.decode_plan(curs)
    n = len(curs)
    q = synth.hash_fill(synth.STREAM_DECODE_Q, (n, W.Hq, W.d), torch.bfloat16, "cuda", 0.5)
    out = torch.empty_like(q)
    lse = torch.empty((n, W.Hq), dtype=torch.float32, device="cuda")
    wsn = dp.decode_workspace_size(W.Hq)
    ws = torch.empty(max(1, wsn), dtype=torch.uint8, device="cuda")
    dp.decode(W.Hq, q, out, lse, W.scale, ws, wsn)
    dp.sync()
    assert dp.kernel_path(W.Hq, 2) == 2
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(0)
    pick = sorted(rng.choice(n, size=12, replace=False).tolist())
    opl = W.orc.pack(W.oroots, 128, tile_stride=1 << 30)
    for i in pick:
        c = curs[i]
        sb = int(opl.seg_row_base[np.nonzero(opl.seg_order == c)[0][0]])
        W.need_kv(opl.row_context(sb + W.orc.seg_info(c)["len"] - 1)[0])
    qs = synth.hash_rows(synth.STREAM_DECODE_Q, np.array(pick), W.Hq * W.d, torch.bfloat16, 0.5)
    want, wl = W.orc.decode([curs[i] for i in pick], qs.reshape(-1, W.Hq, W.d), W.scale)
    _close(out[pick].float().cpu().numpy(), want, "decode out (sampled cursors)")
    _close(lse[pick].cpu().numpy(), wl, "decode lse (sampled cursors)")
