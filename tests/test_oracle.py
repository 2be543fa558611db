"""Pins for the fp64 oracle.  Nothing here compares the oracle with itself: each test
checks it against something the pages or the mathematics fix -- a hand-derived worked
example, textbook causal attention (torch SDPA / autograd in fp64), a flat per-branch
re-derivation of every context, zero-copy mount == physical copy, central finite
differences, and closed-form invariants of softmax attention."""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _replay(oracle_mod, ep, Hkv, d, K=None, V=None, num_pages=4096):
    o = oracle_mod.Oracle(ep.page_size, num_pages, Hkv, d)
    o.replay(ep, K, V)
    return o


def _packed(t, seg_order, arr):
    return np.concatenate([arr[t.seg_off[s]:t.seg_off[s + 1]] for s in seg_order], axis=0)


# ------------------------------------------------------------------ worked example
def test_tiny_golden(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "tiny_tree.json")))
    ep = synth.make_preset("tiny")
    o = _replay(oracle_mod, ep, 1, 64)
    assert o.seg_pos(0).tolist() == list(range(0, 64))
    assert o.seg_pos(1).tolist() == list(range(64, 96))
    assert o.seg_pos(2).tolist() == list(range(64, 80)) + list(range(89, 105))
    for s, pages in g["pages"].items():
        assert o.seg_pages(int(s)).tolist() == pages
    pl = o.pack([0], g["bm"])
    assert np.diff(pl.tile_off).tolist() == g["entries_per_tile"]
    assert pl.pairs == g["pairs_total"]
    # pairs per segment via the rectangle formula over that segment's tiles
    P = g["page_size"]
    per_seg = {}
    for e in pl.entries:
        tile, page, lo, hi, qlo, fl, dg, src = e.tolist()
        rows = pl.tile_rows[tile]
        n = 0
        for r in range(qlo, rows):
            for j in range(lo, hi):
                n += (not fl) or (j <= r + dg)
        s = int(pl.tile_seg[tile])
        per_seg[s] = per_seg.get(s, 0) + n
    assert per_seg == {int(k): v for k, v in g["pairs_per_segment"].items()}
    mounts = [[int(e[1]), int(e[2]), int(e[3]), int(e[4])] for e in pl.entries if e[7] >= 0]
    assert mounts == g["mount_entries"]


def test_mount_offset_closed_form(oracle_mod):
    """s = max(p_B, e_A + 1) for both orders of p_B and e_A (page 'Architecture &
    Co-Design', item 02)."""
    ep = synth.Episode(16)
    o = oracle_mod.Oracle(16, 256, 1, 8)
    r = o.root(); o.append(r, 10)
    a, b = o.fork(r, 2)
    o.append(a, 100)            # A positions 10..109
    o.append(b, 5)              # p_B = 15
    assert o.mount(b, a, 3, 7) == max(15, (10 + 6) + 1 + 1)      # e_A = 17 > p_B
    o.append(b, 40)             # p_B = 18 + 40 = 58
    assert o.mount(b, a, 20, 30) == max(58, (10 + 29) + 1 + 1)   # e_A = 40 < p_B
    del ep


# ------------------------------------------------------------------ textbook attention
@pytest.mark.parametrize("n,Hq,Hkv,d,P", [(1, 2, 1, 8, 4), (37, 4, 2, 16, 16), (70, 2, 2, 32, 16)])
def test_single_segment_is_causal_attention(oracle_mod, n, Hq, Hkv, d, P):
    rng = np.random.default_rng(n)
    Q = rng.standard_normal((n, Hq, d))
    K = rng.standard_normal((n, Hkv, d))
    V = rng.standard_normal((n, Hkv, d))
    dO = rng.standard_normal((n, Hq, d))
    o = oracle_mod.Oracle(P, 64, Hkv, d)
    r = o.root()
    o.append(r, n, K, V)
    pl = o.pack([r], 16)
    scale = 1 / math.sqrt(d)
    O, LSE = pl.fwd(Q, scale)
    dQ, dK, dV = pl.bwd(Q, dO, scale)
    q = torch.tensor(Q, dtype=torch.float64).permute(1, 0, 2).requires_grad_()
    k = torch.tensor(K, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    v = torch.tensor(V, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
    kk, vv = k.detach().requires_grad_(), v.detach().requires_grad_()
    out = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True, scale=scale)
    out.backward(torch.tensor(dO, dtype=torch.float64).permute(1, 0, 2))
    np.testing.assert_allclose(O, out.detach().permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
    s = (q.detach() @ kk.detach().transpose(1, 2)) * scale
    s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), -math.inf)
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dQ, q.grad.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-11)
    G = Hq // Hkv
    gk = kk.grad.reshape(Hkv, G, n, d).sum(1).permute(1, 0, 2).numpy()
    gv = vv.grad.reshape(Hkv, G, n, d).sum(1).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(dK, gk, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dV, gv, rtol=1e-10, atol=1e-11)


# ------------------------------------------------------------------ flat per-branch attention
def _flat_branches(ep):
    """Independent re-derivation of every context: for each segment, the flat sequence
    of keys it sees (walking the op log), with the row index from which each key is
    visible.  Returns {segment: [(token_id, visible_from_row)]}.

    Walk: a segment's sequence is its parent's sequence as it stood when the segment
    was created, cut to the parent's first f tokens, followed by its own tokens and
    mounted spans in the order they were added."""
    seqs = {}          # segment -> list of ('tok', token_id, own_index) | ('span', [token ids], m)
    toks = {}          # segment -> own token ids
    snap = {}          # child -> (parent, f, len(parent's event list) at creation)
    tid = 0
    nseg = 0
    for op in ep.ops:
        kind = op[0]
        if kind == "root":
            seqs[nseg], toks[nseg] = [], []
            nseg += 1
        elif kind == "append":
            _, c, n = op
            for _ in range(n):
                seqs[c].append(("tok", tid, len(toks[c])))
                toks[c].append(tid)
                tid += 1
        elif kind == "fork":
            _, c, n = op
            for _ in range(n):
                snap[nseg] = (c, len(toks[c]), len(seqs[c]))
                seqs[nseg], toks[nseg] = [], []
                nseg += 1
        elif kind == "rewind":
            _, c, k = op
            # events of c up to token k: everything before own token k (mounts at m <= k
            # were added while c had <= k tokens, so they precede token k)
            cut = len(seqs[c])
            for i, ev in enumerate(seqs[c]):
                if ev[0] == "tok" and ev[2] == k:
                    cut = i
                    break
            snap[nseg] = (c, k, cut)
            seqs[nseg], toks[nseg] = [], []
            nseg += 1
        elif kind == "mount":
            _, r, p, a, b = op
            seqs[r].append(("span", toks[p][a:b], len(toks[r])))
    out = {}

    def flat(s):
        if s in out:
            return out[s]
        items = []
        if s in snap:
            par, f, cut = snap[s]
            for tok, _ in flat_cut(par, cut):
                items.append((tok, 0))
        for ev in seqs[s]:
            if ev[0] == "tok":
                items.append((ev[1], ev[2]))
            else:
                items.extend((t, ev[2]) for t in ev[1])
        out[s] = items
        return items

    def flat_cut(s, cut):
        base = []
        if s in snap:
            par, f, c2 = snap[s]
            base = [(t, 0) for t, _ in flat_cut(par, c2)]
        for ev in seqs[s][:cut]:
            if ev[0] == "tok":
                base.append((ev[1], 0))
            else:
                base.extend((t, 0) for t in ev[1])
        return base

    for s in range(nseg):
        flat(s)
    return out, toks


@pytest.mark.parametrize("seed", range(8))
def test_flat_per_branch(oracle_mod, seed):
    ep = synth.random_dag(seed, page_size=8, max_segments=10, max_len=40)
    Hq, Hkv, d = 4, 2, 16
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, seed)
    o = _replay(oracle_mod, ep, Hkv, d, t.K.astype(np.float64), t.V.astype(np.float64))
    pl = o.pack(ep.roots, 16)
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    scale = 0.3
    O, LSE = pl.fwd(Q, scale)
    flat, toks = _flat_branches(ep)
    K = torch.tensor(t.K, dtype=torch.float64)
    V = torch.tensor(t.V, dtype=torch.float64)
    total_pairs = 0
    for si, s in enumerate(pl.seg_order.tolist()):
        items = flat[s]
        n = len(toks[s])
        if n == 0:
            continue
        ids = torch.tensor([it[0] for it in items])
        frm = torch.tensor([it[1] for it in items])
        mask = frm[None, :] <= torch.arange(n)[:, None]          # [rows, keys]
        total_pairs += int(mask.sum())
        r0 = pl.seg_row_base[si]
        q = torch.tensor(Q[r0:r0 + n], dtype=torch.float64).permute(1, 0, 2)
        k = K[ids].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        v = V[ids].permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        np.testing.assert_allclose(O[r0:r0 + n], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
    assert total_pairs == pl.pairs


# ------------------------------------------------------------------ mount == copy
def _copy_variant(ep, K, V, mount_index):
    """The same episode with one mount replaced by appending copies of the span's K/V
    to the reader.  Returns (episode, K, V, copy_map) where copy_map[j] is the token id
    whose K/V the j-th copied token holds."""
    ep2 = synth.Episode(ep.page_size)
    toks = {}
    K2, V2 = [], []
    tid = 0
    nseg = 0
    copy_map = {}
    mi = 0
    for op in ep.ops:
        kind = op[0]
        if kind == "root":
            ep2.root(); toks[nseg] = []; nseg += 1
        elif kind == "append":
            _, c, n = op
            for _ in range(n):
                toks[c].append(tid); K2.append(K[tid]); V2.append(V[tid]); tid += 1
            ep2.append(c, n)
        elif kind == "fork":
            for _ in ep2.fork(op[1], op[2]):
                toks[nseg] = []; nseg += 1
        elif kind == "rewind":
            ep2.rewind(op[1], op[2]); toks[nseg] = []; nseg += 1
        elif kind == "mount":
            _, r, p, a, b = op
            if mi == mount_index:
                ep2.append(r, b - a)
                for j in range(a, b):
                    src = toks[p][j]
                    copy_map[len(K2)] = src
                    K2.append(K[src]); V2.append(V[src])
            else:
                ep2.mount(r, p, a, b)
            mi += 1
        else:
            getattr(ep2, kind)(*op[1:])
    return ep2, np.array(K2), np.array(V2), copy_map


@pytest.mark.parametrize("case", ["tiny", "two_readers"])
def test_mount_equals_copy(oracle_mod, case):
    if case == "tiny":
        ep = synth.make_preset("tiny")
        Hq, Hkv, d = 1, 1, 64
    else:
        ep = synth.Episode(8)
        r = ep.root(); ep.append(r, 13)
        a, b, c = ep.fork(r, 3)
        ep.append(a, 30); ep.append(b, 9)
        ep.mount(b, a, 5, 22)          # e_A > p_B: position jump
        ep.append(b, 11)
        ep.append(c, 40)
        Hq, Hkv, d = 4, 2, 8
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, 3)
    K, V = t.K.astype(np.float64), t.V.astype(np.float64)
    ep2, K2, V2, cmap = _copy_variant(ep, K, V, 0)
    o1 = _replay(oracle_mod, ep, Hkv, d, K, V)
    o2 = _replay(oracle_mod, ep2, Hkv, d, K2, V2)
    p1, p2 = o1.pack(ep.roots, 16), o2.pack(ep2.roots, 16)
    # rows of the original episode inside the copy variant: same segment order, the
    # reader's rows after the mount point shift by the span length
    m = [op for op in ep.ops if op[0] == "mount"][0]
    reader, span = m[1], m[4] - m[3]
    mpt = o1.mount_info(0)[1]
    rows2 = []
    for si, s in enumerate(p1.seg_order.tolist()):
        n = o1.seg_info(s)["len"]
        base2 = p2.seg_row_base[si]
        for i in range(n):
            rows2.append(base2 + (i if (s != reader or i < mpt) else i + span))
    rows2 = np.array(rows2)
    rng = np.random.default_rng(7)
    Q1 = rng.standard_normal((p1.n_rows, Hq, d))
    dO1 = rng.standard_normal((p1.n_rows, Hq, d))
    Q2 = rng.standard_normal((p2.n_rows, Hq, d))
    dO2 = np.zeros((p2.n_rows, Hq, d))        # copies are keys only: no loss on their rows
    Q2[rows2] = Q1
    dO2[rows2] = dO1
    scale = 1 / math.sqrt(d)
    O1, L1 = p1.fwd(Q1, scale)
    O2, L2 = p2.fwd(Q2, scale)
    np.testing.assert_allclose(O2[rows2], O1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L2[:, rows2], L1, rtol=1e-12, atol=1e-12)
    dQ1, dK1, dV1 = p1.bwd(Q1, dO1, scale)
    dQ2, dK2, dV2 = p2.bwd(Q2, dO2, scale)
    np.testing.assert_allclose(dQ2[rows2], dQ1, rtol=1e-10, atol=1e-12)
    # scatter the copies' gradients back onto the tokens they copy
    T1 = o1.n_tokens
    orig_of = np.arange(len(K2))
    for j, src in cmap.items():
        orig_of[j] = src
    # token ids of ep2 that are not copies map to ep's ids in order
    non_copy = [j for j in range(len(K2)) if j not in cmap]
    assert len(non_copy) == T1
    back = np.zeros(len(K2), dtype=np.int64)
    back[non_copy] = np.arange(T1)
    for j, src in cmap.items():
        back[j] = src
    gK = np.zeros_like(dK1); gV = np.zeros_like(dV1)
    np.add.at(gK, back, dK2); np.add.at(gV, back, dV2)
    np.testing.assert_allclose(gK, dK1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gV, dV1, rtol=1e-10, atol=1e-12)
    # the mount itself allocated no page
    assert o1.free_pages() - o2.free_pages() >= 0


# ------------------------------------------------------------------ finite differences
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_finite_differences(oracle_mod, seed):
    ep = synth.random_dag(100 + seed, page_size=4, max_segments=6, max_len=12)
    Hq, Hkv, d = 2, 1, 6
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, seed)
    K, V = t.K.astype(np.float64), t.V.astype(np.float64)
    o = _replay(oracle_mod, ep, Hkv, d, K, V)
    pl = o.pack(ep.roots, 8)
    if pl.n_rows == 0:
        pytest.skip("empty episode")
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    dO = _packed(t, pl.seg_order, t.dO).astype(np.float64)
    scale = 0.7
    dQ, dK, dV = pl.bwd(Q, dO, scale)

    def loss_q(Qx):
        O, _ = pl.fwd(Qx, scale)
        return float((O * dO).sum())

    def loss_kv(Kx, Vx):
        o2 = _replay(oracle_mod, ep, Hkv, d, Kx, Vx)
        O, _ = o2.pack(ep.roots, 8).fwd(Q, scale)
        return float((O * dO).sum())

    h = 1e-6
    rng = np.random.default_rng(seed)
    for _ in range(6):
        idx = tuple(rng.integers(0, s) for s in Q.shape)
        Qp, Qm = Q.copy(), Q.copy()
        Qp[idx] += h; Qm[idx] -= h
        fd = (loss_q(Qp) - loss_q(Qm)) / (2 * h)
        assert abs(fd - dQ[idx]) <= 1e-6 * max(1.0, abs(fd))
    for which, G in (("K", dK), ("V", dV)):
        for _ in range(4):
            idx = tuple(rng.integers(0, s) for s in K.shape)
            Kp, Km, Vp, Vm = K.copy(), K.copy(), V.copy(), V.copy()
            if which == "K":
                Kp[idx] += h; Km[idx] -= h
            else:
                Vp[idx] += h; Vm[idx] -= h
            fd = (loss_kv(Kp, Vp) - loss_kv(Km, Vm)) / (2 * h)
            assert abs(fd - G[idx]) <= 1e-6 * max(1.0, abs(fd))


# ------------------------------------------------------------------ closed forms / invariants
@pytest.mark.parametrize("seed", range(5))
def test_gradient_sum_invariants(oracle_mod, seed):
    """Sum_j dS_ij = 0 per row, so the dK of all tokens sums to zero per kv head; the
    softmax weights of a row sum to 1, so the dV of all tokens sums to the dO of all
    rows of the head group."""
    ep = synth.random_dag(200 + seed, page_size=8, max_segments=10, max_len=50)
    Hq, Hkv, d = 4, 2, 8
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, seed)
    o = _replay(oracle_mod, ep, Hkv, d, t.K.astype(np.float64), t.V.astype(np.float64))
    pl = o.pack(ep.roots, 16)
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    dO = _packed(t, pl.seg_order, t.dO).astype(np.float64)
    dQ, dK, dV = pl.bwd(Q, dO, 0.5)
    # only tokens that some packed row sees get gradient; all tokens here are packed
    np.testing.assert_allclose(dK.sum(0), 0.0, atol=1e-10)
    want = dO.reshape(-1, Hkv, Hq // Hkv, d).sum((0, 2))
    np.testing.assert_allclose(dV.sum(0), want, rtol=1e-10, atol=1e-10)


def test_constant_keys_uniform_weights(oracle_mod):
    """Equal keys give every visible token the same weight: O is the mean of the
    visible V rows and LSE = s + ln(n)."""
    ep = synth.make_preset("tiny")
    d = 64
    t = synth.make_tensors(ep, 1, 1, d, "f32", 1.0, 0)
    K = np.ones_like(t.K, dtype=np.float64) * 0.25
    V = t.V.astype(np.float64)
    o = _replay(oracle_mod, ep, 1, d, K, V)
    pl = o.pack([0], 32)
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    O, LSE = pl.fwd(Q, 0.125)
    for r in [0, 5, 63, 64, 100, 127]:
        tok, _ = pl.row_context(r)
        np.testing.assert_allclose(O[r, 0], V[tok, 0].mean(0), rtol=1e-12, atol=1e-12)
        s = 0.125 * Q[r, 0].sum() * 0.25
        assert abs(LSE[0, r] - (s + math.log(len(tok)))) < 1e-12


def test_decode_is_last_row(oracle_mod):
    ep = synth.random_dag(5, page_size=8, max_segments=10, max_len=30)
    Hq, Hkv, d = 4, 2, 8
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, 5)
    o = _replay(oracle_mod, ep, Hkv, d, t.K.astype(np.float64), t.V.astype(np.float64))
    pl = o.pack(ep.roots, 16)
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    O, LSE = pl.fwd(Q, 0.4)
    curs, rows = [], []
    for si, s in enumerate(pl.seg_order.tolist()):
        n = o.seg_info(s)["len"]
        if n:
            curs.append(s); rows.append(pl.seg_row_base[si] + n - 1)
    out, lse = o.decode(curs, Q[rows], 0.4)
    np.testing.assert_allclose(out, O[rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, LSE[:, rows].T, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ pool semantics
def test_pool_invariants(oracle_mod):
    o = oracle_mod.Oracle(4, 32, 1, 4)
    r = o.root()
    o.append(r, 10)                                 # 3 pages: 0,1,2
    assert o.seg_pages(r).tolist() == [0, 1, 2]
    free0 = o.free_pages()
    kids = o.fork(r, 3)                             # fork: 0 pages, refcount + K
    assert o.free_pages() == free0
    assert o.seg_info(r)["refcount"] == 1 + 3
    o.append(kids[0], 5)                            # a child starts on a new page
    assert o.seg_pages(kids[0]).tolist() == [3, 4]
    o.append(kids[1], 2)
    f1 = o.free_pages()
    o.mount(kids[1], kids[0], 1, 5)                 # mount: 0 pages, producer ref + 1
    assert o.free_pages() == f1
    assert o.seg_info(kids[0])["refcount"] == 2
    o.done(kids[0])                                 # done pins
    o.release(kids[0])
    assert o.seg_info(kids[0])["flags"] & 16 == 0   # pinned + mounted: survives
    o.release(kids[1])                              # drops the mount ref too
    assert o.seg_info(kids[1])["flags"] & 16 == 16
    assert o.seg_info(kids[0])["refcount"] == 1     # the pin
    o.unpin(kids[0])
    assert o.seg_info(kids[0])["flags"] & 16 == 16
    freed_pages = o.free_pages()
    o.append(kids[2], 3)                            # lowest free page first
    assert o.seg_pages(kids[2]).tolist() == [3]
    assert o.free_pages() == freed_pages - 1
    # rewind keeps the tail until release; continuation inherits the prefix
    c2 = o.rewind(kids[2], 1)
    assert o.seg_info(kids[2])["flags"] & 8
    assert o.append(kids[2], 1, check=False) == oracle_mod.ESTATE
    o.append(c2, 4)
    o.release(c2)
    assert o.seg_info(kids[2])["flags"] & 16 and o.seg_info(c2)["flags"] & 16
    o.release(r)
    assert o.free_pages() == 32


def test_rewind_positions_and_mount_inheritance(oracle_mod):
    o = oracle_mod.Oracle(4, 64, 1, 4)
    r = o.root(); o.append(r, 6)
    a, b = o.fork(r, 2)
    o.append(a, 20)
    o.append(b, 3)
    o.mount(b, a, 0, 10)            # at m = 3: p jumps to (6+9)+1+1 = 17
    o.append(b, 4)                  # positions 17..20
    assert o.seg_pos(b).tolist() == [6, 7, 8, 17, 18, 19, 20]
    c = o.rewind(b, 3)              # k == m: the mount is kept (m <= k), p = pos(b,3) = 17
    o.append(c, 2)
    assert o.seg_pos(c).tolist() == [17, 18]
    d_ = o.rewind(c, 0)             # continuation of c at 0 still inherits b's mount
    o.append(d_, 1)
    pl = o.pack([r], 8)
    row = [i for i, s in enumerate(pl.seg_order.tolist()) if s == d_][0]
    tok, src = pl.row_context(int(pl.seg_row_base[row]))
    assert (src >= 0).sum() == 10
    assert len(tok) == 6 + 3 + 10 + 1


def test_mount_validation(oracle_mod):
    E = oracle_mod.EINVAL
    o = oracle_mod.Oracle(4, 64, 1, 4)
    r = o.root(); o.append(r, 8)
    a, b = o.fork(r, 2)
    o.append(a, 8); o.append(b, 8)
    assert o.mount(b, b, 0, 2, check=False) == E          # self: already visible
    assert o.mount(b, r, 0, 2, check=False) == E          # ancestor prefix: visible
    assert o.mount(b, a, 0, 9, check=False) == E          # out of range
    assert o.mount(b, a, 3, 3, check=False) == E          # empty span
    o.mount(b, a, 0, 4)
    assert o.mount(b, a, 2, 6, check=False) == E          # overlaps the earlier mount
    o.mount(b, a, 4, 8)                                   # disjoint: fine
    o.append(r, 4)                                        # parent continues after fork
    assert o.mount(b, r, 8, 12, check=False) == oracle_mod.OK   # parent's tokens past f
    kid = o.fork(b, 1)[0]                                  # inherits b's mounts
    assert o.mount(kid, a, 1, 2, check=False) == E
    o.done(a)
    assert o.append(a, 1, check=False) == oracle_mod.ESTATE
    assert o.mount(kid, a, 1, 2, check=False) == E


@pytest.mark.parametrize("seed", range(3))
def test_subset_backward_matches_full(oracle_mod, seed):
    """The sampled modes (a token subset for dK/dV, a row subset for dQ) give exactly the
    full backward's values on that subset."""
    ep = synth.random_dag(600 + seed, page_size=8, max_segments=10, max_len=50)
    Hq, Hkv, d = 4, 2, 8
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, seed)
    o = _replay(oracle_mod, ep, Hkv, d, t.K.astype(np.float64), t.V.astype(np.float64))
    pl = o.pack(ep.roots, 16)
    Q = _packed(t, pl.seg_order, t.Q).astype(np.float64)
    dO = _packed(t, pl.seg_order, t.dO).astype(np.float64)
    dQ, dK, dV = pl.bwd(Q, dO, 0.5)
    rng = np.random.default_rng(seed)
    T, N = o.n_tokens, pl.n_rows
    tok = rng.random(T) < 0.2
    rows = rng.random(N) < 0.2
    dQs, dKs, dVs = pl.bwd(Q, dO, 0.5, need_dq=rows.astype(np.uint8), need_dkdv=tok.astype(np.uint8))
    np.testing.assert_array_equal(dQs[rows], dQ[rows])
    np.testing.assert_allclose(dKs[tok], dK[tok], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dVs[tok], dV[tok], rtol=1e-13, atol=1e-15)
