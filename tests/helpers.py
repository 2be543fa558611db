"""Test helpers: replay a synth.Episode into the library pool and into the oracle, and
compare their outputs.  Test infrastructure only."""
from __future__ import annotations

import re
import os

import numpy as np

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# tolerances of the parity bar: |err| <= atol + rtol * |ref|
TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 2e-2)}


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "octopus.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(octo_[a-z_0-9]+)\s*\(", txt)))


def header_param_counts():
    """Number of parameters of every octo_ function the header declares (void = 0)."""
    txt = open(os.path.join(ROOT, "include", "octopus.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(octo_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", txt, flags=re.S):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def replay_host(pool, ep):
    """Replays the op log into a library pool without K/V (metadata only)."""
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
        elif k == "release":
            pool.release(op[1])
        elif k == "unpin":
            pool.unpin(op[1])


def replay_device(pool, ep, K_dev, V_dev, stream=None, rope_base=None):
    """Replays the op log into a library pool, appending each token's K/V rows from
    device tensors K_dev/V_dev [T, Hkv, d] (append order); with rope_base the K rows are
    rotated at their positions on the way in (octo_append_rope).  Returns the positions
    the pool gave the tokens, in append order."""
    t = 0
    positions = []
    for op in ep.ops:
        k = op[0]
        if k == "append":
            _, c, n = op
            if rope_base is None:
                positions.extend(pool.append(c, n, K_dev[t:t + n], V_dev[t:t + n], stream=stream).tolist())
            else:
                positions.extend(pool.append_rope(c, n, K_dev[t:t + n], V_dev[t:t + n], rope_base,
                                                  stream=stream).tolist())
            t += n
        elif k == "root":
            pool.root()
        elif k == "fork":
            pool.fork(op[1], op[2])
        elif k == "mount":
            pool.mount(*op[1:])
        elif k == "rewind":
            pool.rewind(op[1], op[2])
        elif k == "done":
            pool.done(op[1])
        elif k == "release":
            pool.release(op[1])
        elif k == "unpin":
            pool.unpin(op[1])
    return np.array(positions, dtype=np.int32)


def compare_pools(pool, orc):
    assert pool.info()["n_segments"] == orc.n_segments
    assert pool.info()["free_pages"] == orc.free_pages()
    assert pool.info()["n_mounts"] == orc.n_mounts
    for s in range(orc.n_segments):
        a, b = pool.seg_info(s), orc.seg_info(s)
        assert a == b, (s, a, b)
        assert np.array_equal(pool.seg_pos(s), orc.seg_pos(s)), s
        assert np.array_equal(pool.seg_pages(s), orc.seg_pages(s)), s


def oracle_entries(opl):
    return opl.entries.astype(np.int64)


def product_entries(ent):
    return np.stack([ent[f].astype(np.int64) for f in ("q_tile", "kv_page", "kv_lo", "kv_hi", "q_lo", "flags",
                                                         "diag", "src")], axis=1) if len(ent) else \
        np.zeros((0, 8), dtype=np.int64)


def compare_plans(gp, opl):
    """Bit-exact comparison of a library plan (copy_out dict) with an oracle plan."""
    assert np.array_equal(gp["seg_order"], opl.seg_order)
    assert np.array_equal(gp["seg_row_base"], opl.seg_row_base)
    assert np.array_equal(gp["row_pos"], opl.row_pos)
    assert np.array_equal(gp["tile_seg"], opl.tile_seg)
    assert np.array_equal(gp["tile_t0"], opl.tile_t0)
    assert np.array_equal(gp["tile_rows"], opl.tile_rows)
    assert np.array_equal(gp["tile_off"], opl.tile_off)
    pe, oe = product_entries(gp["entries"]), oracle_entries(opl)
    assert pe.shape == oe.shape, (pe.shape, oe.shape)
    if not np.array_equal(pe, oe):
        bad = np.nonzero((pe != oe).any(1))[0][:5]
        raise AssertionError("entries differ at %s:\nlib %s\noracle %s" % (bad, pe[bad], oe[bad]))
    assert np.array_equal(gp["csc_perm"], opl.csc_perm)
    assert np.array_equal(gp["page_off"], opl.page_off)


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        raise AssertionError("%s: %d of %d outside |err| <= %g + %g|ref|; worst at %s: got %r ref %r" % (
            what, int(bad.sum()), bad.size, atol, rtol, np.unravel_index(i, got.shape), got.flat[i], ref.flat[i]))


def packed(t, seg_order, arr):
    if len(seg_order) == 0:
        return arr[:0]
    return np.concatenate([arr[t.seg_off[s]:t.seg_off[s + 1]] for s in seg_order], axis=0)


def pool_pages_needed(ep):
    P = ep.page_size
    return sum((L + P - 1) // P for L in ep.length) + 4


def oracle_checked_dag(oracle_mod, seed, page_size=16, max_segments=12, max_len=80, n_roots=1, steps=160):
    """Random episodes whose mounts are drawn from every segment and span, kept only when
    the oracle's own pool accepts them: besides sibling spans this gives spans of an
    ancestor's tokens past the fork point, second and third disjoint spans of a producer
    the lineage already mounted, and spans of segments the reader's parent mounted.  Forks,
    rewinds and appends as in synth.random_dag."""
    rng = np.random.default_rng(np.random.PCG64(seed))
    ep = synth.Episode(page_size)
    orc = oracle_mod.Oracle(page_size, 1 << 16, 1, 8)
    fork_of = {}
    for _ in range(n_roots):
        r = ep.root()
        orc.root()
        n = int(rng.integers(1, max_len))
        ep.append(r, n)
        orc.append(r, n)

    def lineage(c):
        out = []
        while c >= 0:
            out.append(c)
            c = ep.parent[c]
        return out

    def try_mount(c, p, a, b):
        if orc.mount(c, p, a, b, check=False) == oracle_mod.OK:
            ep.mount(c, p, a, b, checked=False)
            return True
        return False

    for _ in range(steps):
        if ep.n_segments >= max_segments * n_roots:
            break
        live = [c for c in range(ep.n_segments) if ep.appendable[c]]
        if not live:
            break
        c = live[int(rng.integers(0, len(live)))]
        u = rng.random()
        if u < 0.3:
            n = int(rng.integers(1, max_len))
            ep.append(c, n)
            orc.append(c, n)
        elif u < 0.45:
            k = int(rng.integers(1, 4))
            kids = ep.fork(c, k)
            orc.fork(c, k)
            for kid in kids:
                fork_of[kid] = ep.length[c]
                n = int(rng.integers(0, max_len))
                ep.append(kid, n)
                orc.append(kid, n)
        elif u < 0.85:
            lin = lineage(c)
            kind = rng.random()
            if kind < 0.35 and len(lin) > 1:
                # an ancestor's own tokens past the point its lineage child forked at
                j = int(rng.integers(1, len(lin)))
                x, f = lin[j], fork_of.get(lin[j - 1], 0)
                if ep.length[x] > f:
                    a = int(rng.integers(f, ep.length[x]))
                    b = int(rng.integers(a + 1, ep.length[x] + 1))
                    try_mount(c, x, a, b)
            else:
                # any other segment: a producer mounted before on the lineage half the time
                prev = [p for (rr, p) in ep.mounted if rr in lin]
                if prev and kind < 0.65:
                    p = prev[int(rng.integers(0, len(prev)))]
                else:
                    p = int(rng.integers(0, ep.n_segments))
                if ep.length[p] > 0:
                    a = int(rng.integers(0, ep.length[p]))
                    b = int(rng.integers(a + 1, min(ep.length[p], a + max_len) + 1))
                    try_mount(c, p, a, b)
            n = int(rng.integers(0, max_len // 2 + 1))
            ep.append(c, n)
            orc.append(c, n)
        elif u < 0.95:
            if ep.length[c] > 0:
                k = int(rng.integers(0, ep.length[c] + 1))
                nid = ep.rewind(c, k)
                orc.rewind(c, k)
                fork_of[nid] = k
                n = int(rng.integers(0, max_len))
                ep.append(nid, n)
                orc.append(nid, n)
        else:
            ep.done(c)
            orc.done(c)
    return ep


def mount_kinds(ep):
    """Counts of the mount kinds in an op log: (ancestor spans, repeated producers)."""
    parent, anc, rep = {}, 0, 0
    seen = set()
    nseg = 0
    for op in ep.ops:
        if op[0] == "root":
            parent[nseg] = -1
            nseg += 1
        elif op[0] == "fork":
            for _ in range(op[2]):
                parent[nseg] = op[1]
                nseg += 1
        elif op[0] == "rewind":
            parent[nseg] = op[1]
            nseg += 1
        elif op[0] == "mount":
            r, p = op[1], op[2]
            lin = []
            x = r
            while x >= 0:
                lin.append(x)
                x = parent[x]
            if p in lin:
                anc += 1
            if any((y, p) in seen for y in lin):
                rep += 1
            seen.add((r, p))
    return anc, rep
