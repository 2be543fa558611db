"""The oracle's rotary embedding pinned to closed forms, and the two properties the pages
tie it to: a mount reads keys rotation-free (zero-copy mount == copy of the stored, rotated
rows), and the monotonic offset keeps every mounted key before the reader's later queries
(without it a longer sibling's keys overtake them: the "RoPE flip" of unshifted
zero-copy KV in the Octopus project page's cross-branch sharing table)."""
import math

import numpy as np
import pytest

import synth
from test_oracle import _copy_variant, _replay


def test_rope_is_identity_at_position_zero(oracle_mod):
    x = np.random.default_rng(0).standard_normal((3, 2, 8))
    y = oracle_mod.rope(x, [0, 0, 0], 10000.0)
    assert np.array_equal(y, x)


def test_rope_d2_is_the_rotation_matrix(oracle_mod):
    # d = 2: one pair, angle pos * base^0 = pos radians, whatever the base
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 2))
    pos = [0, 1, 7, 1000, 123457]
    y = oracle_mod.rope(x, pos, 500.0)
    for t, p in enumerate(pos):
        R = np.array([[math.cos(p), -math.sin(p)], [math.sin(p), math.cos(p)]])
        for h in range(3):
            np.testing.assert_allclose(y[t, h], R @ x[t, h], rtol=0, atol=1e-12)


def test_rope_d4_pairs_and_frequencies(oracle_mod):
    # d = 4: pair (0, 2) turns by pos, pair (1, 3) by pos * base^(-1/2)
    base = 10000.0
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    p = 3
    y = oracle_mod.rope(x, [p], base)[0, 0]
    t0, t1 = p, p * base ** -0.5
    want = [math.cos(t0) * 1 - math.sin(t0) * 3, math.cos(t1) * 2 - math.sin(t1) * 4,
            math.sin(t0) * 1 + math.cos(t0) * 3, math.sin(t1) * 2 + math.cos(t1) * 4]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_rope_inverse_and_norm(oracle_mod):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 4, 128))
    pos = rng.integers(0, 1_000_000, 16)
    y = oracle_mod.rope(x, pos, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=2), np.linalg.norm(x, axis=2), rtol=1e-13)
    z = oracle_mod.rope(y, pos, 10000.0, inverse=True)
    np.testing.assert_allclose(z, x, rtol=0, atol=1e-11)


def test_rope_scores_depend_on_position_difference(oracle_mod):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    base = 10000.0
    s0 = float(np.sum(oracle_mod.rope(q, [40], base) * oracle_mod.rope(k, [13], base)))
    for shift in (1, 977, 250_000):
        s1 = float(np.sum(oracle_mod.rope(q, [40 + shift], base) * oracle_mod.rope(k, [13 + shift], base)))
        assert abs(s1 - s0) <= 1e-9 * (1 + abs(s0))
    # and only on it: another difference gives another score
    s2 = float(np.sum(oracle_mod.rope(q, [41], base) * oracle_mod.rope(k, [13], base)))
    assert abs(s2 - s0) > 1e-6


def _longer_sibling():
    ep = synth.Episode(8)
    r = ep.root(); ep.append(r, 13)
    a, b, c = ep.fork(r, 3)
    ep.append(a, 30); ep.append(b, 9)
    ep.mount(b, a, 5, 22)          # the sibling's span ends past the reader's position
    ep.append(b, 11)
    ep.append(c, 40)
    return ep


@pytest.mark.parametrize("seed", [None, 11, 12, 13])
def test_offset_keeps_mounted_keys_before_the_reader(oracle_mod, seed):
    """With s = max(p_B, e_A + 1) every reader row after the mount point sits at least two
    positions past every mounted key; the unshifted rule (s = p_B) would put some of
    them at or before a longer sibling's keys."""
    ep = _longer_sibling() if seed is None else synth.random_dag(seed, page_size=8, max_segments=12, max_len=60)
    o = _replay(oracle_mod, ep, 1, 8)
    flips = 0
    for i in range(o.n_mounts):
        reader, m, prod, a, b = o.mount_info(i)
        kpos = o.seg_pos(prod)[a:b]
        rpos = o.seg_pos(reader)
        after = rpos[m:]
        if len(after) == 0:
            continue
        assert int(after.min()) >= int(kpos.max()) + 2
        # unshifted: the reader's first row after the mount would be at p_B, its position
        # with nothing mounted (one past its previous row)
        p_b = int(rpos[m - 1]) + 1 if m > 0 else None
        if p_b is not None and p_b <= int(kpos.max()):
            flips += 1
    if seed is None:
        assert flips == 1


@pytest.mark.parametrize("case", ["tiny", "two_readers"])
def test_rotation_free_mount_equals_copy(oracle_mod, case):
    """Keys rotated once at their own positions and read as stored by the mount give the
    same outputs and gradients as a physical copy of those stored rows (queries rotated at
    the reader's positions in both)."""
    if case == "tiny":
        ep = synth.make_preset("tiny")
        Hq, Hkv, d = 1, 1, 64
    else:
        ep = _longer_sibling()
        Hq, Hkv, d = 4, 2, 8
    base = 10000.0
    t = synth.make_tensors(ep, Hq, Hkv, d, "f32", 1.0, 5)
    tok_pos = _replay_positions(oracle_mod, ep, Hkv, d)
    K = oracle_mod.rope(t.K, tok_pos, base)
    V = t.V.astype(np.float64)
    ep2, K2, V2, cmap = _copy_variant(ep, K, V, 0)
    o1 = _replay(oracle_mod, ep, Hkv, d, K, V)
    o2 = _replay(oracle_mod, ep2, Hkv, d, K2, V2)
    p1, p2 = o1.pack(ep.roots, 16), o2.pack(ep2.roots, 16)
    m = [op for op in ep.ops if op[0] == "mount"][0]
    reader, span = m[1], m[4] - m[3]
    mpt = o1.mount_info(0)[1]
    rows2 = []
    for si, s in enumerate(p1.seg_order.tolist()):
        n = o1.seg_info(s)["len"]
        for i in range(n):
            rows2.append(p2.seg_row_base[si] + (i if (s != reader or i < mpt) else i + span))
    rows2 = np.array(rows2)
    rng = np.random.default_rng(9)
    # queries rotated at the mount variant's row positions, the same values in both
    Q1 = oracle_mod.rope(rng.standard_normal((p1.n_rows, Hq, d)), p1.row_pos, base)
    Q2 = np.zeros((p2.n_rows, Hq, d))
    Q2[rows2] = Q1
    scale = 1 / math.sqrt(d)
    O1, L1 = p1.fwd(Q1, scale)
    O2, L2 = p2.fwd(Q2, scale)
    np.testing.assert_allclose(O2[rows2], O1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L2[:, rows2], L1, rtol=1e-12, atol=1e-12)


def _replay_positions(oracle_mod, ep, Hkv, d):
    o = oracle_mod.Oracle(ep.page_size, 4096, Hkv, d)
    return o.replay(ep)
