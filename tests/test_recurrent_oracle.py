"""Pins of the fp64 tree-packed recurrent layer reference (oracle/recurrent.py): closed forms
of the gated delta rule, the DAG propagation against per-row replays of each path taken
from the oracle's own materialised contexts, the mount/fork/rewind rules of the pages,
and finite differences of the backward."""
import numpy as np
import pytest

import synth
import oracle
from oracle import recurrent
from oracle.token_logprob import path_predecessors
from helpers import pool_pages_needed


def _packed(ep, bm=16):
    orc = oracle.Oracle(ep.page_size, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, bm)
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, opl.n_rows)
    return orc, opl, pred


def _inputs(N, H, dk, dv, seed, unit_keys=True):
    rng = np.random.default_rng(seed)
    q = rng.normal(0, 1, (N, H, dk))
    k = rng.normal(0, 1, (N, H, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=2, keepdims=True)
    v = rng.normal(0, 1, (N, H, dv))
    a = rng.uniform(0.6, 1.0, (N, H))
    b = rng.uniform(0.0, 1.0, (N, H))
    return q, k, v, a, b


def _context_path(orc, opl, r):
    """Rows of the path tokens (source -1) of row r's materialised context, in order."""
    tseg, tidx = orc.token_owner()
    base = {int(s): int(x) for s, x in zip(opl.seg_order, opl.seg_row_base)}
    tok, src = opl.row_context(r)
    return [base[int(tseg[t])] + int(tidx[t]) for t, s in zip(tok, src) if s == -1]


@pytest.mark.parametrize("seed", [1, 9, 33])
def test_each_row_equals_a_replay_of_its_path(seed):
    ep = synth.random_dag(seed, page_size=16, max_segments=12, max_len=30)
    orc, opl, pred = _packed(ep)
    N, H, dk, dv = opl.n_rows, 2, 4, 3
    q, k, v, a, b = _inputs(N, H, dk, dv, seed)
    o, _ = recurrent.forward(q, k, v, a, b, pred)
    for r in range(N):
        path = _context_path(orc, opl, r)
        assert path[-1] == r
        for h in range(H):
            S = np.zeros((dv, dk))
            for t in path:                       # one flat sequence, from a zero state
                S = a[t, h] * (S - b[t, h] * np.outer(S @ k[t, h], k[t, h])) + b[t, h] * np.outer(v[t, h], k[t, h])
            np.testing.assert_allclose(o[r, h], S @ q[r, h], rtol=1e-12, atol=1e-12)


def test_unit_write_is_retrieved_exactly():
    """beta = 1 with a unit key: whatever the history and the gate, S_t k_t = v_t."""
    N, H, dk, dv = 40, 3, 5, 4
    q, k, v, a, b = _inputs(N, H, dk, dv, 4)
    b[7], b[23], b[39] = 1.0, 1.0, 1.0
    _, S = recurrent.forward(q, k, v, a, b, np.arange(-1, N - 1))
    for t in (7, 23, 39):
        for h in range(H):
            np.testing.assert_allclose(S[t, h] @ k[t, h], v[t, h], rtol=0, atol=1e-12)


def test_orthogonal_keys_give_gated_linear_attention():
    """Orthonormal keys never interfere, so the delta correction vanishes and
    o_t = sum_{s<=t} (prod_{s<u<=t} alpha_u) beta_s v_s (k_s . q_t)."""
    N, dk, dv = 8, 8, 3
    rng = np.random.default_rng(2)
    basis = np.linalg.qr(rng.normal(0, 1, (dk, dk)))[0]
    k = basis.T[:N][:, None, :]
    q = rng.normal(0, 1, (N, 1, dk))
    v = rng.normal(0, 1, (N, 1, dv))
    a = rng.uniform(0.5, 1.0, (N, 1))
    b = rng.uniform(0.1, 1.0, (N, 1))
    o, _ = recurrent.forward(q, k, v, a, b, np.arange(-1, N - 1))
    for t in range(N):
        want = np.zeros(dv)
        for s in range(t + 1):
            want += np.prod(a[s + 1:t + 1, 0]) * b[s, 0] * v[s, 0] * (k[s, 0] @ q[t, 0])
        np.testing.assert_allclose(o[t, 0], want, rtol=1e-12, atol=1e-12)


def test_second_write_to_a_key_overwrites_the_first():
    k = np.zeros((3, 1, 4))
    k[:, 0, 2] = 1.0
    v = np.array([[[1.0, 2.0]], [[-3.0, 5.0]], [[0.0, 0.0]]])
    q = k.copy()
    a = np.ones((3, 1))
    b = np.array([[1.0], [1.0], [0.0]])
    o, _ = recurrent.forward(q, k, v, a, b, np.array([-1, 0, 1]))
    np.testing.assert_allclose(o[1, 0], [-3.0, 5.0], atol=1e-15)
    np.testing.assert_allclose(o[2, 0], [-3.0, 5.0], atol=1e-15)


def _tree(with_mount):
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 12)
    x, y = ep.fork(r, 2)
    ep.append(x, 9)
    ep.append(y, 14)
    if with_mount:
        ep.mount(x, y, 3, 11)
    ep.append(x, 6)
    x2 = ep.rewind(x, 4)
    ep.append(x2, 5)
    return ep, r, x, y, x2


def test_mounted_spans_are_skipped():
    ep0, *_ = _tree(False)
    ep1, *_ = _tree(True)
    _, opl0, pred0 = _packed(ep0)
    _, opl1, pred1 = _packed(ep1)
    assert opl0.n_rows == opl1.n_rows and np.array_equal(pred0, pred1)
    q, k, v, a, b = _inputs(opl0.n_rows, 2, 4, 3, 6)
    o0, _ = recurrent.forward(q, k, v, a, b, pred0)
    o1, _ = recurrent.forward(q, k, v, a, b, pred1)
    assert np.array_equal(o0, o1)


def test_fork_clones_and_rewind_restores():
    ep, r, x, y, x2 = _tree(True)
    orc, opl, pred = _packed(ep)
    base = {int(s): int(b) for s, b in zip(opl.seg_order, opl.seg_row_base)}
    N, H, dk, dv = opl.n_rows, 1, 4, 3
    q, k, v, a, b = _inputs(N, H, dk, dv, 8)
    for s in (x, y):                      # the children's first tokens see the same inputs
        for arr in (q, k, v, a, b):
            arr[base[s]] = arr[base[x]]
    o, S = recurrent.forward(q, k, v, a, b, pred)
    np.testing.assert_array_equal(o[base[x]], o[base[y]])       # both start from the clone
    # the rewind continuation starts from the state after x's token 3 (h_4 restored)
    want = a[base[x2], 0] * S[base[x] + 3, 0] @ (np.eye(dk) - b[base[x2], 0] * np.outer(k[base[x2], 0], k[base[x2], 0])) \
        + b[base[x2], 0] * np.outer(v[base[x2], 0], k[base[x2], 0])
    np.testing.assert_allclose(S[base[x2], 0], want, rtol=1e-13, atol=1e-13)


def test_backward_by_finite_differences():
    ep, *_ = _tree(True)
    _, opl, pred = _packed(ep)
    N, H, dk, dv = opl.n_rows, 2, 3, 2
    q, k, v, a, b = _inputs(N, H, dk, dv, 11, unit_keys=False)
    rng = np.random.default_rng(12)
    do = rng.normal(0, 1, (N, H, dv))
    grads = recurrent.backward(q, k, v, a, b, pred, do)
    loss = lambda *xs: np.sum(do * recurrent.forward(*xs, pred)[0])
    h = 1e-6
    ins = [q, k, v, a, b]
    for which, g in enumerate(grads):
        x = ins[which]
        flat = x.reshape(-1)
        for idx in rng.choice(flat.size, size=min(flat.size, 40), replace=False):
            keep = flat[idx]
            flat[idx] = keep + h
            lp = loss(*ins)
            flat[idx] = keep - h
            lm = loss(*ins)
            flat[idx] = keep
            num = (lp - lm) / (2 * h)
            assert abs(g.reshape(-1)[idx] - num) <= 1e-6 * max(1.0, abs(num)), (which, idx, g.reshape(-1)[idx], num)
