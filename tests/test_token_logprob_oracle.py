"""Pins of the fp64 per-token log-probability / loss reference (oracle/token_logprob.py)
against things other than itself: the oracle's own path-ordered context lists, library
log-softmax and autograd on a flat sequence, closed forms, and finite differences."""
import math

import numpy as np
import pytest

import synth
import oracle
from oracle.token_logprob import path_predecessors, token_logprob
from helpers import pool_pages_needed

torch = pytest.importorskip("torch")
scipy_special = pytest.importorskip("scipy.special")


def _packed(ep, bm=16):
    orc = oracle.Oracle(ep.page_size, pool_pages_needed(ep), 1, 8)
    orc.replay(ep)
    opl = orc.pack(ep.roots, bm)
    pred = path_predecessors(orc.seg_info, opl.seg_order, opl.seg_row_base, opl.n_rows)
    return orc, opl, pred


def _pred_from_contexts(orc, opl):
    """The previous path token (source -1) of each row's materialised context, whose items
    come in path order with mounted spans spliced in at their points."""
    tseg, tidx = orc.token_owner()
    base = {int(s): int(b) for s, b in zip(opl.seg_order, opl.seg_row_base)}
    out = np.full(opl.n_rows, -1, dtype=np.int64)
    for r in range(opl.n_rows):
        tok, src = opl.row_context(r)
        path = [int(t) for t, s in zip(tok, src) if s == -1]
        assert base[int(tseg[path[-1]])] + int(tidx[path[-1]]) == r   # the row's own token is last
        if len(path) >= 2:
            p = path[-2]
            out[r] = base[int(tseg[p])] + int(tidx[p])
    return out


@pytest.mark.parametrize("seed", [3, 11, 27, 58])
def test_predecessors_match_the_context_order(seed):
    ep = synth.random_dag(seed, page_size=16, max_segments=14, max_len=60)
    orc, opl, pred = _packed(ep)
    assert np.array_equal(pred, _pred_from_contexts(orc, opl))


def test_fork_rewind_and_mount_predecessors():
    # root 20 tokens, forked in three; child 0 rewound to 5 (tail 5..12 stays, the
    # continuation starts after token 4); child 2 mounts a span of child 1
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 20)
    a, b, c = ep.fork(r, 3)
    ep.append(a, 12)
    ep.append(b, 9)
    a2 = ep.rewind(a, 5)
    ep.append(a2, 4)
    ep.append(c, 3)
    ep.mount(c, b, 2, 7)
    ep.append(c, 6)
    orc, opl, pred = _packed(ep)
    base = {int(s): int(x) for s, x in zip(opl.seg_order, opl.seg_row_base)}
    last_root = base[r] + 19
    assert pred[base[r]] == -1
    for s in (a, b, c):                       # every child starts after the root's last token
        assert pred[base[s]] == last_root
    assert pred[base[a2]] == base[a] + 4      # the continuation follows token 4 of the rewound child
    assert pred[base[a] + 5] == base[a] + 4   # and so does the dead-end tail
    assert pred[base[c] + 3] == base[c] + 2   # the mount changes no predecessor
    # rows feeding several terms: the root's last row (3 children), child a's row 4 (2)
    counts = np.bincount(pred[pred >= 0], minlength=opl.n_rows)
    assert counts[last_root] == 3 and counts[base[a] + 4] == 2
    assert np.array_equal(pred, _pred_from_contexts(orc, opl))


def test_single_sequence_is_library_log_softmax():
    rng = np.random.default_rng(0)
    N, V = 40, 57
    x = rng.normal(0, 2.0, (N, V))
    ids = rng.integers(0, V, N)
    w = rng.uniform(0, 1, N)
    pred = np.arange(-1, N - 1)
    logp, lse, loss, dx = token_logprob(x, ids, w, pred)
    ref = scipy_special.log_softmax(x[:-1], axis=1)[np.arange(N - 1), ids[1:]]
    assert logp[0] == 0.0
    np.testing.assert_allclose(logp[1:], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, scipy_special.logsumexp(x, axis=1), rtol=1e-14)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    lp = torch.log_softmax(xt[:-1], dim=1).gather(1, torch.tensor(ids[1:]).unsqueeze(1))[:, 0]
    lt = -(torch.tensor(w[1:]) * lp).sum()
    lt.backward()
    assert abs(loss - lt.item()) < 1e-10
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-12)


def test_uniform_logits_closed_form():
    N, V = 9, 1000
    x = np.full((N, V), 3.25)
    ids = np.arange(N) * 7
    w = np.linspace(0.5, 2.0, N)
    pred = np.array([-1, 0, 1, 2, 2, 4, 5, 5, 5])   # rows 2 and 5 feed several tokens
    logp, lse, loss, dx = token_logprob(x, ids, w, pred)
    np.testing.assert_allclose(lse, 3.25 + math.log(V), rtol=1e-15)
    np.testing.assert_allclose(logp[1:], -math.log(V), rtol=1e-13)
    assert abs(loss - w[1:].sum() * math.log(V)) < 1e-11
    for r in range(N):
        kids = np.nonzero(pred == r)[0]
        want = np.full(V, w[kids].sum() / V)
        for t in kids:
            want[ids[t]] -= w[t]
        np.testing.assert_allclose(dx[r], want, rtol=0, atol=1e-15)


def test_two_token_vocabulary():
    x = np.array([[0.3, -1.7], [2.0, 2.5], [-4.0, 1.0]])
    ids = np.array([0, 1, 0])
    logp, _, _, _ = token_logprob(x, ids, None, np.array([-1, 0, 1]))
    # log p(token k) with two classes = -log(1 + exp(x_other - x_k))
    assert abs(logp[1] - (-math.log1p(math.exp(0.3 - (-1.7))))) < 1e-14
    assert abs(logp[2] - (-math.log1p(math.exp(2.5 - 2.0)))) < 1e-14


def test_gradient_by_finite_differences():
    ep = synth.Episode(16)
    r = ep.root()
    ep.append(r, 6)
    a, b = ep.fork(r, 2)
    ep.append(a, 4)
    ep.append(b, 3)
    a2 = ep.rewind(a, 2)
    ep.append(a2, 2)
    orc, opl, pred = _packed(ep)
    N, V = opl.n_rows, 5
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (N, V))
    ids = rng.integers(0, V, N)
    w = rng.uniform(-1, 1, N)
    _, _, _, dx = token_logprob(x, ids, w, pred)
    h = 1e-6
    num = np.zeros_like(x)
    for i in range(N):
        for v in range(V):
            xp, xm = x.copy(), x.copy()
            xp[i, v] += h
            xm[i, v] -= h
            num[i, v] = (token_logprob(xp, ids, w, pred)[2] - token_logprob(xm, ids, w, pred)[2]) / (2 * h)
    np.testing.assert_allclose(dx, num, rtol=0, atol=1e-7)


def test_each_owned_token_counted_once():
    """Single ownership: summing the per-path flat losses of every root-to-leaf path, each
    owned token taken once (the first path that reaches it), gives the packed loss."""
    ep = synth.random_dag(41, page_size=16, max_segments=12, max_len=40)
    orc, opl, pred = _packed(ep)
    N, V = opl.n_rows, 11
    rng = np.random.default_rng(2)
    x = rng.normal(0, 1, (N, V))
    ids = rng.integers(0, V, N)
    w = rng.uniform(0, 1, N)
    _, _, loss, _ = token_logprob(x, ids, w, pred)
    ctx_pred = _pred_from_contexts(orc, opl)
    seen = np.zeros(N, dtype=bool)
    total = 0.0
    for leaf in range(N):                     # every row's path ends at that row
        t = leaf
        while t >= 0 and not seen[t]:
            seen[t] = True
            p = ctx_pred[t]
            if p >= 0:
                row = x[p]
                total -= w[t] * (row[ids[t]] - scipy_special.logsumexp(row))
            t = p
    assert seen.all()
    assert abs(total - loss) < 1e-9 * max(1.0, abs(loss))
