"""fp64 reference of the per-token log-probability and loss over packed rows -- TEST
INFRASTRUCTURE ONLY (like the rest of this package: only tests/, the smoke check and the
CPU baseline may import it; the library never does).

What the pages fix, and the readings taken where they leave a step open:

* Octopus project page, "Architecture & Co-Design" item 03 (1D packed DAG-GRPO): every
  branch of an episode is trained in one unpadded packed pass, and single-ownership
  masking deduplicates the shared prefixes.  rit.work summary, section "the neighbour's
  context attaches only to attention layers": the shared prefix enters the loss once.
  Reading: each owned token is one packed row, and its term enters the loss exactly once.
* The term of a token is its log-probability under the model output at the row of the
  token right before it on its path (next-token prediction; the pages do not spell the
  objective out).  That predecessor is the previous own token of its segment; for a
  segment's first token it is the parent's token at the fork point minus one, walking up
  through forks at point 0; a root's first token has none (its term is 0 and it is not
  counted).  A row can therefore feed several terms: the last row before a fork feeds
  every child's first token, and the row before a rewind point feeds both the
  continuation and the dead-end tail (which the five-primitives table, row rewind, keeps
  in the credit graph).
* Mounted spans are context only: the five-primitives table, row read_thread, has the
  recurrent layers skip the span, so the reader's sequence continues from its own last
  token and a mount changes no predecessor.
* Five-primitives table, row done: the close reminder is untrainable (mask m = 0); the
  mask and the branch's credit enter as one weight per token, w_t = m_{l,t} * A_l,
  supplied by the caller (the leave-one-branch-out credit itself is not computed here).

Definitions (x the logits rows, y the token ids, w the weights):
    pred(t)     as above, -1 when none
    lse(r)      = log sum_v exp(x[r, v])
    logp(t)     = x[pred(t), y_t] - lse(pred(t))           (0 when pred(t) = -1)
    loss        = - sum_t w_t logp(t)
    dloss/dx[r, v] = sum over t with pred(t) = r of  w_t (exp(x[r, v] - lse(r)) - [v == y_t])
"""
from __future__ import annotations

import numpy as np


def path_predecessors(seg_info, seg_order, seg_row_base, n_rows):
    """pred[t] for every packed row t: the packed row of the token before it on its path.

    seg_info(s) -> dict with the segment's "parent", "fork" and "len"; seg_order and
    seg_row_base are the packed segments and their first rows."""
    base = {int(s): int(b) for s, b in zip(seg_order, seg_row_base)}
    pred = np.full(n_rows, -1, dtype=np.int64)
    for s, b in base.items():
        info = seg_info(s)
        n = info["len"]
        if n == 0:
            continue
        pred[b + 1:b + n] = np.arange(b, b + n - 1)
        parent, f = info["parent"], info["fork"]
        while parent >= 0 and f == 0:       # a fork at point 0 shows none of the parent
            up = seg_info(parent)
            parent, f = up["parent"], up["fork"]
        if parent >= 0:
            pred[b] = base[parent] + f - 1
    return pred


def logsumexp_rows(x):
    """log sum exp of every row, shifted by the row maximum."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=1)
    return m + np.log(np.exp(x - m[:, None]).sum(axis=1))


def token_logprob(x, ids, weight, pred):
    """Returns logp [N], lse [N], loss, dx [N, V] (all fp64) for logits x [N, V] (rows in
    packed order), token ids [N], weights [N] (None: ones) and predecessors [N]."""
    x = np.asarray(x, dtype=np.float64)
    N, V = x.shape
    ids = np.asarray(ids, dtype=np.int64)
    w = np.ones(N) if weight is None else np.asarray(weight, dtype=np.float64)
    pred = np.asarray(pred, dtype=np.int64)
    lse = logsumexp_rows(x)
    logp = np.zeros(N)
    dx = np.zeros_like(x)
    loss = 0.0
    for t in range(N):
        r = pred[t]
        if r < 0:
            continue
        logp[t] = x[r, ids[t]] - lse[r]
        loss -= w[t] * logp[t]
        dx[r] += w[t] * np.exp(x[r] - lse[r])
        dx[r, ids[t]] -= w[t]
    return logp, lse, loss, dx
