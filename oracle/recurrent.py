"""fp64 reference of the tree-packed recurrent layer -- TEST INFRASTRUCTURE ONLY (like the
rest of this package: only tests/, the smoke check and the CPU baseline may import it).

What the pages fix:
* ia.com.br summary, section on associative versus working memory: the hybrid model pairs
  full-attention layers with linear-recurrent layers (Gated DeltaNet / Mamba-2) whose
  state is the branch's mutable working memory h.
* Octopus project page, five-primitives table: fork clones the recurrent checkpoint at the
  fork point; read_thread mounts a sibling's KV into the attention layers only and the
  recurrent layers skip the span; rewind restores the exact state h_k of step k.
* "Architecture & Co-Design" item 03: the packed pass compiles the branched trees together
  with the recurrent boundary checkpoints.

Readings (the pages name the family, not the equations):
* The recurrence is the gated delta rule of Gated DeltaNet, per head, state S of shape
  [d_v, d_k]:   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
                o_t = S_t q_t.
  q, k, v, alpha, beta are the scan's inputs (feature maps, normalisation and gate
  activations are computed before the scan and are outside it).
* Over the episode DAG the state of a token is the recurrence along its path: the state
  after a token t starts from the state after pred(t), the token before t on its path --
  the previous own token, or for a segment's first token the parent's token at the fork
  point minus one (so a fork clones the state there and a rewind continuation restores the
  state after step k); mounted spans never enter the recurrence.  A path start begins from
  S = 0.  pred is the same map as for the per-token log-probability
  (oracle.token_logprob.path_predecessors); packed rows come parents-first, so pred(t) < t.
"""
from __future__ import annotations

import numpy as np


def forward(q, k, v, alpha, beta, pred):
    """o [N, H, d_v] and the state after every row S [N, H, d_v, d_k] (fp64) for inputs
    q, k [N, H, d_k], v [N, H, d_v], alpha, beta [N, H] in packed row order."""
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    alpha, beta = np.asarray(alpha, dtype=np.float64), np.asarray(beta, dtype=np.float64)
    N, H, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((N, H, dv, dk))
    o = np.zeros((N, H, dv))
    eye = np.eye(dk)
    for t in range(N):
        p = pred[t]
        for h in range(H):
            prev = S[p, h] if p >= 0 else np.zeros((dv, dk))
            kt = k[t, h]
            S[t, h] = alpha[t, h] * prev @ (eye - beta[t, h] * np.outer(kt, kt)) + beta[t, h] * np.outer(v[t, h], kt)
            o[t, h] = S[t, h] @ q[t, h]
    return o, S


def backward(q, k, v, alpha, beta, pred, do):
    """Gradients dq, dk, dv, dalpha, dbeta of sum(do * o) through the DAG recurrence: the
    gradient reaching a row's previous state goes to pred(row), summed over every row that
    continues from it (fork and rewind points feed several)."""
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    alpha, beta = np.asarray(alpha, dtype=np.float64), np.asarray(beta, dtype=np.float64)
    N, H, dk = k.shape
    dv = v.shape[2]
    _, S = forward(q, k, v, alpha, beta, pred)
    G = np.zeros((N, H, dv, dk))          # gradient with respect to the state after each row
    dq, dkk, dvv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    da, db = np.zeros_like(alpha), np.zeros_like(beta)
    eye = np.eye(dk)
    for t in range(N - 1, -1, -1):        # successors come later in packed order
        p = pred[t]
        for h in range(H):
            A = S[p, h] if p >= 0 else np.zeros((dv, dk))
            kt, vt, a, b = k[t, h], v[t, h], alpha[t, h], beta[t, h]
            g = G[t, h] + np.outer(do[t, h], q[t, h])
            M = eye - b * np.outer(kt, kt)
            dq[t, h] = S[t, h].T @ do[t, h]
            dvv[t, h] = b * g @ kt
            da[t, h] = np.sum(g * (A @ M))
            db[t, h] = -a * kt @ g.T @ A @ kt + vt @ g @ kt
            dkk[t, h] = -a * b * (A.T @ g + g.T @ A) @ kt + b * g.T @ vt
            if p >= 0:
                G[p, h] += a * g @ M
    return dq, dkk, dvv, da, db
