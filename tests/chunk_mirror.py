"""Chunk-form KDA in fp64 numpy -- a test artifact, not a kernel.

A second, independent evaluation of the gated delta rule with per-channel
decay, written in the chunked (WY / UT) form that the CUDA prefill uses, so
that the algebra of that form is checked against the token-by-token oracle
before any GPU code is trusted.  Within a chunk of rows r = 0..C-1 with
inclusive cumulative log-decay G_r = g_0 + ... + g_r (per key channel) and
chunk-start state S:

  A[r,j]   = beta_r sum_c k_r[c] k_j[c] exp(G_r[c] - G_j[c])      (j < r)
  Aqk[r,j] = sum_c q_r[c] k_j[c] exp(G_r[c] - G_j[c])             (j <= r)
  Tm       = (I + A)^-1                    (unit lower-triangular)
  W        = Tm Diag(beta) (K * exp(G)),   U0 = Tm Diag(beta) V
  U        = U0 - W S                      (the delta-rule residuals u_r)
  O        = scale ((Q * exp(G)) S + Aqk U)
  S_next   = Diag(exp(G_last)) S + (K * exp(G_last - G))^T U

Chunks restart at every sequence start; the last chunk may be partial.
"""
from __future__ import annotations

import numpy as np


def chunk_prefill(q, k, v, g, beta, cu_seqlens, state_indices, pool, *, chunk,
                  checkpoint_every=0, scale=None):
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    pool = np.array(pool, np.float64, copy=True)
    cu = np.asarray(cu_seqlens, np.int64)
    T, H, dk = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    out = np.zeros((T, H, dv))
    ckpts = []
    for i in range(len(cu) - 1):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        slot = int(state_indices[i])
        if slot < 0 or t1 == t0:
            continue
        seq_ck = []
        for h in range(H):
            S = pool[slot, h].copy()
            per_head = []
            for c0 in range(t0, t1, chunk):
                c1 = min(c0 + chunk, t1)
                Q, K, V = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
                B = beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h], axis=0)
                n = c1 - c0
                low = np.tril(np.ones((n, n), bool))
                D = G[:, None, :] - G[None, :, :]
                D = np.where(low[:, :, None], D, -np.inf)
                E = np.exp(D)
                Akk = B[:, None] * np.einsum("rc,jc,rjc->rj", K, K, E)
                Akk = np.tril(Akk, -1)
                Aqk = np.einsum("rc,jc,rjc->rj", Q, K, E)
                Tm = np.linalg.inv(np.eye(n) + Akk)
                W = Tm @ (B[:, None] * K * np.exp(G))
                U0 = Tm @ (B[:, None] * V)
                U = U0 - W @ S
                out[c0:c1, h] = scale * ((Q * np.exp(G)) @ S + Aqk @ U)
                gl = G[-1]
                S = np.exp(gl)[:, None] * S + (K * np.exp(gl - G)).T @ U
                if checkpoint_every and (c1 - t0) % checkpoint_every == 0:
                    per_head.append(S.copy())
            pool[slot, h] = S
            seq_ck.append(per_head)
        if checkpoint_every:
            for m in range(len(seq_ck[0])):
                ckpts.append(np.stack([seq_ck[h][m] for h in range(H)]))
    ck = np.stack(ckpts) if ckpts else np.zeros((0, H, dk, dv))
    return out, pool, ck
