"""Chunk-wise (WY / UT-transform) form of the gated delta-rule recurrence, fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It exists to pin the
chunk algebra that the CUDA scan is built on: the tests require it to agree
with the token-sequential oracle to fp64 round-off.

Within a chunk of n tokens starting from state S0, with G_i the running sum
of lam = log g inside the chunk (G_i = lam_1 + ... + lam_i):

  unrolling S_i = g_i S_{i-1} + k_i u_i^T gives
      S_i = e^{G_i} S0 + sum_{j<=i} e^{G_i - G_j} k_j u_j^T,
  and substituting it into u_i = beta_i (v_i - (g_i S_{i-1})^T k_i) gives
      u_i + sum_{j<i} A_ij u_j = beta_i v_i - beta_i e^{G_i} S0^T k_i,
      A_ij = beta_i e^{G_i - G_j} (k_i . k_j)   (j < i),
  i.e.  (I + A) U = X  with  X = diag(beta) V - diag(beta e^G) K S0.
  Then
      O     = diag(e^G) Qs S0 + P U,  P_ij = e^{G_i - G_j} (qs_i . k_j) (j <= i)
      S_end = e^{G_n} S0 + (diag(e^{G_n - G_j}) K)^T U
  with qs = q / sqrt(dk).  The unit lower-triangular system is solved with a
  library triangular solve; every other step is a plain matrix product.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def scan_head_chunked(q, k, v, lam, beta, S0, chunk: int = 64):
    """One value head.  q, k [T, dk]; v [T, dv]; lam, beta [T]; S0 [dk, dv]
    -> (o [T, dv], S_end [dk, dv]), all float64."""
    q, k, v, lam, beta, S = (np.asarray(x, dtype=np.float64) for x in (q, k, v, lam, beta, S0))
    S = S.copy()
    T, dk = q.shape
    o = np.empty((T, v.shape[1]))
    qs = q / np.sqrt(dk)
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        n = c1 - c0
        K, Q, V, b = k[c0:c1], qs[c0:c1], v[c0:c1], beta[c0:c1]
        G = np.cumsum(lam[c0:c1])
        ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        diff = G[:, None] - G[None, :]
        # e^{G_i - G_j} on and below the diagonal, 0 above it (never exponentiate
        # the positive differences above the diagonal)
        decay_incl = np.exp(np.where(jj <= ii, diff, -np.inf))
        decay_strict = np.where(jj < ii, decay_incl, 0.0)
        A = b[:, None] * decay_strict * (K @ K.T)
        X = b[:, None] * V - (b * np.exp(G))[:, None] * (K @ S)
        U = solve_triangular(np.eye(n) + A, X, lower=True, unit_diagonal=True)
        P = decay_incl * (Q @ K.T)
        o[c0:c1] = np.exp(G)[:, None] * (Q @ S) + P @ U
        S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * K).T @ U
    return o, S
