"""fp64 NumPy restatement of the chunkwise form of the KLA / gated delta-rule recurrence.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows GeekNews "Revisando las variantes de atencion lineal de la familia
DeltaNet", section "KDA por chunks: reordenar la recurrencia como
multiplicaciones de matrices", step by step and in that page's own orientation:
the state is kept as a d_v x d_k matrix ``M`` (value rows, key columns), keys act
from the right, and the read is ``o = M q``. The result is transposed to the
d_k x d_v orientation of the KLA page only at the very end, so a transposition
mistake on either side shows up when the two oracles are compared.

The step size is the KLA coefficient beta_i = eta_i / (||k_i||^2 + eps)
(Gist.science KLA summary, "La Regola di Aggiornamento KLA"); that page's
"Implementazione" section states that it enters the chunk solver only through
the diagonal B = Diag(beta_1..beta_C). The read scale ``s`` of the chunk page
is 1 (the KLA recurrence has no query scale).

Per chunk c with incoming state M_c, tokens i = 0..L-1 (L <= C):

  G_i          = sum_{m<=i} log alpha_m           (in-chunk prefix of log-gates)
  D_{j+1:i}    = Diag(exp(G_i - G_j))             (difference of two prefix sums)
  ebar_i       = beta_i (v_i - M_c D_{0:i} k_i)   (provisional error, all i at once)
  rho_ij       = beta_i k_j^T D_{j+1:i} k_i, j<i  (strictly lower R)
  e_i          = ebar_i - sum_{j<i} rho_ij e_j    (unit-lower triangular solve)
  M_{c+1}      = M_c D_{0:L-1} + E K_end           (K_end rows: k_j^T D_{j+1:L-1})
  chi_ij       = k_j^T D_{j+1:i} q_i, j<=i         (lower A_qk, diagonal included)
  O_c          = M_c Q_boundary + E A_qk^T         (Q_boundary columns: D_{0:i} q_i)
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _chain(q, k, v, alpha, eta, eps, S0, chunk):
    """One (b, h) chain. q,k: [T,dk]; v: [T,dv]; alpha: [T] or [T,dk]; eta: [T]; S0: [dk,dv]."""
    T, dk = k.shape
    dv = v.shape[1]
    M = np.zeros((dv, dk)) if S0 is None else S0.T.copy()       # page orientation: d_v x d_k
    o = np.zeros((T, dv))
    if alpha.ndim == 1:
        alpha = np.repeat(alpha[:, None], dk, axis=1)            # scalar gate = same value on every key channel
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        L = c1 - c0
        Kc, Qc, Vc = k[c0:c1], q[c0:c1], v[c0:c1]                # rows are tokens
        G = np.cumsum(np.log(alpha[c0:c1]), axis=0)              # [L, dk], inclusive prefix
        n2 = np.sum(Kc * Kc, axis=1)
        den = n2 + eps
        beta = np.where(den == 0.0, 0.0, eta[c0:c1] / np.where(den == 0.0, 1.0, den))

        # provisional errors, all tokens in parallel: columns of Ebar (d_v x L)
        Kb = (np.exp(G) * Kc).T                                  # columns D_{0:i} k_i
        Ebar = (Vc.T - M @ Kb) * beta[None, :]

        # rho_ij = beta_i k_j^T D_{j+1:i} k_i for j < i
        R = np.zeros((L, L))
        for i in range(L):
            for j in range(i):
                R[i, j] = beta[i] * np.sum(Kc[j] * np.exp(G[i] - G[j]) * Kc[i])
        # e_i = ebar_i - sum_{j<i} rho_ij e_j  <=>  (I + R) E^T = Ebar^T
        E = solve_triangular(np.eye(L) + R, Ebar.T, lower=True, unit_diagonal=True).T   # d_v x L

        # in-chunk outputs: O = M Q_boundary + E A_qk^T
        Aqk = np.zeros((L, L))
        for i in range(L):
            for j in range(i + 1):
                Aqk[i, j] = np.sum(Kc[j] * np.exp(G[i] - G[j]) * Qc[i])
        Qb = (np.exp(G) * Qc).T
        o[c0:c1] = (M @ Qb + E @ Aqk.T).T

        # end-of-chunk state: M D_{0:L-1} + E K_end
        Kend = np.exp(G[L - 1][None, :] - G) * Kc                # rows k_j^T D_{j+1:L-1}
        M = M * np.exp(G[L - 1])[None, :] + E @ Kend
    return o, M.T


def chunkwise(q, k, v, alpha, eta, eps, S0=None, chunk: int = 16):
    """Chunkwise fp64 evaluation with the same layouts and results as ``recurrent``.

    q, k: [B,T,H,d_k]; v: [B,T,H,d_v]; alpha: [B,T,H] or [B,T,H,d_k]; eta: [B,T,H];
    S0: [B,H,d_k,d_v] or None. Returns (o [B,T,H,d_v], S_T [B,H,d_k,d_v]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    alpha = np.asarray(alpha, dtype=np.float64)
    eta = np.asarray(eta, dtype=np.float64)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            s0 = None if S0 is None else np.asarray(S0[b, h], dtype=np.float64)
            ob, sb = _chain(q[b, :, h], k[b, :, h], v[b, :, h], alpha[b, :, h], eta[b, :, h], eps, s0, chunk)
            o[b, :, h] = ob
            ST[b, h] = sb
    return o, ST
