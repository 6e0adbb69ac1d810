"""Chunked (block-matrix) form of KDA in float64 numpy (test infrastructure).

The yunthe.com "Kimi K3 open-source practice" page (FlashKDA paragraph) says the
fast KDA kernels split the linear attention into block-matrix operations.  This
module writes that form out for one (sequence, head), straight from the token
recurrence

    S' = Diag(alpha_t) S ;  u_t = beta_t (v_t - S'^T k_t) ;  S = S' + k_t u_t^T ;
    o_t = scale * S^T q_t

and is used only to check that chunking changes nothing (for every chunk size).

Derivation, for one chunk of n tokens r = 0..n-1 starting from state S0.
Let g_r = sum_{tau <= r} log alpha_tau (per channel) and G_r = exp(g_r).  Then

    S_r = Diag(G_r) S0 + sum_{s <= r} Diag(G_r / G_s) k_s u_s^T,
    u_r = beta_r (v_r - S0^T (G_r * k_r) - sum_{s < r} A'_rs u_s),
    A'_rs = sum_c k_rc k_sc exp(g_rc - g_sc).

With A_rs = beta_r A'_rs (s < r) the rows stack to (I + A) U = diag(beta) (V - (G*K) S0),
so U = Ut - W S0 with T = (I + A)^{-1}, W = T diag(beta) (G * K), Ut = T diag(beta) V.
The outputs are O = scale * ((G * Q) S0 + P U) with P_rs = sum_c q_rc k_sc
exp(g_rc - g_sc) for s <= r, and the state leaving the chunk is
S_n = Diag(G_{n-1}) S0 + (exp(g_{n-1} - g) * K)^T U.  Only relative exponents
g_r - g_s with s <= r are ever exponentiated, so nothing overflows.

Chunk boundaries sit at absolute positions that are multiples of the chunk
size, counted from ``start_pos``.
"""
import numpy as np
from scipy.linalg import solve_triangular


def _chunk(q, k, v, alpha, beta, S, scale):
    n = q.shape[0]
    g = np.cumsum(np.log(alpha), axis=0)                       # [n, d_k]
    lower_incl = np.tril(np.ones((n, n), dtype=bool))
    strict = np.tril(np.ones((n, n), dtype=bool), -1)
    diff = g[:, None, :] - g[None, :, :]                       # [r, s, c]
    diff = np.where(lower_incl[:, :, None], diff, -np.inf)
    D = np.exp(diff)                                           # exp(g_r - g_s), 0 above diagonal
    A = beta[:, None] * np.einsum("rc,sc,rsc->rs", k, k, D) * strict
    P = np.einsum("rc,sc,rsc->rs", q, k, D) * lower_incl
    G = np.exp(g)
    M = np.eye(n) + A
    W = solve_triangular(M, beta[:, None] * G * k, lower=True, unit_diagonal=True)
    Ut = solve_triangular(M, beta[:, None] * v, lower=True, unit_diagonal=True)
    U = Ut - W @ S
    O = scale * ((G * q) @ S + P @ U)
    gl = g[-1]
    Kbar = np.exp(gl[None, :] - g) * k
    S_new = np.exp(gl)[:, None] * S + Kbar.T @ U
    return O, S_new


def chunked(q, k, v, alpha, beta, chunk, S0=None, scale=1.0, start_pos=0,
            snap_interval=None):
    """Chunked float64 KDA for one sequence and one head.

    q, k [T, d_k]; v [T, d_v]; alpha [T, d_k]; beta [T]; float-convertible.
    Returns (O [T, d_v], S_final [d_k, d_v], snaps dict ordinal -> state).  Snapshots
    are taken at chunk ends whose absolute position is a multiple of
    ``snap_interval`` (which must then be a multiple of ``chunk``).
    """
    q, k, v, alpha, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, alpha, beta))
    T, d_k = q.shape
    d_v = v.shape[1]
    S = np.zeros((d_k, d_v)) if S0 is None else np.array(S0, dtype=np.float64)
    if snap_interval is not None and snap_interval % chunk != 0:
        raise ValueError("snapshot interval must be a multiple of the chunk size")
    O = np.zeros((T, d_v))
    snaps = {}
    a = 0
    while a < T:
        p = start_pos + a
        b = min(T, a + (chunk - p % chunk))
        O[a:b], S = _chunk(q[a:b], k[a:b], v[a:b], alpha[a:b], beta[a:b], S, scale)
        p_end = start_pos + b
        if snap_interval is not None and p_end % snap_interval == 0:
            snaps[p_end // snap_interval - 1] = S.copy()
        a = b
    return O, S, snaps
