"""Forgetting bounds for checking long sequences on windows (test infrastructure).

One token maps the state by S -> M_t S + beta_t k_t v_t^T with
M_t = (I - beta_t k_t k_t^T) Diag(alpha_t).  For 0 <= beta_t |k_t|^2 <= 2 the factor
I - beta_t k_t k_t^T has eigenvalues 1 and 1 - beta_t |k_t|^2, so its spectral
norm is at most 1, and |M_t|_2 <= max_c alpha_tc.  Two runs over the same tokens
that start from states differing by D therefore differ after tokens a..b-1 by at
most prod_{t=a}^{b-1} max_c alpha_tc * |D|_F in Frobenius norm, and their
outputs o_t = scale * S_t^T q_t by that times |scale| |q_t|.

``state_norm_bound`` bounds |S_t|_F for the run from a zero state by the same
argument: |S_t|_F <= max_c alpha_tc |S_{t-1}|_F + beta_t |k_t| |v_t|.
"""
import numpy as np


def window_bound(alpha_window) -> float:
    """prod over tokens of max over channels of alpha ([W, d_k] array)."""
    a = np.asarray(alpha_window, dtype=np.float64)
    if a.shape[0] == 0:
        return 1.0
    return float(np.exp(np.sum(np.log(a.max(axis=1)))))


def state_norm_bound(alpha, beta, k, v, S0_norm: float = 0.0) -> float:
    """Upper bound on |S_T|_F after tokens alpha [T,d_k], beta [T], k [T,d_k],
    v [T,d_v], starting from a state of norm S0_norm."""
    a = np.asarray(alpha, dtype=np.float64).max(axis=1)
    b = np.asarray(beta, dtype=np.float64)
    kn = np.linalg.norm(np.asarray(k, dtype=np.float64), axis=1)
    vn = np.linalg.norm(np.asarray(v, dtype=np.float64), axis=1)
    if np.any(b * kn * kn > 2.0):
        raise ValueError("bound needs beta |k|^2 <= 2")
    bound = float(S0_norm)
    for t in range(a.shape[0]):
        bound = a[t] * bound + b[t] * kn[t] * vn[t]
    return bound
