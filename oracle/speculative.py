"""Multi-token verification and commit of a speculative decoding step
(test infrastructure).

"Kimi K3 Tech Intro", section 6: a draft model proposes 7 tokens.  The target
model verifies them in one step, accepts a prefix, and falls back on the rest.
A recurrent KDA state cannot be rolled back, so a verification step must leave
the state untouched.  It reports for every candidate token t:
  * its output o_t;
  * its update vector u_t = beta_t (v_t - (Diag(alpha_t) S_{t-1})^T k_t).
Once the number of accepted tokens is known, a commit applies
S_t = Diag(alpha_t) S_{t-1} + k_t u_t^T for those tokens only.

This is the recurrence of ``oracle.run`` written out token by token in float64
numpy, for the small batches a decoding step has.  It returns what ``run`` does
not: every u_t and every intermediate state.
"""
import numpy as np


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def verify_steps(S0, q, k, v, alpha, beta, scale=1.0):
    """Run T candidate tokens from the states S0 without committing them.

    S0: [n, H, d_k, d_v]; q, k, alpha: [n, T, H, d_k]; v: [n, T, H, d_v];
    beta: [n, T, H].  Returns (o [n, T, H, d_v], u [n, T, H, d_v],
    states [n, T, H, d_k, d_v]), where states[:, t] is the state after token t.
    """
    S = _f64(S0).copy()
    q, k, v, alpha, beta = (_f64(x) for x in (q, k, v, alpha, beta))
    n, T, H, dk = q.shape
    dv = v.shape[3]
    o = np.zeros((n, T, H, dv))
    u = np.zeros((n, T, H, dv))
    states = np.zeros((n, T, H, dk, dv))
    for t in range(T):
        Sp = alpha[:, t, :, :, None] * S                               # Diag(alpha) S
        pred = np.einsum("nhi,nhij->nhj", k[:, t], Sp)                 # S'^T k
        u[:, t] = beta[:, t, :, None] * (v[:, t] - pred)
        S = Sp + k[:, t, :, :, None] * u[:, t, :, None, :]             # S' + k u^T
        o[:, t] = scale * np.einsum("nhi,nhij->nhj", q[:, t], S)      # S_t^T q_t
        states[:, t] = S
    return o, u, states


def commit_steps(S0, k, alpha, u, n_accept):
    """Apply the first n_accept[i] updates of sequence i to its state:
    S <- Diag(alpha_t) S + k_t u_t^T for t < n_accept[i].  Returns the states."""
    S = _f64(S0).copy()
    k, alpha, u = _f64(k), _f64(alpha), _f64(u)
    for i, m in enumerate(n_accept):
        for t in range(int(m)):
            S[i] = alpha[i, t, :, :, None] * S[i] + k[i, t, :, :, None] * u[i, t, :, None, :]
    return S
