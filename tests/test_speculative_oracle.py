"""Pins of the speculative-decoding oracle (verify without committing, then
commit the accepted tokens) against the C token recurrence, which the other
oracle pins fix.

* The outputs and the state after every candidate token equal those of the C
  recurrence run on the same tokens from the same states.
* Each update vector u_t is recovered from the C recurrence's consecutive states
  alone: k_t u_t^T = S_t - Diag(alpha_t) S_{t-1}, so
  u_t = (S_t - Diag(alpha_t) S_{t-1})^T k_t / (k_t . k_t).
* Committing m tokens gives the state after token m; committing none leaves the
  state as it was.
"""
import numpy as np
import pytest

import oracle


def _case(n=3, T=8, H=2, d=16, seed=0, decay_shift=-1.0):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit(rng.standard_normal((n, T, H, d)))
    k = unit(rng.standard_normal((n, T, H, d)))
    v = rng.standard_normal((n, T, H, d))
    alpha = np.exp(-np.log1p(np.exp(rng.standard_normal((n, T, H, d)) + decay_shift)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((n, T, H))))
    S0 = 0.05 * rng.standard_normal((n, H, d, d))
    return S0, q, k, v, alpha, beta


def _c_run(S0, q, k, v, alpha, beta, tokens):
    """The C recurrence on the first `tokens` tokens of every sequence."""
    n, T, H, d = q.shape
    pack = lambda x: np.ascontiguousarray(x[:, :tokens].reshape((n * tokens,) + x.shape[2:]))
    cu = np.arange(n + 1) * tokens
    return oracle.run(pack(q), pack(k), pack(v), pack(alpha), pack(beta), cu, init_state=S0)


def test_verify_matches_the_c_recurrence():
    S0, q, k, v, alpha, beta = _case()
    o, u, states = oracle.verify_steps(S0, q, k, v, alpha, beta)
    n, T = q.shape[:2]
    ref = _c_run(S0, q, k, v, alpha, beta, T)
    np.testing.assert_allclose(o.reshape(ref["o"].shape), ref["o"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(states[:, -1], ref["final"], rtol=1e-12, atol=1e-14)
    for t in range(1, T):
        np.testing.assert_allclose(states[:, t - 1], _c_run(S0, q, k, v, alpha, beta, t)["final"],
                                   rtol=1e-12, atol=1e-14)


def test_update_vectors_follow_from_consecutive_states():
    S0, q, k, v, alpha, beta = _case(seed=1)
    _, u, _ = oracle.verify_steps(S0, q, k, v, alpha, beta)
    n, T = q.shape[:2]
    prev = S0
    for t in range(T):
        cur = _c_run(S0, q, k, v, alpha, beta, t + 1)["final"]
        rank1 = cur - alpha[:, t, :, :, None] * prev                    # k_t u_t^T
        kt = k[:, t]
        u_rec = np.einsum("nhi,nhij->nhj", kt, rank1) / np.einsum("nhi,nhi->nh", kt, kt)[..., None]
        np.testing.assert_allclose(u[:, t], u_rec, rtol=1e-9, atol=1e-12)
        # and the update really is rank one along k_t
        np.testing.assert_allclose(rank1, kt[..., :, None] * u_rec[..., None, :], rtol=1e-9, atol=1e-12)
        prev = cur


@pytest.mark.parametrize("accept", [[0, 0, 0], [8, 8, 8], [1, 5, 8], [0, 3, 7]])
def test_commit_gives_the_state_after_the_accepted_tokens(accept):
    S0, q, k, v, alpha, beta = _case(seed=2)
    _, u, states = oracle.verify_steps(S0, q, k, v, alpha, beta)
    S = oracle.commit_steps(S0, k, alpha, u, accept)
    for i, m in enumerate(accept):
        expect = S0[i] if m == 0 else states[i, m - 1]
        np.testing.assert_allclose(S[i], expect, rtol=1e-12, atol=1e-15)
        if m:
            c = _c_run(S0[i:i + 1], q[i:i + 1], k[i:i + 1], v[i:i + 1], alpha[i:i + 1], beta[i:i + 1], m)
            np.testing.assert_allclose(S[i], c["final"][0], rtol=1e-12, atol=1e-14)


def test_zero_beta_writes_nothing():
    S0, q, k, v, alpha, beta = _case(seed=3)
    beta[:] = 0.0
    o, u, states = oracle.verify_steps(S0, q, k, v, alpha, beta)
    assert np.all(u == 0.0)
    decay = np.cumprod(alpha, axis=1)
    np.testing.assert_allclose(states[:, -1], decay[:, -1, :, :, None] * S0, rtol=1e-12)
