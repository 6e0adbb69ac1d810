"""Pins of the fused decode step oracle ("Kimi K3 Tech Intro", section 4.1).

The recurrent core is checked against the C token recurrence, which the other
pins fix.  The prologue and epilogue are checked against properties that fix
them independently of their formulas:
* a single-tap convolution delays its input by a fixed number of tokens;
* the convolution state holds exactly the last K-1 raw inputs;
* exp(-softplus(a)) = 1 / (1 + e^a);
* normalised q and k have unit length;
* the gated RMSNorm ignores the scale of o, has RMS |gamma| when the gate is
  fully open, and halves at g = 0.
"""
import numpy as np
import pytest

import oracle
from oracle import fused_decode as fd


def _inputs(n=2, H=3, d=16, seed=0):
    rng = np.random.default_rng(seed)
    return dict(xq=rng.standard_normal((n, H, d)), xk=rng.standard_normal((n, H, d)),
                xv=rng.standard_normal((n, H, d)), a=rng.standard_normal((n, H, d)) + 2.0,
                b=rng.standard_normal((n, H)), g=rng.standard_normal((n, H, d)))


def test_single_tap_convolution_delays_its_input():
    rng = np.random.default_rng(1)
    n, H, d, K = 1, 2, 8, fd.K_CONV
    for tau in range(K):
        w = np.zeros((K, d))
        w[tau] = 1.0
        C = np.zeros((n, H, K - 1, d))
        xs = [rng.standard_normal((n, H, d)) for _ in range(7)]
        for t, x in enumerate(xs):
            y, C = fd.causal_conv(C, x, w)
            lag = K - 1 - tau
            expect = fd.silu(xs[t - lag]) if t - lag >= 0 else fd.silu(np.zeros_like(x))
            np.testing.assert_allclose(y, expect, rtol=1e-15)
        np.testing.assert_array_equal(C, np.stack(xs[-(K - 1):], axis=2))


def test_gate_identities():
    a = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(np.exp(-fd.softplus(a)), 1.0 / (1.0 + np.exp(a)), rtol=1e-12)
    assert fd.sigmoid(0.0) == 0.5


def test_qk_norm_is_unit_length():
    x = np.random.default_rng(2).standard_normal((5, 64)) * 3.0
    np.testing.assert_allclose(np.linalg.norm(fd.l2norm(x), axis=-1), 1.0, rtol=1e-6)


def test_gated_rmsnorm_properties():
    rng = np.random.default_rng(3)
    o, gamma = rng.standard_normal((4, 32)), rng.standard_normal(32)
    big = np.full((4, 32), 50.0)
    y = fd.gated_rmsnorm(o, big, gamma, 0.0)
    np.testing.assert_allclose(fd.gated_rmsnorm(7.5 * o, big, gamma, 0.0), y, rtol=1e-12)
    np.testing.assert_allclose(np.sqrt(np.mean((y / gamma) ** 2, axis=-1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(fd.gated_rmsnorm(o, np.zeros_like(o), gamma, 0.0), 0.5 * y, rtol=1e-12)


def test_recurrent_core_matches_the_c_recurrence():
    """Identity-like prologue/epilogue pieces are applied by hand; the state and
    the pre-norm output must be those of oracle.run on the transformed inputs."""
    n, H, d, K = 2, 3, 16, fd.K_CONV
    rng = np.random.default_rng(4)
    x = _inputs(n, H, d, seed=5)
    S0 = 0.05 * rng.standard_normal((n, H, d, d))
    C0 = rng.standard_normal((n, H, 3, K - 1, d))
    conv_w = rng.standard_normal((H, 3, K, d)) * 0.5
    norm_w = rng.standard_normal((H, d))
    y, S1, C1 = fd.fused_step(S0, C0, x["xq"], x["xk"], x["xv"], x["a"], x["b"], x["g"], conv_w, norm_w)
    # the same step with the inputs transformed separately
    def conv(i, xi):
        win = np.concatenate([C0[:, :, i], xi[:, :, None, :]], axis=2)
        return fd.silu(np.einsum("nhkd,hkd->nhd", win, conv_w[:, i]))
    q = fd.l2norm(conv(0, x["xq"]))
    k = fd.l2norm(conv(1, x["xk"]))
    v = conv(2, x["xv"])
    alpha = 1.0 / (1.0 + np.exp(x["a"]))
    beta = fd.sigmoid(x["b"])
    ref = oracle.run(q.reshape(n, H, d), k, v, alpha, beta, np.arange(n + 1), init_state=S0)
    np.testing.assert_allclose(S1, ref["final"], rtol=1e-11, atol=1e-14)
    o = ref["o"]
    expect_y = norm_w[None] * o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + 1e-6) * fd.sigmoid(x["g"])
    np.testing.assert_allclose(y, expect_y, rtol=1e-10, atol=1e-13)
    np.testing.assert_array_equal(C1[:, :, 0, -1], x["xq"])
    np.testing.assert_array_equal(C1[:, :, 2, :-1], C0[:, :, 2, 1:])
