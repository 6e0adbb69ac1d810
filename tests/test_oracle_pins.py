"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test fixes the oracle to something independent of its own code: an
invariant of the gated delta rule, a closed form, a hand calculation, exact
rational arithmetic of the matrix form of the update, or the worked
prefix-match example printed in "Kimi K3 Tech Intro" section 2.1.  Each is chosen
so that a plausible slip in the oracle (a dropped beta, a sign, the decay on the
wrong index or after the update, S_{t-1} instead of S_t in the output, a
transposed product, an off-by-one snapshot) fails at least one of them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, T, d_k, d_v, decay="config", H=1):
    q = rng.standard_normal((T, H, d_k))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((T, H, d_k))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d_v))
    shift = {"config": 2.0, "mild": -5.0}[decay]
    x = rng.standard_normal((T, H, d_k)) + shift
    alpha = np.exp(-np.logaddexp(0.0, x))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, alpha, beta


def _one(q, k, v, alpha, beta, S0=None, **kw):
    T = q.shape[0]
    init = None if S0 is None else np.asarray(S0, np.float64)[None, None]
    return oracle.run(q, k, v, alpha, beta, [0, T], init_state=init, **kw)


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ---------------------------------------------------------------- invariants

def test_beta0_alpha1_leaves_state_unchanged():
    """beta = 0 with alpha = 1: S_t = S_0 and o_t = S_0^T q_t (d_k != d_v)."""
    rng = np.random.default_rng(1)
    T, d_k, d_v = 9, 3, 5
    q, k, v, _, _ = _rand_inputs(rng, T, d_k, d_v)
    alpha = np.ones((T, 1, d_k))
    beta = np.zeros((T, 1))
    S0 = rng.standard_normal((d_k, d_v))
    r = _one(q, k, v, alpha, beta, S0)
    assert np.array_equal(r["final"][0, 0], S0)
    np.testing.assert_allclose(r["o"][:, 0], q[:, 0] @ S0, rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("S0_kind", ["zero", "random"])
def test_orthonormal_keys_retrieve_values(S0_kind):
    """alpha = 1, beta = 1, orthonormal keys: S_T^T k_j = v_j for every j."""
    rng = np.random.default_rng(2)
    d_k, d_v = 16, 7
    T = d_k
    basis, _ = np.linalg.qr(rng.standard_normal((d_k, d_k)))
    k = basis.T[:, None, :]                       # rows are orthonormal keys
    q = rng.standard_normal((T, 1, d_k))
    v = rng.standard_normal((T, 1, d_v))
    alpha = np.ones((T, 1, d_k))
    beta = np.ones((T, 1))
    S0 = None if S0_kind == "zero" else rng.standard_normal((d_k, d_v))
    r = _one(q, k, v, alpha, beta, S0)
    S = r["final"][0, 0]
    np.testing.assert_allclose(k[:, 0] @ S, v[:, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("decay", ["config", "mild"])
@pytest.mark.parametrize("T", [300, 257])
def test_chunked_matches_recurrent_every_chunk_size(decay, T):
    rng = np.random.default_rng(3 + T)
    d_k, d_v = 8, 6
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, decay)
    S0 = rng.standard_normal((d_k, d_v))
    ref = _one(q, k, v, alpha, beta, S0)
    for C in [1, 2, 3, 4, 7, 8, 16, 32, 64, 128, T]:
        O, S, _ = oracle.chunked(q[:, 0], k[:, 0], v[:, 0], alpha[:, 0], beta[:, 0], C, S0=S0)
        assert _rel(O, ref["o"][:, 0]) < 1e-10, C
        assert _rel(S, ref["final"][0, 0]) < 1e-10, C


def test_resume_reproduces_full_run_bit_for_bit():
    rng = np.random.default_rng(4)
    T, d_k, d_v = 700, 8, 8
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild")
    full = oracle.run(q, k, v, alpha, beta, [0, T], snap_req=[(0, 0), (0, 1)])
    for ordinal in (0, 1):
        p = 256 * (ordinal + 1)
        snap = full["snaps"][ordinal][None]
        res = oracle.run(q[p:], k[p:], v[p:], alpha[p:], beta[p:], [0, T - p],
                         start_pos=[p], init_state=snap, snap_req=[(0, 1)])
        assert np.array_equal(res["o"], full["o"][p:])
        assert np.array_equal(res["final"], full["final"])
        if ordinal == 0:
            assert np.array_equal(res["snaps"][0], full["snaps"][1])


def test_chunked_resume_bit_for_bit():
    rng = np.random.default_rng(5)
    T, d_k, d_v = 600, 6, 5
    q, k, v, alpha, beta = (x[:, 0] for x in _rand_inputs(rng, T, d_k, d_v, "mild"))
    O, S, snaps = oracle.chunked(q, k, v, alpha, beta, 64, snap_interval=256)
    p = 256
    O2, S2, snaps2 = oracle.chunked(q[p:], k[p:], v[p:], alpha[p:], beta[p:], 64,
                                    S0=snaps[0], start_pos=p, snap_interval=256)
    assert np.array_equal(O2, O[p:])
    assert np.array_equal(S2, S)
    assert np.array_equal(snaps2[1], snaps[1])


# ---------------------------------------------------------------- closed forms

def test_beta0_is_pure_decay():
    """beta = 0: S_t = Diag(prod_{tau<=t} alpha_tau) S_0 (decay on the d_k rows)."""
    rng = np.random.default_rng(6)
    T, d_k, d_v = 11, 4, 6
    q, k, v, alpha, _ = _rand_inputs(rng, T, d_k, d_v, "mild")
    beta = np.zeros((T, 1))
    S0 = rng.standard_normal((d_k, d_v))
    r = _one(q, k, v, alpha, beta, S0)
    cum = np.cumprod(alpha[:, 0], axis=0)              # [T, d_k]
    np.testing.assert_allclose(r["final"][0, 0], cum[-1][:, None] * S0, rtol=1e-13)
    expect_o = np.stack([(cum[t][:, None] * S0).T @ q[t, 0] for t in range(T)])
    np.testing.assert_allclose(r["o"][:, 0], expect_o, rtol=1e-12, atol=1e-15)


def test_alpha0_keeps_only_the_current_token():
    """alpha = 0: S_t = beta_t k_t v_t^T and o_t = beta_t (k_t . q_t) v_t."""
    rng = np.random.default_rng(7)
    T, d_k, d_v = 6, 5, 3
    q, k, v, _, beta = _rand_inputs(rng, T, d_k, d_v)
    alpha = np.zeros((T, 1, d_k))
    S0 = rng.standard_normal((d_k, d_v))
    r = _one(q, k, v, alpha, beta, S0)
    t = T - 1
    np.testing.assert_allclose(r["final"][0, 0], beta[t, 0] * np.outer(k[t, 0], v[t, 0]),
                               rtol=1e-14, atol=1e-16)
    expect_o = beta[:, 0:1] * np.sum(k[:, 0] * q[:, 0], axis=1, keepdims=True) * v[:, 0]
    np.testing.assert_allclose(r["o"][:, 0], expect_o, rtol=1e-13, atol=1e-16)


def test_scalar_recurrence_closed_form():
    """d_k = d_v = 1, k_t = +-1: S_T = S_0 prod (1-b)a + sum_t b_t k_t v_t prod_{tau>t} (1-b)a."""
    rng = np.random.default_rng(8)
    T = 40
    k = rng.choice([-1.0, 1.0], size=(T, 1, 1))
    q = rng.standard_normal((T, 1, 1))
    v = rng.standard_normal((T, 1, 1))
    a = rng.uniform(0.5, 1.0, size=T)
    b = rng.uniform(0.0, 1.0, size=T)
    S0 = 0.75
    r = _one(q, k, v, a.reshape(T, 1, 1), b.reshape(T, 1), np.array([[S0]]))
    f = (1.0 - b) * a
    expect = S0 * np.prod(f) + sum(b[t] * k[t, 0, 0] * v[t, 0, 0] * np.prod(f[t + 1:])
                                   for t in range(T))
    assert abs(r["final"][0, 0, 0, 0] - expect) <= 1e-13 * max(1.0, abs(expect))
    # every output o_t = q_t S_t, with S_t the same closed form truncated at t
    for t in (0, 17, T - 1):
        St = S0 * np.prod(f[:t + 1]) + sum(b[s] * k[s, 0, 0] * v[s, 0, 0] * np.prod(f[s + 1:t + 1])
                                           for s in range(t + 1))
        assert abs(r["o"][t, 0, 0] - q[t, 0, 0] * St) <= 1e-13 * max(1.0, abs(St))


def test_single_token_by_hand():
    """T = 1, d_k = d_v = 2, worked by hand.

    S0 = [[1, 2], [3, 4]], alpha = (1/2, 1/4), beta = 1/2, k = (0.6, 0.8), v = (1, -1),
    q = (1, 0):
      S' = Diag(alpha) S0        = [[0.5, 1], [0.75, 1]]
      S'^T k                     = [0.5*0.6 + 0.75*0.8, 1*0.6 + 1*0.8] = [0.9, 1.4]
      u = beta (v - S'^T k)      = 0.5 * [0.1, -2.4] = [0.05, -1.2]
      S1 = S' + k u^T            = [[0.53, 0.28], [0.79, 0.04]]
      o1 = S1^T q                = [0.53, 0.28]
    """
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[0.6, 0.8]]])
    v = np.array([[[1.0, -1.0]]])
    alpha = np.array([[[0.5, 0.25]]])
    beta = np.array([[0.5]])
    S0 = np.array([[1.0, 2.0], [3.0, 4.0]])
    r = _one(q, k, v, alpha, beta, S0)
    np.testing.assert_allclose(r["final"][0, 0], [[0.53, 0.28], [0.79, 0.04]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["o"][0, 0], [0.53, 0.28], rtol=0, atol=1e-15)


def test_matrix_form_in_exact_arithmetic():
    """The update as one matrix product, S_t = (I - b k k^T) Diag(a) S + b k v^T,
    evaluated in exact rationals, against the oracle's split form.  Inputs are
    dyadic so the oracle reads them exactly."""
    rng = np.random.default_rng(9)
    T, d_k, d_v = 4, 2, 3

    def dyadic(shape, lo, hi):
        return rng.integers(lo, hi, size=shape) / 16.0

    q = dyadic((T, 1, d_k), -16, 17)
    k = dyadic((T, 1, d_k), -16, 17)
    v = dyadic((T, 1, d_v), -32, 33)
    alpha = dyadic((T, 1, d_k), 1, 16)
    beta = dyadic((T, 1), 1, 16)
    S0 = dyadic((d_k, d_v), -16, 17)
    r = _one(q, k, v, alpha, beta, S0)

    F = Fraction
    S = [[F(S0[i, j]) for j in range(d_v)] for i in range(d_k)]
    for t in range(T):
        kk = [F(x) for x in k[t, 0]]
        b = F(beta[t, 0])
        M = [[(1 if i == j else 0) - b * kk[i] * kk[j] for j in range(d_k)] for i in range(d_k)]
        DS = [[F(alpha[t, 0, i]) * S[i][j] for j in range(d_v)] for i in range(d_k)]
        S = [[sum(M[i][m] * DS[m][j] for m in range(d_k)) + b * kk[i] * F(v[t, 0, j])
              for j in range(d_v)] for i in range(d_k)]
        o = [sum(S[i][j] * F(q[t, 0, i]) for i in range(d_k)) for j in range(d_v)]
        np.testing.assert_allclose(r["o"][t, 0], [float(x) for x in o], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(r["final"][0, 0], [[float(x) for x in row] for row in S],
                               rtol=1e-14, atol=1e-14)


def test_linear_in_initial_state_and_values():
    """For fixed q, k, alpha, beta the map (S_0, V) -> (S_T, O) is linear."""
    rng = np.random.default_rng(10)
    T, d_k, d_v = 50, 6, 4
    q, k, v1, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild")
    v2 = rng.standard_normal(v1.shape)
    A0, B0 = rng.standard_normal((d_k, d_v)), rng.standard_normal((d_k, d_v))
    a, b = 0.7, -1.3
    r1 = _one(q, k, v1, alpha, beta, A0)
    r2 = _one(q, k, v2, alpha, beta, B0)
    r3 = _one(q, k, a * v1 + b * v2, alpha, beta, a * A0 + b * B0)
    np.testing.assert_allclose(r3["final"], a * r1["final"] + b * r2["final"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r3["o"], a * r1["o"] + b * r2["o"], rtol=1e-11, atol=1e-12)


def test_state_norm_obeys_contraction_bound():
    """|S_t|_F <= max_c alpha_tc |S_{t-1}|_F + beta_t |k_t| |v_t| at every token."""
    rng = np.random.default_rng(11)
    T, d_k, d_v = 64, 8, 8
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild")
    S0 = rng.standard_normal((d_k, d_v))
    r = _one(q, k, v, alpha, beta, S0, snap_interval=1, snap_req=[(0, t) for t in range(T)])
    prev = np.linalg.norm(S0)
    for t in range(T):
        cur = np.linalg.norm(r["snaps"][t, 0])
        bound = alpha[t, 0].max() * prev + beta[t, 0] * np.linalg.norm(k[t, 0]) * np.linalg.norm(v[t, 0])
        assert cur <= bound * (1 + 1e-12)
        prev = cur


# ---------------------------------------------------------------- snapshots

def test_snapshot_is_state_after_token_p_minus_1():
    """Snapshot ordinal m of a long run = final state of the run cut at p = 256 (m+1)."""
    rng = np.random.default_rng(12)
    T, d_k, d_v = 800, 4, 4
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild")
    full = oracle.run(q, k, v, alpha, beta, [0, T], snap_req=[(0, 0), (0, 1), (0, 2), (0, 3)])
    for m in range(3):
        p = 256 * (m + 1)
        cut = oracle.run(q[:p], k[:p], v[:p], alpha[:p], beta[:p], [0, p])
        assert np.array_equal(full["snaps"][m], cut["final"][0])
    assert np.isnan(full["snaps"][3]).all()           # p = 1024 > T: never reached
    assert oracle.snapshot_positions(0, T, 256) == [256, 512, 768]
    assert oracle.snapshot_positions(256, 300, 256) == [512]
    assert oracle.snapshot_positions(0, 512, 256) == [256, 512]


def test_prefix_match_worked_example():
    with open(os.path.join(GOLDEN, "prefix_match_example.json")) as f:
        g = json.load(f)
    block, unit = g["physical_block"], g["match_unit"]
    for shared, reused, recomputed in zip(g["shared_prefix_tokens"],
                                          g["reused_with_physical_block"],
                                          g["recomputed_with_physical_block"]):
        assert oracle.reusable_prefix(shared, block) == reused
        assert shared - oracle.reusable_prefix(shared, block) == recomputed
        # the finer match unit recomputes less than one unit
        assert 0 <= shared - oracle.reusable_prefix(shared, unit) < unit


def test_varlen_batch_equals_separate_runs():
    """Packing sequences with cu_seqlens changes nothing per sequence and head."""
    rng = np.random.default_rng(13)
    lens = [5, 0, 300, 1, 64]
    H, d_k, d_v = 2, 4, 3
    T = sum(lens)
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild", H=H)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    starts = [0, 256, 512, 0, 768]
    init = rng.standard_normal((len(lens), H, d_k, d_v))
    packed = oracle.run(q, k, v, alpha, beta, cu, start_pos=starts, init_state=init)
    for s, L in enumerate(lens):
        a, b = cu[s], cu[s + 1]
        one = oracle.run(q[a:b], k[a:b], v[a:b], alpha[a:b], beta[a:b], [0, L],
                         start_pos=[starts[s]], init_state=init[s:s + 1])
        assert np.array_equal(one["o"], packed["o"][a:b])
        assert np.array_equal(one["final"][0], packed["final"][s])
    assert np.array_equal(packed["final"][1], init[1])     # empty sequence keeps its state


def test_bf16_inputs_are_widened_exactly():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(14)
    T, H, d = 33, 2, 8
    q, k, v = (torch.randn((T, H, d), generator=g).to(torch.bfloat16) for _ in range(3))
    alpha = torch.rand((T, H, d), generator=g) * 0.5 + 0.4
    beta = torch.rand((T, H), generator=g)
    a = oracle.run(q, k, v, alpha, beta, [0, T])
    b = oracle.run(q.double(), k.double(), v.double(), alpha.double(), beta.double(), [0, T])
    assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["final"], b["final"])


def test_heads_are_independent_and_restrictable():
    rng = np.random.default_rng(15)
    T, H, d_k, d_v = 40, 3, 4, 4
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild", H=H)
    full = oracle.run(q, k, v, alpha, beta, [0, T])
    part = oracle.run(q, k, v, alpha, beta, [0, T], heads=(1, 2))
    assert np.array_equal(part["o"][:, 1], full["o"][:, 1])
    assert not part["o"][:, 0].any() and not part["o"][:, 2].any()


# ---------------------------------------------------------------- window bound

def test_window_bound_holds():
    """Two runs from different start states differ by at most the forgetting bound."""
    rng = np.random.default_rng(16)
    T, d_k, d_v = 120, 6, 5
    q, k, v, alpha, beta = _rand_inputs(rng, T, d_k, d_v, "mild")
    A0 = rng.standard_normal((d_k, d_v))
    B0 = rng.standard_normal((d_k, d_v))
    ra = _one(q, k, v, alpha, beta, A0, snap_interval=1, snap_req=[(0, t) for t in range(T)])
    rb = _one(q, k, v, alpha, beta, B0, snap_interval=1, snap_req=[(0, t) for t in range(T)])
    d0 = np.linalg.norm(A0 - B0)
    for t in (0, 10, 60, T - 1):
        bound = oracle.window_bound(alpha[:t + 1, 0]) * d0
        assert np.linalg.norm(ra["snaps"][t, 0] - rb["snaps"][t, 0]) <= bound * (1 + 1e-9)
    nb = oracle.state_norm_bound(alpha[:, 0], beta[:, 0], k[:, 0], v[:, 0], np.linalg.norm(A0))
    assert np.linalg.norm(ra["final"]) <= nb * (1 + 1e-12)
