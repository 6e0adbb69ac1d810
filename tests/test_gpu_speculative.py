"""Speculative decoding through the C ABI (kda_decode_verify / kda_decode_commit)
against the float64 oracle ("Kimi K3 Tech Intro", section 6: 7 draft tokens
plus the current one verified per step, the accepted prefix kept).

Inputs follow the decode workload: states N(0, 0.05^2), q and k L2-normalised,
gates from the decode recipe; T = 8 candidate tokens per sequence.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_kda_gb300 import inputs, KDA_DEV_BAD_ACCEPT, KDA_DEV_BAD_SLOT
from _helpers import BF16_OUT_TOL, FP32_TOL

pytestmark = pytest.mark.gpu


def frob_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _tokens(n, T, H, d, seed, step, dtype):
    z = inputs.gen_decode(n * T, H, d, d, seed, step, dtype=dtype)
    return {k: t.reshape((n, T) + tuple(t.shape[1:])) for k, t in z.items()}


def _verify(kda, dev, z, pool, slots):
    n, T, H, d = z["q"].shape
    zd = {k: t.to(dev) for k, t in z.items()}
    o = torch.empty((n, T, H, d), dtype=z["v"].dtype, device=dev)
    u = torch.empty((n, T, H, d), dtype=torch.float32, device=dev)
    kda.kda_decode_verify(zd["q"], zd["k"], zd["v"], zd["alpha"], zd["beta"], pool, slots, o, u)
    return zd, o, u


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_verify_and_commit_match_the_oracle(kda, cuda_device, dtype, d):
    dev = cuda_device
    n, T, H = 8, 8, 4
    S0 = inputs.gen_states(n, H, d, d, 31, std=0.05)
    pool = torch.zeros((n + 3, H, d, d), device=dev)
    slots = torch.tensor([3 + i for i in range(n)], dtype=torch.int32, device=dev)
    pool[3:] = S0.to(dev)
    before = pool.clone()
    z = _tokens(n, T, H, d, 32, 0, dtype)
    zd, o, u = _verify(kda, dev, z, pool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    assert torch.equal(pool, before)                            # verification writes no state
    o_ref, u_ref, states = oracle.verify_steps(S0.double().numpy(), z["q"], z["k"], z["v"], z["alpha"], z["beta"])
    tol_o = BF16_OUT_TOL if dtype == torch.bfloat16 else FP32_TOL
    for i in range(n):
        for h in range(H):
            assert frob_rel(o[i, :, h].float().cpu(), o_ref[i, :, h]) < tol_o, (i, h)
            assert frob_rel(u[i, :, h].cpu(), u_ref[i, :, h]) < FP32_TOL, (i, h)
    accept = torch.tensor([0, 8, 1, 5, 3, 8, 2, 7], dtype=torch.int32)
    kda.kda_decode_commit(zd["k"], zd["alpha"], u, accept.to(dev), pool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    S_ref = oracle.commit_steps(S0.double().numpy(), z["k"], z["alpha"], u_ref, accept.tolist())
    for i in range(n):
        if accept[i] == 0:
            assert torch.equal(pool[3 + i], before[3 + i])
        for h in range(H):
            assert frob_rel(pool[3 + i, h].cpu(), S_ref[i, h]) < FP32_TOL, (i, h)
    assert torch.equal(pool[:3], before[:3])                    # other slots untouched


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_verify_one_then_commit_one_is_the_decode_step(kda, cuda_device, dtype, d):
    """Same per-thread data and arithmetic order as kda_decode_step: bit for bit."""
    dev = cuda_device
    n, H = 16, 4
    S0 = inputs.gen_states(n, H, d, d, 41, std=0.05).to(dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    z = _tokens(n, 1, H, d, 42, 0, dtype)
    pool_a = S0.clone()
    zd, o, u = _verify(kda, dev, z, pool_a, slots)
    kda.kda_decode_commit(zd["k"], zd["alpha"], u, torch.ones(n, dtype=torch.int32, device=dev), pool_a, slots)
    pool_b = S0.clone()
    o_b = torch.empty((n, H, d), dtype=dtype, device=dev)
    kda.kda_decode_step(zd["q"][:, 0], zd["k"][:, 0], zd["v"][:, 0], zd["alpha"][:, 0], zd["beta"][:, 0],
                        pool_b, slots, o_b)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    assert torch.equal(o[:, 0], o_b)
    assert torch.equal(pool_a, pool_b)


def test_speculative_loop_keeps_only_accepted_tokens(kda, cuda_device):
    """12 steps of verify + commit with random acceptance; the final states and
    every accepted output equal the oracle run over the accepted tokens only."""
    dev = cuda_device
    n, T, H, d = 6, 8, 4, 128
    rng = np.random.default_rng(5)
    S0 = inputs.gen_states(n, H, d, d, 51, std=0.05)
    pool = S0.to(dev).clone()
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    kept = {key: [[] for _ in range(n)] for key in ("q", "k", "v", "alpha", "beta")}
    outs = [[] for _ in range(n)]
    for step in range(12):
        z = _tokens(n, T, H, d, 52, step, torch.bfloat16)
        zd, o, u = _verify(kda, dev, z, pool, slots)
        acc = rng.integers(0, T + 1, size=n).astype(np.int32)
        kda.kda_decode_commit(zd["k"], zd["alpha"], u, torch.from_numpy(acc).to(dev), pool, slots)
        torch.cuda.synchronize()
        assert kda.kda_check_status() == 0
        for i in range(n):
            for key in kept:
                kept[key][i].append(z[key][i, :acc[i]])
            outs[i].append(o[i, :acc[i]].float().cpu())
    cat = {key: [torch.cat(kept[key][i]) for i in range(n)] for key in kept}
    lens = [len(c) for c in cat["q"]]
    packed = {key: torch.cat(cat[key]) for key in cat}
    cu = np.concatenate([[0], np.cumsum(lens)])
    ref = oracle.run(packed["q"], packed["k"], packed["v"], packed["alpha"], packed["beta"], cu,
                     init_state=S0.double().numpy())
    got_o = torch.cat([torch.cat(outs[i]) for i in range(n)])
    for i in range(n):
        for h in range(H):
            assert frob_rel(pool[i, h].cpu(), ref["final"][i, h]) < FP32_TOL, (i, h)
            if lens[i]:
                assert frob_rel(got_o[cu[i]:cu[i + 1], h], ref["o"][cu[i]:cu[i + 1], h]) < BF16_OUT_TOL, (i, h)


@pytest.mark.parametrize("T", [3, 16])
def test_verify_and_commit_at_other_candidate_counts(kda, cuda_device, T):
    """An odd candidate count and the largest one the call takes (16)."""
    dev = cuda_device
    n, H, d = 4, 2, 128
    S0 = inputs.gen_states(n, H, d, d, 71 + T, std=0.05)
    pool = S0.to(dev).clone()
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    z = _tokens(n, T, H, d, 72 + T, 0, torch.bfloat16)
    zd, o, u = _verify(kda, dev, z, pool, slots)
    accept = torch.tensor([T, 0, 1, T - 1], dtype=torch.int32)
    kda.kda_decode_commit(zd["k"], zd["alpha"], u, accept.to(dev), pool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    o_ref, u_ref, _ = oracle.verify_steps(S0.double().numpy(), z["q"], z["k"], z["v"], z["alpha"], z["beta"])
    S_ref = oracle.commit_steps(S0.double().numpy(), z["k"], z["alpha"], u_ref, accept.tolist())
    for i in range(n):
        for h in range(H):
            assert frob_rel(o[i, :, h].float().cpu(), o_ref[i, :, h]) < BF16_OUT_TOL, (i, h)
            assert frob_rel(u[i, :, h].cpu(), u_ref[i, :, h]) < FP32_TOL, (i, h)
            assert frob_rel(pool[i, h].cpu(), S_ref[i, h]) < FP32_TOL, (i, h)
    assert torch.equal(pool[1], S0[1].to(dev))                 # none accepted: untouched


def test_bad_accept_and_slot_are_flagged(kda, cuda_device):
    dev = cuda_device
    n, T, H, d = 4, 4, 2, 64
    pool = inputs.gen_states(n, H, d, d, 61).to(dev)
    before = pool.clone()
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    z = _tokens(n, T, H, d, 62, 0, torch.float32)
    zd, o, u = _verify(kda, dev, z, pool, slots)
    kda.kda_decode_commit(zd["k"], zd["alpha"], u, torch.tensor([1, 5, -1, 0], dtype=torch.int32, device=dev),
                          pool, slots)
    torch.cuda.synchronize()
    bits = kda.kda_check_status()
    assert bits == KDA_DEV_BAD_ACCEPT
    assert torch.equal(pool[1:], before[1:])                   # bad counts (and 0) skip the sequence
    assert not torch.equal(pool[0], before[0])
    bad_slots = torch.tensor([0, 1, 2, n + 7], dtype=torch.int32, device=dev)
    _verify(kda, dev, z, pool, bad_slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == KDA_DEV_BAD_SLOT


def test_full_decode_batch_sampled(kda, cuda_device):
    """512 sequences x 32 heads x 8 candidates (1 GiB of states): the verified
    outputs and committed states of sampled (sequence, head) pairs."""
    dev = cuda_device
    w = inputs.WORKLOADS["decode_512x32"]
    n, H, d, T = w["n_seqs"], w["H"], w["d"], 8
    S0 = inputs.gen_states(n, H, d, d, w["seed"], std=w["state_std"])
    pool = S0.to(dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    z = _tokens(n, T, H, d, w["seed"], 100, torch.bfloat16)
    zd, o, u = _verify(kda, dev, z, pool, slots)
    acc = torch.from_numpy(np.random.default_rng(7).integers(0, T + 1, size=n).astype(np.int32))
    kda.kda_decode_commit(zd["k"], zd["alpha"], u, acc.to(dev), pool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    rng = np.random.default_rng(8)
    seqs = rng.choice(n, size=6, replace=False)
    heads = rng.choice(H, size=6)
    S_s = S0[seqs].double().numpy()
    o_ref, u_ref, _ = oracle.verify_steps(S_s, *(z[key][seqs] for key in ("q", "k", "v", "alpha", "beta")))
    S_ref = oracle.commit_steps(S_s, z["k"][seqs], z["alpha"][seqs], u_ref, acc[seqs].tolist())
    for r, (i, h) in enumerate(zip(seqs, heads)):
        assert frob_rel(o[i, :, h].float().cpu(), o_ref[r, :, h]) < BF16_OUT_TOL
        assert frob_rel(u[i, :, h].cpu(), u_ref[r, :, h]) < FP32_TOL
        assert frob_rel(pool[i, h].cpu(), S_ref[r, h]) < FP32_TOL
