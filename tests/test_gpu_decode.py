"""Batched single-token decode on the GPU against the float64 oracle.

The GPU state pool and the oracle's float64 states start from the same fp32
states and then evolve independently, step after step; outputs and states are
compared after every step, per (sequence, head).
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_kda_gb300 import inputs
from _helpers import BF16_OUT_TOL, BF16_STATE_TOL, FP32_TOL

pytestmark = pytest.mark.gpu


def _per_pair_rel(got, ref, dims):
    """Relative RMS of got vs ref per leading (seq, head) pair, on the device in float64."""
    diff = (got.double() - ref).pow(2).mean(dim=dims).sqrt()
    den = ref.pow(2).mean(dim=dims).sqrt()
    rel = torch.where(den > 0, diff / den.clamp_min(1e-300),
                      torch.where(diff > 0, torch.full_like(diff, float("inf")), diff))
    return rel


def _run_steps(kda, dev, n, H, d, dtype, steps, seed, std=0.05, n_slots=None, decay="config"):
    n_slots = n_slots or n + 3
    S0 = inputs.gen_states(n, H, d, d, seed, std=std)
    g = torch.Generator().manual_seed(seed)
    slots = torch.randperm(n_slots, generator=g)[:n].to(torch.int32)
    pool = torch.zeros((n_slots, H, d, d), dtype=torch.float32, device=dev)
    pool[slots.long().to(dev)] = S0.to(dev)
    slots_d = slots.to(dev)
    ref_state = S0.double().numpy()
    worst_o = worst_s = 0.0
    for step in range(steps):
        x = inputs.gen_decode(n, H, d, d, seed, step, dtype=dtype, decay=decay)
        xd = {key: t.to(dev) for key, t in x.items()}
        o = torch.empty((n, H, d), dtype=dtype, device=dev)
        kda.kda_decode_step(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], pool, slots_d, o)
        r = oracle.run(x["q"], x["k"], x["v"], x["alpha"], x["beta"], np.arange(n + 1),
                       init_state=ref_state)
        ref_state = r["final"]
        ref_o = torch.from_numpy(r["o"]).to(dev)
        ref_s = torch.from_numpy(ref_state).to(dev)
        worst_o = max(worst_o, float(_per_pair_rel(o, ref_o, (2,)).max()))
        worst_s = max(worst_s, float(_per_pair_rel(pool[slots_d.long()], ref_s, (2, 3)).max()))
        del ref_s
    assert kda.kda_check_status() == 0
    return worst_o, worst_s, pool, slots


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_small_matches_oracle(kda, cuda_device, d, dtype):
    wo, ws, _, _ = _run_steps(kda, cuda_device, n=7, H=3, d=d, dtype=dtype, steps=5, seed=11 + d)
    if dtype == torch.float32:
        assert wo < FP32_TOL and ws < FP32_TOL, (wo, ws)
    else:
        assert wo < BF16_OUT_TOL and ws < BF16_STATE_TOL, (wo, ws)


def test_decode_mild_decay_many_steps(kda, cuda_device):
    """alpha near 1: the state carries over many steps, so errors would accumulate."""
    wo, ws, _, _ = _run_steps(kda, cuda_device, n=9, H=2, d=128, dtype=torch.bfloat16, steps=48,
                              seed=5, decay="mild")
    assert wo < BF16_OUT_TOL and ws < BF16_STATE_TOL, (wo, ws)


def test_decode_512x32_64_steps(kda, cuda_device):
    """512 sequences x 32 heads, d = 128, 64 consecutive steps, states N(0, 0.05^2)."""
    w = inputs.WORKLOADS["decode_512x32"]
    wo, ws, _, _ = _run_steps(kda, cuda_device, n=w["n_seqs"], H=w["H"], d=w["d"],
                              dtype=torch.bfloat16, steps=w["steps"], seed=w["seed"],
                              std=w["state_std"], n_slots=w["n_seqs"] + 64)
    assert wo < BF16_OUT_TOL and ws < BF16_STATE_TOL, (wo, ws)


def test_decode_leaves_other_slots_untouched(kda, cuda_device):
    dev = cuda_device
    n, H, d = 4, 2, 128
    pool = torch.randn((10, H, d, d), device=dev)
    before = pool.clone()
    slots = torch.tensor([7, 2, 9, 0], dtype=torch.int32, device=dev)
    x = {key: t.to(dev) for key, t in inputs.gen_decode(n, H, d, d, 3, 0).items()}
    o = torch.empty((n, H, d), dtype=torch.bfloat16, device=dev)
    kda.kda_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], pool, slots, o)
    torch.cuda.synchronize()
    untouched = [i for i in range(10) if i not in (7, 2, 9, 0)]
    assert torch.equal(pool[untouched], before[untouched])
    assert not torch.equal(pool[7], before[7])


def test_decode_bad_slot_sets_status_without_touching_memory(kda, cuda_device):
    dev = cuda_device
    n, H, d = 3, 2, 64
    pool = torch.randn((4, H, d, d), device=dev)
    before = pool.clone()
    slots = torch.tensor([1, 4, -2], dtype=torch.int32, device=dev)   # 4 and -2 are outside
    x = {key: t.to(dev) for key, t in inputs.gen_decode(n, H, d, d, 3, 0).items()}
    o = torch.zeros((n, H, d), dtype=torch.bfloat16, device=dev)
    kda.kda_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], pool, slots, o)
    bits = kda.kda_check_status()
    assert bits & kda.KDA_DEV_BAD_SLOT
    assert kda.kda_check_status() == 0                 # reading clears the word
    assert torch.equal(pool[[0, 2, 3]], before[[0, 2, 3]])


def test_decode_is_deterministic(kda, cuda_device):
    dev = cuda_device
    n, H, d = 16, 4, 128
    x = {key: t.to(dev) for key, t in inputs.gen_decode(n, H, d, d, 9, 0).items()}
    S0 = inputs.gen_states(n, H, d, d, 9).to(dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    outs = []
    for _ in range(2):
        pool = S0.clone()
        o = torch.empty((n, H, d), dtype=torch.bfloat16, device=dev)
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], pool, slots, o)
        outs.append((pool, o))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
