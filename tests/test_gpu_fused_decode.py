"""The fused decode step (kda_decode_fused) against the float64 oracle
("Kimi K3 Tech Intro", section 4.1): causal convolution with its state, q/k
norm, gates, recurrent update and gated RMSNorm in one kernel.

The GPU and the oracle each evolve their own convolution and recurrent states
over 16 consecutive tokens.  After every token the test compares:
* the output, bf16, relative RMS per (sequence, head);
* the recurrent state, relative Frobenius per (sequence, head);
* the convolution state, which holds exact copies of the raw bf16 inputs, bit
  for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_kda_gb300 import inputs, KDA_DEV_BAD_SLOT
from _helpers import BF16_OUT_TOL, FP32_TOL, rel_rms

pytestmark = pytest.mark.gpu


def frob_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _step(kda, dev, z, conv_w, norm_w, pool, conv_state, slots):
    n, H, d = z["xq"].shape
    zd = {k: t.to(dev) for k, t in z.items()}
    y = torch.empty((n, H, d), dtype=torch.bfloat16, device=dev)
    kda.decode_fused(zd["xq"], zd["xk"], zd["xv"], zd["a"], zd["b"], zd["g"], conv_w, norm_w, pool,
                     conv_state, slots, y)
    return y


@pytest.mark.parametrize("d", [64, 128])
def test_fused_steps_match_the_oracle(kda, cuda_device, d):
    dev = cuda_device
    n, H, steps = 8, 4, 16
    conv_w, norm_w = inputs.gen_fused_params(H, d, 71)
    S = inputs.gen_states(n, H, d, d, 72, std=0.05)
    C = inputs.gen_conv_states(n, H, d, 73)
    slots = torch.tensor([2 * i + 1 for i in range(n)], dtype=torch.int32, device=dev)
    pool = torch.zeros((2 * n + 1, H, d, d), device=dev)
    cpool = torch.zeros((2 * n + 1, H, 3, 3, d), dtype=torch.bfloat16, device=dev)
    pool[slots.long()] = S.to(dev)
    cpool[slots.long()] = C.to(dev)
    untouched = pool[0::2].clone()
    cw, nw = conv_w.to(dev), norm_w.to(dev)
    S_ref, C_ref = S.double().numpy(), C.double().numpy()
    for t in range(steps):
        z = inputs.gen_fused_step(n, H, d, 74, t)
        y = _step(kda, dev, z, cw, nw, pool, cpool, slots)
        torch.cuda.synchronize()
        assert kda.kda_check_status() == 0
        y_ref, S_ref, C_ref = oracle.fused_step(S_ref, C_ref, z["xq"], z["xk"], z["xv"], z["a"], z["b"], z["g"],
                                                conv_w, norm_w)
        got_S = pool[slots.long()].cpu()
        got_C = cpool[slots.long()].cpu()
        assert torch.equal(got_C.double(), torch.from_numpy(C_ref)), t
        for i in range(n):
            for h in range(H):
                assert rel_rms(y[i, h].float().cpu(), y_ref[i, h]) < BF16_OUT_TOL, (t, i, h)
                assert frob_rel(got_S[i, h], S_ref[i, h]) < FP32_TOL, (t, i, h)
    assert torch.equal(pool[0::2], untouched)


def test_bad_slot_is_flagged(kda, cuda_device):
    dev = cuda_device
    n, H, d = 3, 2, 128
    conv_w, norm_w = inputs.gen_fused_params(H, d, 81)
    pool = inputs.gen_states(n, H, d, d, 82).to(dev)
    cpool = inputs.gen_conv_states(n, H, d, 83).to(dev)
    before, cbefore = pool.clone(), cpool.clone()
    slots = torch.tensor([0, n + 4, 2], dtype=torch.int32, device=dev)
    _step(kda, dev, inputs.gen_fused_step(n, H, d, 84, 0), conv_w.to(dev), norm_w.to(dev), pool, cpool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == KDA_DEV_BAD_SLOT
    assert torch.equal(pool[1], before[1]) and torch.equal(cpool[1], cbefore[1])
    assert not torch.equal(pool[0], before[0])


def test_full_decode_batch_sampled(kda, cuda_device):
    """512 sequences x 32 heads, d = 128 (1 GiB of states): sampled heads."""
    dev = cuda_device
    w = inputs.WORKLOADS["decode_512x32"]
    n, H, d = w["n_seqs"], w["H"], w["d"]
    conv_w, norm_w = inputs.gen_fused_params(H, d, w["seed"])
    S = inputs.gen_states(n, H, d, d, w["seed"], std=w["state_std"])
    C = inputs.gen_conv_states(n, H, d, w["seed"])
    pool, cpool = S.to(dev), C.to(dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    z = inputs.gen_fused_step(n, H, d, w["seed"], 0)
    y = _step(kda, dev, z, conv_w.to(dev), norm_w.to(dev), pool, cpool, slots)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    seqs = np.random.default_rng(9).choice(n, size=8, replace=False)
    y_ref, S_ref, C_ref = oracle.fused_step(S[seqs].double().numpy(), C[seqs].double().numpy(),
                                            *(z[k][seqs] for k in ("xq", "xk", "xv", "a", "b", "g")),
                                            conv_w, norm_w)
    for r, i in enumerate(seqs):
        for h in range(H):
            assert rel_rms(y[i, h].float().cpu(), y_ref[r, h]) < BF16_OUT_TOL
            assert frob_rel(pool[i, h].cpu(), S_ref[r, h]) < FP32_TOL
        assert torch.equal(cpool[i].cpu().double(), torch.from_numpy(C_ref[r]))
