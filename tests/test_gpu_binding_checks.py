"""With CUDA tensors, the binding refuses each operand whose dtype, shape or
layout differs from what the C header states, and launches nothing."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _prefill_tensors(dev, T=300, H=2, d=128):
    bf = torch.bfloat16
    return dict(q=torch.zeros((T, H, d), dtype=bf, device=dev), k=torch.zeros((T, H, d), dtype=bf, device=dev),
                v=torch.zeros((T, H, d), dtype=bf, device=dev), alpha=torch.ones((T, H, d), device=dev),
                beta=torch.zeros((T, H), device=dev),
                cu_seqlens=torch.tensor([0, 100, T], dtype=torch.int32, device=dev))


@pytest.mark.parametrize("key, make, msg", [
    ("alpha", lambda x: x["alpha"].bfloat16(), "alpha must be"),
    ("beta", lambda x: x["beta"][:, :1], "beta must have shape"),
    ("k", lambda x: x["k"].float(), "k must be"),
    ("v", lambda x: x["v"][:200], "v must have shape"),
    ("cu_seqlens", lambda x: x["cu_seqlens"].long(), "cu_seqlens must be"),
    ("alpha", lambda x: x["alpha"].transpose(1, 2).contiguous().transpose(1, 2), "alpha must be contiguous"),
])
def test_prefill_refuses_each_bad_operand(kda, cuda_device, key, make, msg):
    x = _prefill_tensors(cuda_device)
    x[key] = make(x)
    before = kda.kda_launch_count()
    with pytest.raises((TypeError, ValueError), match=msg):
        kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"])
    assert kda.kda_launch_count() == before


def test_prefill_refuses_bad_optional_operands(kda, cuda_device):
    dev = cuda_device
    x = _prefill_tensors(dev)
    pool = torch.zeros((4, 2, 128, 128), device=dev)
    before = kda.kda_launch_count()
    cases = [
        (dict(start_pos=torch.zeros(2, dtype=torch.int64, device=dev)), "start_pos must be"),
        (dict(init_slot=torch.zeros(3, dtype=torch.int32, device=dev), pool=pool), "init_slot must have shape"),
        (dict(pool=pool[:, :1]), "pool must have shape"),
        (dict(pool=pool, snap_table=torch.zeros((1, 4), dtype=torch.int32, device=dev)), "snap_table must have shape"),
        (dict(final_state=torch.zeros((2, 2, 128, 128), dtype=torch.bfloat16, device=dev)), "final_state must be"),
        (dict(o=torch.zeros((300, 2, 128), device=dev)), "o must be"),
    ]
    for kw, msg in cases:
        with pytest.raises((TypeError, ValueError), match=msg):
            kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], **kw)
    with pytest.raises(ValueError, match="total_tokens 301 outside"):
        kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], total_tokens=301)
    assert kda.kda_launch_count() == before


def test_decode_calls_refuse_bad_operands(kda, cuda_device):
    dev = cuda_device
    n, T, H, d = 4, 2, 2, 128
    bf = torch.bfloat16
    q = torch.zeros((n, H, d), dtype=bf, device=dev)
    pool = torch.zeros((n, H, d, d), device=dev)
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    alpha, beta = torch.ones((n, H, d), device=dev), torch.zeros((n, H), device=dev)
    before = kda.kda_launch_count()
    with pytest.raises(TypeError, match="state_slot must be"):
        kda.kda_decode_step(q, q, q, alpha, beta, pool, slots.long(), q)
    with pytest.raises(TypeError, match="alpha must be"):
        kda.kda_decode_step(q, q, q, alpha.bfloat16(), beta, pool, slots, q)
    with pytest.raises(ValueError, match="pool must have shape"):
        kda.kda_decode_step(q, q, q, alpha, beta, pool[:, :, :64], slots, q)
    q4 = torch.zeros((n, T, H, d), dtype=bf, device=dev)
    a4, b4 = torch.ones((n, T, H, d), device=dev), torch.zeros((n, T, H), device=dev)
    with pytest.raises(TypeError, match="u must be"):
        kda.kda_decode_verify(q4, q4, q4, a4, b4, pool, slots, q4, q4)
    with pytest.raises(TypeError, match="n_accept must be"):
        kda.kda_decode_commit(q4, a4, torch.zeros((n, T, H, d), device=dev), slots.float(), pool, slots)
    with pytest.raises(ValueError, match="dst must have shape"):
        kda.kda_snapshot_gather(pool, slots, torch.zeros((n - 1, H, d, d), device=dev))
    with pytest.raises(ValueError, match="conv_state must have shape"):
        kda.decode_fused(q, q, q, q, torch.zeros((n, H), dtype=bf, device=dev), q,
                         torch.zeros((H, 3, 4, d), device=dev), torch.ones((H, d), device=dev), pool,
                         torch.zeros((n, H, 3, 4, d), dtype=bf, device=dev), slots, q)
    assert kda.kda_launch_count() == before
