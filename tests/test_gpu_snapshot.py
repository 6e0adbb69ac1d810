"""Snapshot gather / restore on the GPU: bit-exact copies between the state pool
and contiguous buffers, and the copy-on-write pattern of "Kimi K3 Tech Intro",
section 2.3 (copy the cached state, continue on the copy, the original stays
unchanged)."""
import pytest
import torch

from hybrid_linear_attention_kda_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_gather_restore_round_trip_is_bit_exact(kda, cuda_device, d):
    dev = cuda_device
    H, n_slots = 3, 11
    pool = torch.randn((n_slots, H, d, d), device=dev)
    slots = torch.tensor([4, 0, 10, -1, 7], dtype=torch.int32, device=dev)
    dst = torch.full((5, H, d, d), 123.0, device=dev)
    kda.kda_snapshot_gather(pool, slots, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst[0], pool[4]) and torch.equal(dst[1], pool[0])
    assert torch.equal(dst[2], pool[10]) and torch.equal(dst[4], pool[7])
    assert torch.count_nonzero(dst[3]) == 0                   # slot -1 gives zeros

    pool2 = torch.zeros_like(pool)
    back = torch.tensor([1, 2, 3, -1, 9], dtype=torch.int32, device=dev)
    kda.kda_snapshot_restore(dst, pool2, back)
    torch.cuda.synchronize()
    assert torch.equal(pool2[1], pool[4]) and torch.equal(pool2[2], pool[0])
    assert torch.equal(pool2[3], pool[10]) and torch.equal(pool2[9], pool[7])
    assert torch.count_nonzero(pool2[[0, 4, 5, 6, 7, 8, 10]]) == 0
    assert kda.kda_check_status() == 0


def test_bad_slots_flag_status_and_skip(kda, cuda_device):
    dev = cuda_device
    pool = torch.randn((3, 1, 64, 64), device=dev)
    before = pool.clone()
    dst = torch.zeros((2, 1, 64, 64), device=dev)
    kda.kda_snapshot_gather(pool, torch.tensor([3, 1], dtype=torch.int32, device=dev), dst)
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_SLOT
    assert torch.equal(dst[1], pool[1]) and torch.count_nonzero(dst[0]) == 0
    kda.kda_snapshot_restore(dst, pool, torch.tensor([-7, 0], dtype=torch.int32, device=dev))
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_SLOT
    assert torch.equal(pool[1:], before[1:]) and torch.equal(pool[0], dst[1])


def test_copy_on_write_leaves_the_shared_snapshot_unchanged(kda, cuda_device):
    """Copy a shared cached state to a private slot, decode there: the shared
    original stays bit-identical and later requests still see it."""
    dev = cuda_device
    H, d, n = 4, 128, 2
    pool = torch.zeros((8, H, d, d), device=dev)
    pool[5] = inputs.gen_states(1, H, d, d, 77)[0].to(dev)       # the shared snapshot
    shared = pool[5].clone()
    tmp = torch.empty((n, H, d, d), device=dev)
    kda.kda_snapshot_gather(pool, torch.tensor([5, 5], dtype=torch.int32, device=dev), tmp)
    priv = torch.tensor([1, 2], dtype=torch.int32, device=dev)
    kda.kda_snapshot_restore(tmp, pool, priv)
    for step in range(3):
        x = {key: t.to(dev) for key, t in inputs.gen_decode(n, H, d, d, 78, step).items()}
        o = torch.empty((n, H, d), dtype=torch.bfloat16, device=dev)
        kda.kda_decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], pool, priv, o)
    torch.cuda.synchronize()
    assert torch.equal(pool[5], shared)
    assert not torch.equal(pool[1], shared)
    assert kda.kda_check_status() == 0
