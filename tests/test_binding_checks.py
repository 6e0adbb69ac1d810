"""The Python binding checks every tensor before its address crosses the C
boundary.  The C calls take bare pointers and trust the dtype, shape and dense
row-major layout their header states, so a mismatch there would make a kernel
read or write outside the tensor.  These checks need no GPU: structure is
checked before placement, and a CPU tensor is refused before the library is
loaded or called."""
import pytest
import torch

import hybrid_linear_attention_kda_gb300 as kda
from hybrid_linear_attention_kda_gb300.prefix_cache import PrefixCache


@pytest.fixture
def no_library(monkeypatch):
    """Any call that reaches the library fails the test."""
    def refuse():
        raise AssertionError("the binding reached the library with an unchecked tensor")
    monkeypatch.setattr(kda, "load", refuse)


def test_dev_accepts_a_matching_cpu_tensor_only_up_to_placement():
    t = torch.zeros((4, 2, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA device"):
        kda._dev(t, "t", torch.float32, (4, 2, 8))


@pytest.mark.parametrize("bad, kwargs, exc, msg", [
    (3, {}, TypeError, "torch.Tensor"),
    (torch.zeros((4, 2, 8), dtype=torch.bfloat16), {"dtype": torch.float32}, TypeError, "float32"),
    (torch.zeros((4, 2, 8), dtype=torch.int64), {"dtype": (torch.bfloat16, torch.float32)}, TypeError, "bfloat16 or"),
    (torch.zeros((4, 2, 8)), {"shape": (4, 2, 16)}, ValueError, "shape"),
    (torch.zeros((4, 2, 8)), {"shape": (4, 16)}, ValueError, "shape"),
    (torch.zeros((5,), dtype=torch.int32), {"min_numel": 6}, ValueError, "at least 6"),
    (torch.zeros((8, 4)).t(), {}, ValueError, "contiguous"),
    (torch.zeros((4, 2, 16))[:, :, :8], {"shape": (4, 2, 8)}, ValueError, "contiguous"),
])
def test_dev_refuses_each_mismatch(bad, kwargs, exc, msg):
    with pytest.raises(exc, match=msg):
        kda._dev(bad, "t", **kwargs)


def test_dims_requires_the_rank():
    assert kda._dims(torch.zeros((2, 3)), "x", 2) == (2, 3)
    with pytest.raises(ValueError, match="3 dimensions"):
        kda._dims(torch.zeros((2, 3)), "x", 3)


def _prefill_tensors(T=100, H=2, d=64, n=2, dtype=torch.bfloat16):
    return dict(q=torch.zeros((T, H, d), dtype=dtype), k=torch.zeros((T, H, d), dtype=dtype),
                v=torch.zeros((T, H, d), dtype=dtype), alpha=torch.ones((T, H, d)),
                beta=torch.zeros((T, H)), cu_seqlens=torch.tensor([0, 40, T][:n + 1], dtype=torch.int32),
                o=torch.zeros((T, H, d), dtype=dtype))


def test_prefill_args_refuse_more_tokens_than_rows(no_library):
    x = _prefill_tensors()
    with pytest.raises(ValueError, match="total_tokens 101 outside"):
        kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], 101, x["o"])


def test_prefill_args_refuse_host_tensors(no_library):
    x = _prefill_tensors()
    with pytest.raises(ValueError, match="q must be on a CUDA device"):
        kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], 100, x["o"])
    with pytest.raises(ValueError, match="q must have 3 dimensions"):
        kda.prefill(x["q"][0], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"])


@pytest.mark.parametrize("which, bad, msg", [
    ("q", torch.zeros((100, 2, 64), dtype=torch.float16), "q must be"),
    ("q", torch.zeros((100, 2, 64), dtype=torch.bfloat16).transpose(0, 1).contiguous().transpose(0, 1),
     "q must be contiguous"),
])
def test_prefill_args_check_q_before_anything_else(no_library, which, bad, msg):
    x = _prefill_tensors()
    x[which] = bad
    with pytest.raises((TypeError, ValueError), match=msg):
        kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], 100, x["o"])


def test_decode_calls_refuse_host_tensors_before_the_library(no_library):
    n, H, d = 3, 2, 64
    q = torch.zeros((n, H, d), dtype=torch.bfloat16)
    pool = torch.zeros((4, H, d, d))
    slots = torch.zeros(n, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_decode_step(q, q, q, torch.ones((n, H, d)), torch.zeros((n, H)), pool, slots, q)
    q4 = q[:, None]
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_decode_verify(q4, q4, q4, torch.ones((n, 1, H, d)), torch.zeros((n, 1, H)), pool, slots, q4,
                              torch.zeros((n, 1, H, d)))
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_decode_commit(q4, torch.ones((n, 1, H, d)), torch.zeros((n, 1, H, d)), slots, pool, slots)
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_snapshot_gather(pool, slots, torch.zeros((n, H, d, d)))
    with pytest.raises(ValueError, match="CUDA device"):
        kda.kda_snapshot_restore(torch.zeros((n, H, d, d)), pool, slots)
    with pytest.raises(ValueError, match="CUDA device"):
        kda.decode_fused(q, q, q, q, torch.zeros((n, H), dtype=torch.bfloat16), q, torch.zeros((H, 3, 4, d)),
                         torch.ones((H, d)), pool, torch.zeros((4, H, 3, 3, d), dtype=torch.bfloat16), slots, q)


def test_decode_calls_refuse_wrong_dtypes_and_shapes(no_library):
    n, H, d = 3, 2, 64
    q = torch.zeros((n, H, d), dtype=torch.bfloat16)
    pool = torch.zeros((4, H, d, d))
    # q itself is checked through to its placement first; give it the wrong rank or dtype
    with pytest.raises(ValueError, match="q must have 3 dimensions"):
        kda.kda_decode_step(q[0], q, q, torch.ones((n, H, d)), torch.zeros((n, H)), pool,
                            torch.zeros(n, dtype=torch.int32), q)
    with pytest.raises(TypeError, match="q must be"):
        kda.kda_decode_step(q.half(), q, q, torch.ones((n, H, d)), torch.zeros((n, H)), pool,
                            torch.zeros(n, dtype=torch.int32), q)
    with pytest.raises(ValueError, match="pool must have 4 dimensions"):
        kda.kda_snapshot_gather(pool[0], torch.zeros(n, dtype=torch.int32), torch.zeros((n, H, d, d)))
    with pytest.raises(TypeError, match="pool must be"):
        kda.kda_snapshot_gather(pool.double(), torch.zeros(n, dtype=torch.int32), torch.zeros((n, H, d, d)))


def test_state_transfer_refuses_unchecked_buffers():
    pc = PrefixCache(4, slot_base=0, match_unit=256, retention_interval=256)
    pool = torch.zeros((4, 2, 64, 64))
    with pytest.raises(TypeError, match="pool must be"):
        pc.export_states([b"\0" * 32], pool.double(), torch.zeros((2, 2, 64, 64)), torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="pool must have 4 dimensions"):
        pc.import_states([b"\0" * 32], [256], torch.zeros((1, 2, 64, 64)), pool[0],
                         torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA device"):
        pc.import_states([b"\0" * 32], [256], torch.zeros((1, 2, 64, 64)), pool, torch.zeros(1, dtype=torch.int32))
