"""The prefill entry point for callers that cannot allocate device memory.

kda_prefill_chunked_noalloc serves callers such as a serving process whose
device memory is all reserved up front, or code that may not call cudaMalloc on
its latency path: it takes its scratch from a fixed 64 MiB array in the
library's own device memory instead of a caller-provided workspace.  Its results
must match kda_prefill_chunked's, call after call (the array keeps the previous
call's contents, and nothing of it may leak into the next result).

This file is collected last so that a stop-at-first-failure run has already
run every other test when it gets here."""
import ctypes

import pytest
import torch

from hybrid_linear_attention_kda_gb300 import inputs

pytestmark = pytest.mark.gpu


def _noalloc(kda):
    lib = kda.load()
    fn = lib.kda_prefill_chunked_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kda.PrefillArgs), ctypes.c_void_p]
    return fn


def _case(dev, seed):
    lens = [300, 64, 1000, 1, 513]
    H, d = 4, 128
    data = inputs.gen_prefill(lens, H, d, d, seed)
    x = {key: data[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
    n = len(lens)
    table = torch.full((n, 4), -1, dtype=torch.int32)
    slot = 2
    for s, L in enumerate(lens):
        for m in range(L // 256):
            table[s, m] = slot
            slot += 1
    init_states = inputs.gen_states(2, H, d, d, seed + 1, std=0.3).to(dev)
    return data, x, table.to(dev), init_states, slot, sum(lens)


def _run(kda, fn, x, table, init_states, n_slots, total, use_noalloc, stream):
    dev = x["q"].device
    H, d = x["q"].shape[1], x["q"].shape[2]
    n = x["cu_seqlens"].shape[0] - 1
    pool = torch.zeros((n_slots, H, d, d), device=dev)
    pool[:2] = init_states
    init_slot = torch.tensor([-1, 0, -1, 1, -1], dtype=torch.int32, device=dev)
    o = torch.full((total, H, d), float("nan"), dtype=torch.bfloat16, device=dev)
    fin = torch.full((n, H, d, d), float("nan"), device=dev)
    if use_noalloc:
        args = kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"],
                                     total, o, init_slot=init_slot, pool=pool, snap_table=table,
                                     final_state=fin)
        assert fn(ctypes.byref(args), stream.cuda_stream) == 0, kda.load().kda_last_error()
    else:
        kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], total_tokens=total,
                    init_slot=init_slot, pool=pool, snap_table=table, o=o, final_state=fin,
                    stream=stream)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    return o, fin, pool


def _dirty_the_scratch(kda, fn, dev, stream):
    """A different, larger batch through the no-alloc call first, with gates that
    leave the kernels' usual range in some channels, so that the static scratch
    holds another batch's chunk table and intermediates when the compared calls
    run."""
    lens = [2000, 3000, 7]
    H, d = 4, 128
    data = inputs.gen_prefill(lens, H, d, d, 97)
    data["alpha"][100:180, :, :20] = 1e-30
    data["alpha"][900:1000] = 1.0
    x = {key: data[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
    total = sum(lens)
    o = torch.empty((total, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((len(lens), H, d, d), device=dev)
    args = kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"], total, o,
                                 final_state=fin)
    assert fn(ctypes.byref(args), stream.cuda_stream) == 0, kda.load().kda_last_error()
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0


def test_noalloc_prefill_matches_the_workspace_prefill(kda, cuda_device):
    """Two no-alloc calls in a row, after another batch has used the scratch,
    give exactly the workspace prefill's outputs, final states and snapshots:
    the same kernels run on the same bytes, so any difference would be stale
    scratch leaking into a result."""
    fn = _noalloc(kda)
    stream = torch.cuda.current_stream(cuda_device)
    _dirty_the_scratch(kda, fn, cuda_device, stream)
    data, x, table, init_states, n_slots, total = _case(cuda_device, 91)
    o_ref, fin_ref, pool_ref = _run(kda, fn, x, table, init_states, n_slots, total, False, stream)
    assert not torch.isnan(o_ref.float()).any() and not torch.isnan(fin_ref).any()
    for call in range(2):
        o, fin, pool = _run(kda, fn, x, table, init_states, n_slots, total, True, stream)
        assert torch.equal(o, o_ref), call
        assert torch.equal(fin, fin_ref), call
        assert torch.equal(pool, pool_ref), call


def test_noalloc_rejects_a_batch_beyond_its_scratch(kda, cuda_device):
    fn = _noalloc(kda)
    H, d, T = 32, 128, 64 * 1024          # (1024 + 1) chunks x 32 heads x 72.5 KiB > 64 MiB
    q = torch.empty((T, H, d), dtype=torch.bfloat16, device=cuda_device)
    a = torch.empty((T, H, d), dtype=torch.float32, device=cuda_device)
    b = torch.empty((T, H), dtype=torch.float32, device=cuda_device)
    cu = torch.tensor([0, T], dtype=torch.int32, device=cuda_device)
    o = torch.empty_like(q)
    args = kda.make_prefill_args(q, q, q, a, b, cu, T, o)
    assert fn(ctypes.byref(args), None) == kda.KDA_ERR_UNSUPPORTED
    assert b"64 MiB" in kda.load().kda_last_error()
