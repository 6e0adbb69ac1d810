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

import numpy as np
import pytest
import torch

from hybrid_linear_attention_kda_gb300 import inputs
from _helpers import BF16_OUT_TOL, BF16_STATE_TOL, rel_rms

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


def test_noalloc_prefill_matches_the_workspace_prefill(kda, cuda_device):
    fn = _noalloc(kda)
    stream = torch.cuda.current_stream(cuda_device)
    data, x, table, init_states, n_slots, total = _case(cuda_device, 91)
    o_ref, fin_ref, pool_ref = _run(kda, fn, x, table, init_states, n_slots, total, False, stream)
    for call in range(2):
        o, fin, pool = _run(kda, fn, x, table, init_states, n_slots, total, True, stream)
        assert not torch.isnan(o.float()).any() and not torch.isnan(fin).any(), call
        assert rel_rms(o.float().cpu(), o_ref.float().cpu()) <= BF16_OUT_TOL, call
        assert rel_rms(fin.cpu(), fin_ref.cpu()) <= BF16_STATE_TOL, call
        assert rel_rms(pool.cpu(), pool_ref.cpu()) <= BF16_STATE_TOL, call


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
