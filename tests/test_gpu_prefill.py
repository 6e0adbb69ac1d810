"""Chunked prefill on the GPU against the float64 oracle.

Covers the five workloads (the tiny fp32 check, 4 x 8192 prefill, the 2^20-token
sequence, the mixed varlen batch with resumes from a shared prefix) plus edge
cases: empty and one-token sequences, ragged tails, resume at snapshot
boundaries, mild and pathological gates, bad indices reported by the device.

Snapshots follow "Kimi K3 Tech Intro", sections 2.2-2.4: a state after every
256th absolute position, written into a block-indexed pool, reused by later
requests through copy-on-write.
"""
import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_kda_gb300 import inputs
from _helpers import (BF16_OUT_TOL, BF16_STATE_TOL, FP32_TOL, rel_rms, to_dev,
                      worst_out_err, worst_state_err)

pytestmark = pytest.mark.gpu


def run_gpu(kda, dev, d, *, start_pos=None, init_slot=None, pool=None, snap_table=None,
            scale=1.0, check=True):
    x = to_dev(d, dev)
    cu = d["cu_seqlens"].to(dev)
    sp = None if start_pos is None else torch.as_tensor(start_pos, dtype=torch.int32).to(dev)
    ins = None if init_slot is None else torch.as_tensor(init_slot, dtype=torch.int32).to(dev)
    st = None if snap_table is None else torch.as_tensor(snap_table, dtype=torch.int32).to(dev)
    # outputs start as NaN: anything the library leaves unwritten fails the comparison
    T, H, d_k = x["q"].shape
    d_v = x["v"].shape[2]
    o = torch.full((T, H, d_v), float("nan"), dtype=x["v"].dtype, device=dev)
    fin = torch.full((cu.shape[0] - 1, H, d_k, d_v), float("nan"), device=dev)
    o, fin = kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], cu,
                         total_tokens=int(d["cu_seqlens"][-1]), start_pos=sp, init_slot=ins,
                         pool=pool, snap_table=st, scale=scale, o=o, final_state=fin)
    torch.cuda.synchronize()
    if check:
        assert kda.kda_check_status() == 0
    return o, fin


def frob_rel(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


# ------------------------------------------------------------------ tiny fp32

def test_tiny_fp32_with_snapshots_and_resume(kda, cuda_device):
    """B=1, H=2, T=512, d=64, fp32; snapshots at 256 and 512; resume at 256."""
    w = inputs.WORKLOADS["tiny_fp32"]
    dev = cuda_device
    d = inputs.gen_prefill([w["T"]], w["H"], w["d"], w["d"], w["seed"], dtype=torch.float32)
    pool = torch.zeros((4, w["H"], w["d"], w["d"]), device=dev)
    o, fin = run_gpu(kda, dev, d, pool=pool, snap_table=[[0, 1]])
    ref = oracle.run(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["cu_seqlens"],
                     snap_req=[(0, 0), (0, 1)])
    for h in range(w["H"]):
        assert frob_rel(o[:, h].cpu(), ref["o"][:, h]) < FP32_TOL
        assert frob_rel(fin[0, h].cpu(), ref["final"][0, h]) < FP32_TOL
        for m in (0, 1):
            assert frob_rel(pool[m, h].cpu(), ref["snaps"][m, h]) < FP32_TOL
    assert torch.equal(pool[1], fin[0])               # p = T = 512 is a snapshot position

    p = w["resume_at"]
    tail = {key: d[key][p:] for key in ("q", "k", "v", "alpha", "beta")}
    tail["cu_seqlens"] = torch.tensor([0, w["T"] - p], dtype=torch.int32)
    o2, fin2 = run_gpu(kda, dev, tail, start_pos=[p], init_slot=[0], pool=pool,
                       snap_table=[[-1, 2]])
    assert torch.equal(o2, o[p:]) and torch.equal(fin2, fin)
    assert torch.equal(pool[2], pool[1])
    ref2 = oracle.run(tail["q"], tail["k"], tail["v"], tail["alpha"], tail["beta"],
                      tail["cu_seqlens"], start_pos=[p], init_state=ref["snaps"][0:1])
    assert np.array_equal(ref2["o"], ref["o"][p:])        # the oracle resumes bit for bit too
    assert frob_rel(o2.cpu(), ref2["o"]) < FP32_TOL


# ------------------------------------------------------------------ small mixed batches

LENS = [300, 1, 64, 129, 0, 700, 256, 513, 65]
STARTS = [0, 256, 0, 512, 0, 0, 768, 0, 256]
INITS = [-1, 3, -1, 5, 1, -1, 0, -1, 2]


def _mixed_case(dtype, d, decay, seed, H=4):
    data = inputs.gen_prefill(LENS, H, d, d, seed, dtype=dtype, decay=decay)
    init_states = inputs.gen_states(6, H, d, d, seed + 1, std=0.3)
    stride = 8
    n = len(LENS)
    table = np.full((n, stride), -1, np.int32)
    req = []
    for s in range(n):
        for p in oracle.snapshot_positions(STARTS[s], LENS[s], 256):
            m = p // 256 - 1
            table[s, m] = 6 + s * stride + m
            req.append((s, m))
    return data, init_states, table, req


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 128), (torch.float32, 64)])
@pytest.mark.parametrize("decay", ["config", "mild"])
def test_mixed_varlen_resume_snapshots(kda, cuda_device, dtype, d, decay):
    dev = cuda_device
    H = 4
    data, init_states, table, req = _mixed_case(dtype, d, decay, 31 + d, H)
    n = len(LENS)
    pool = torch.zeros((6 + n * 8, H, d, d), device=dev)
    pool[:6] = init_states.to(dev)
    o, fin = run_gpu(kda, dev, data, start_pos=STARTS, init_slot=INITS, pool=pool,
                     snap_table=table)
    init64 = np.zeros((n, H, d, d))
    for s, slot in enumerate(INITS):
        if slot >= 0:
            init64[s] = init_states[slot].double().numpy()
    ref = oracle.run(data["q"], data["k"], data["v"], data["alpha"], data["beta"],
                     data["cu_seqlens"], start_pos=STARTS, init_state=init64, snap_req=req)
    snaps = np.stack([pool[table[s, m]].cpu().numpy() for s, m in req])
    if dtype == torch.float32:
        cu = data["cu_seqlens"].tolist()
        for s in range(n):
            for h in range(H):
                if cu[s + 1] > cu[s]:
                    assert frob_rel(o[cu[s]:cu[s + 1], h].cpu(), ref["o"][cu[s]:cu[s + 1], h]) < FP32_TOL
                assert frob_rel(fin[s, h].cpu(), ref["final"][s, h]) < FP32_TOL
        for i in range(len(req)):
            for h in range(H):
                assert frob_rel(snaps[i, h], ref["snaps"][i, h]) < FP32_TOL
    else:
        assert worst_out_err(o.float().cpu(), ref["o"], data["cu_seqlens"]) < BF16_OUT_TOL
        assert worst_state_err(fin.cpu(), ref["final"]) < BF16_STATE_TOL
        assert worst_state_err(snaps, ref["snaps"]) < BF16_STATE_TOL
    # an empty sequence keeps its initial state exactly
    assert torch.equal(fin[4], pool[1])
    # pool slots that no snapshot maps to are untouched
    used = set(int(x) for x in table.ravel() if x >= 0)
    unused = [i for i in range(6, pool.shape[0]) if i not in used]
    assert torch.count_nonzero(pool[unused]) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_resume_is_bit_exact_against_the_full_run(kda, cuda_device, dtype):
    """Resuming at every snapshot boundary of a 1100-token run (mild decay, so the
    carried state matters) reproduces the full run's outputs, final state and
    later snapshots bit for bit."""
    dev = cuda_device
    T, H, d = 1100, 3, 128
    data = inputs.gen_prefill([T], H, d, d, 41, dtype=dtype, decay="mild")
    pool = torch.zeros((8, H, d, d), device=dev)
    o, fin = run_gpu(kda, dev, data, pool=pool, snap_table=[[0, 1, 2, 3]])
    for m in range(4):
        p = 256 * (m + 1)
        tail = {key: data[key][p:] for key in ("q", "k", "v", "alpha", "beta")}
        tail["cu_seqlens"] = torch.tensor([0, T - p], dtype=torch.int32)
        table = [[-1] * 4]
        for mm in range(m + 1, 4):
            table[0][mm] = 4 + mm
        pool[4:] = 0
        o2, fin2 = run_gpu(kda, dev, tail, start_pos=[p], init_slot=[m], pool=pool,
                           snap_table=table)
        assert torch.equal(o2, o[p:]), m
        assert torch.equal(fin2, fin), m
        for mm in range(m + 1, 4):
            assert torch.equal(pool[4 + mm], pool[mm]), (m, mm)


def test_pathological_gates(kda, cuda_device):
    """alpha exactly 1, alpha down to 1e-30 and exactly 0, beta 0 and 1, in runs
    of tokens: the chunks whose decay factors leave the tensor-core operand range
    are rewritten from exact products of alphas."""
    dev = cuda_device
    T, H, d = 333, 2, 128
    data = inputs.gen_prefill([T], H, d, d, 53, dtype=torch.bfloat16)
    a = data["alpha"]
    a[10:40] = 1.0
    a[50:90, :, :17] = 1e-30
    a[100:140] = 1e-12
    a[200:230, 1] = 0.999999
    a[260:262, 0, 40:48] = 0.0          # outside (0, 1): a hard reset of those channels
    b = data["beta"]
    b[20:30] = 0.0
    b[150:170] = 1.0
    o, fin = run_gpu(kda, dev, data)
    ref = oracle.run(data["q"], data["k"], data["v"], a, b, data["cu_seqlens"])
    assert worst_out_err(o.float().cpu(), ref["o"], data["cu_seqlens"]) < BF16_OUT_TOL
    assert worst_state_err(fin.cpu(), ref["final"]) < BF16_STATE_TOL


def test_output_scale(kda, cuda_device):
    dev = cuda_device
    data = inputs.gen_prefill([200, 77], 2, 128, 128, 61, dtype=torch.float32)
    o, fin = run_gpu(kda, dev, data, scale=0.125)
    ref = oracle.run(data["q"], data["k"], data["v"], data["alpha"], data["beta"],
                     data["cu_seqlens"], scale=0.125)
    assert frob_rel(o.cpu(), ref["o"]) < FP32_TOL
    assert frob_rel(fin.cpu(), ref["final"]) < FP32_TOL


def test_prefill_is_deterministic(kda, cuda_device):
    dev = cuda_device
    data = inputs.gen_prefill([700, 333], 4, 128, 128, 71)
    o1, f1 = run_gpu(kda, dev, data)
    o2, f2 = run_gpu(kda, dev, data)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


# ------------------------------------------------------------------ device-reported errors

def test_bad_start_position_is_reported_and_skipped(kda, cuda_device):
    dev = cuda_device
    data = inputs.gen_prefill([100, 100], 2, 128, 128, 81)
    o = torch.full((200, 2, 128), 7.0, dtype=torch.bfloat16, device=dev)
    x = to_dev(data, dev)
    kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], data["cu_seqlens"].to(dev),
                total_tokens=200, start_pos=torch.tensor([0, 100], dtype=torch.int32, device=dev),
                o=o)
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_START
    assert torch.all(o[100:] == 7.0)                      # the bad sequence wrote nothing
    assert not torch.all(o[:100] == 7.0)


def test_bad_slots_and_ordinals_are_reported(kda, cuda_device):
    dev = cuda_device
    H, d = 2, 128
    data = inputs.gen_prefill([600], H, d, d, 83)
    pool = torch.zeros((3, H, d, d), device=dev)
    run_gpu(kda, dev, data, pool=pool, snap_table=[[0]], check=False)   # ordinal 1 has no entry
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_ORDINAL
    run_gpu(kda, dev, data, pool=pool, snap_table=[[0, 9]], check=False)  # slot 9 >= 3
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_SLOT
    run_gpu(kda, dev, data, init_slot=[5], pool=pool, check=False)
    assert kda.kda_check_status() & kda.KDA_DEV_BAD_SLOT


# ------------------------------------------------------------------ 4 x 8192 prefill

def test_prefill_4x8k_every_head(kda, cuda_device):
    """4 sequences x 8192 tokens, 32 heads, d = 128, bf16, in the launch
    configuration the benchmark times: every output, final state and snapshot of
    every (sequence, head) against the oracle."""
    w = inputs.WORKLOADS["prefill_4x8k"]
    dev = cuda_device
    H, d, T, n = w["H"], w["d"], w["T"], w["n_seqs"]
    data = inputs.gen_prefill([T] * n, H, d, d, w["seed"])
    n_ord = T // 256
    table = np.arange(n * n_ord, dtype=np.int32).reshape(n, n_ord)
    pool = torch.zeros((n * n_ord, H, d, d), device=dev)
    o, fin = run_gpu(kda, dev, data, pool=pool, snap_table=table)
    req = [(s, m) for s in range(n) for m in range(n_ord)]
    ref = oracle.run(data["q"], data["k"], data["v"], data["alpha"], data["beta"],
                     data["cu_seqlens"], snap_req=req)
    assert worst_out_err(o.float().cpu(), ref["o"], data["cu_seqlens"]) < BF16_OUT_TOL
    assert worst_state_err(fin.cpu(), ref["final"]) < BF16_STATE_TOL
    snaps = pool[torch.as_tensor([table[s, m] for s, m in req], device=dev).long()].cpu()
    assert worst_state_err(snaps, ref["snaps"]) < BF16_STATE_TOL
    assert torch.equal(pool[table[:, -1]], fin)         # p = T is the last snapshot


# ------------------------------------------------------------------ 2^20-token sequence

def _state_bound(alpha, beta, k, v):
    """sup_t |S_t|_F for a run from zero: |S_t| <= a |S_{t-1}| + b_t |k_t||v_t|
    with a = max alpha < 1, so |S| <= max_t(b_t |k_t| |v_t|) / (1 - a)."""
    amax = float(alpha.max())
    assert amax < 1.0
    kn = torch.linalg.vector_norm(k.float(), dim=-1)
    vn = torch.linalg.vector_norm(v.float(), dim=-1)
    return float((beta * kn * vn).max()) * 1.001 / (1.0 - amax)


def test_long_1m_windows_and_resume(kda, cuda_device):
    """One sequence of 2^20 tokens, 8 heads: snapshots every 256 tokens (4096 per
    head), a resume from the snapshot at 2^19 reproduces the full run bit for bit,
    and the oracle checks windows along the sequence.  Each window runs the oracle
    from a zero state 512 tokens early; the forgetting bound (at most
    prod(max alpha) times the largest possible state) shows the skipped history
    changes the window's states by far less than the tolerance."""
    w = inputs.WORKLOADS["long_1m"]
    dev = cuda_device
    H, d, T = w["H"], w["d"], w["T"]
    data = inputs.gen_prefill([T], H, d, d, w["seed"])
    n_ord = T // 256
    pool = torch.zeros((n_ord + n_ord // 2, H, d, d), device=dev)
    table = np.arange(n_ord, dtype=np.int32)[None]
    o, fin = run_gpu(kda, dev, data, pool=pool, snap_table=table)
    assert torch.equal(pool[n_ord - 1], fin[0])

    p = w["resume_at"]
    tail = {key: data[key][p:] for key in ("q", "k", "v", "alpha", "beta")}
    tail["cu_seqlens"] = torch.tensor([0, T - p], dtype=torch.int32)
    table2 = np.full((1, n_ord), -1, np.int32)
    table2[0, p // 256:] = n_ord + np.arange(n_ord - p // 256)
    o2, fin2 = run_gpu(kda, dev, tail, start_pos=[p], init_slot=[p // 256 - 1], pool=pool,
                       snap_table=table2)
    assert torch.equal(o2, o[p:])
    assert torch.equal(fin2, fin)
    assert torch.equal(pool[n_ord:], pool[p // 256:n_ord])
    del o2, tail

    S_bound = _state_bound(data["alpha"], data["beta"], data["k"], data["v"])
    burn, W = 512, 512
    for start in (0, 262144, p, T - W):
        lo = max(0, start - burn)
        win = {key: data[key][lo:start + W] for key in ("q", "k", "v", "alpha", "beta")}
        snaps = [(0, m) for m in range(start // 256, (start + W) // 256)]
        ref = oracle.run(win["q"], win["k"], win["v"], win["alpha"], win["beta"],
                         [0, start + W - lo], start_pos=[lo], snap_req=snaps)
        if lo > 0:
            bound = oracle.window_bound(win["alpha"][:start - lo].double().amax(dim=1).numpy()) * S_bound
            assert bound < 1e-30
        go = o[start:start + W].float().cpu()
        for h in range(H):
            assert rel_rms(go[:, h], ref["o"][start - lo:, h]) < BF16_OUT_TOL
            for i, (_, m) in enumerate(snaps):
                assert rel_rms(pool[m, h].cpu(), ref["snaps"][i, h]) < BF16_STATE_TOL
        if start + W == T:
            for h in range(H):
                assert rel_rms(fin[0, h].cpu(), ref["final"][0, h]) < BF16_STATE_TOL


# ------------------------------------------------------------------ mixed varlen batch

def test_varlen_64_shared_prefix_resume(kda, cuda_device):
    """64 sequences, lengths uniform in [1, 16384]; 32 resume from the shared
    prefix's snapshots (a prefix run fills them first).  Resumed sequences
    re-create the prefix's later snapshots bit for bit; the oracle checks every
    head of every sequence (outputs, final states and every snapshot), starting
    resumed ones from its own prefix states."""
    w = inputs.WORKLOADS["varlen_64"]
    dev = cuda_device
    H, d, P = w["H"], w["d"], w["prefix_len"]
    data = inputs.gen_varlen_resume(w["n_seqs"], H, d, d, w["max_len"], P, w["n_resume"],
                                    w["seed"])
    n = w["n_seqs"]
    n_pref = P // 256
    # slots: [0, n_pref) prefix snapshots; then one block of ordinals per sequence
    max_ord = (w["max_len"] + 255) // 256
    table = np.full((n, max_ord), -1, np.int32)
    nxt = n_pref
    for s in range(n):
        for pos in oracle.snapshot_positions(int(data["start_pos"][s]), data["lens"][s] - int(data["start_pos"][s]), 256):
            table[s, pos // 256 - 1] = nxt
            nxt += 1
    pool = torch.zeros((nxt, H, d, d), device=dev)

    pref = dict(data["prefix"])
    pref["cu_seqlens"] = torch.tensor([0, P], dtype=torch.int32)
    run_gpu(kda, dev, pref, pool=pool, snap_table=[list(range(n_pref))])

    start = data["start_pos"].tolist()
    init = [(p // 256 - 1) if p > 0 else -1 for p in start]
    o, fin = run_gpu(kda, dev, data, start_pos=start, init_slot=init, pool=pool, snap_table=table)

    for s in data["resumed"]:
        for m in range(start[s] // 256, n_pref):
            if table[s, m] >= 0:
                assert torch.equal(pool[table[s, m]], pool[m]), (s, m)

    # every head, four at a time (the float64 reference of all 32 would not fit
    # in host memory at once); every snapshot the batch wrote
    cu = data["cu_seqlens"].tolist()
    req = [(s, int(m)) for s in range(n) for m in np.nonzero(table[s] >= 0)[0]]
    snap_idx = torch.as_tensor([table[s, m] for s, m in req], device=dev).long()
    keys = ("q", "k", "v", "alpha", "beta")
    for h0 in range(0, H, 4):
        sl = slice(h0, h0 + 4)
        pv = {key: pref[key][:, sl].contiguous() for key in keys}
        pr = oracle.run(pv["q"], pv["k"], pv["v"], pv["alpha"], pv["beta"], [0, P],
                        snap_req=[(0, m) for m in range(n_pref)])
        init64 = np.zeros((n, 4, d, d))
        for s in range(n):
            if start[s] > 0:
                init64[s] = pr["snaps"][start[s] // 256 - 1]
        dv = {key: data[key][:, sl].contiguous() for key in keys}
        ref = oracle.run(dv["q"], dv["k"], dv["v"], dv["alpha"], dv["beta"],
                         data["cu_seqlens"], start_pos=start, init_state=init64, snap_req=req)
        og = o[:, sl].float().cpu()
        fg = fin[:, sl].cpu()
        sg = pool[snap_idx, sl].cpu()
        for s in range(n):
            for j in range(4):
                if cu[s + 1] > cu[s]:
                    assert rel_rms(og[cu[s]:cu[s + 1], j], ref["o"][cu[s]:cu[s + 1], j]) < BF16_OUT_TOL, (s, h0 + j)
                assert rel_rms(fg[s, j], ref["final"][s, j]) < BF16_STATE_TOL, (s, h0 + j)
        for i in range(len(req)):
            for j in range(4):
                assert rel_rms(sg[i, j], ref["snaps"][i, j]) < BF16_STATE_TOL, (req[i], h0 + j)
        del ref, og, fg, sg, dv


# ------------------------------------------------------------------ long chains split into segments

# The segment length of split chains (absolute positions at its multiples are
# segment boundaries, where a resumed run splits as the full run does).
SEG_TOKENS = 57344

def test_split_chain_matches_oracle_and_resumes(kda, cuda_device):
    """One sequence of 2^18 tokens, 4 heads, mild decay (the state carried over a
    segment boundary matters): the chain is split at multiples of the library's
    segment length (57,344 tokens) and the segments run in parallel from scanned
    start states.  The whole run
    is checked against the oracle; a resume at a segment boundary reproduces the
    full run bit for bit, a resume inside a segment stays within tolerance."""
    dev = cuda_device
    H, d, T = 4, 128, 1 << 18
    data = inputs.gen_prefill([T], H, d, d, 20268, decay="mild")
    n_ord = T // 256
    pool = torch.zeros((n_ord + n_ord, H, d, d), device=dev)
    table = np.arange(n_ord, dtype=np.int32)[None]
    o, fin = run_gpu(kda, dev, data, pool=pool, snap_table=table)
    checks = [SEG_TOKENS, 100096, 2 * SEG_TOKENS, 3 * SEG_TOKENS + 2560]
    ref = oracle.run(data["q"], data["k"], data["v"], data["alpha"], data["beta"], [0, T],
                     snap_req=[(0, p // 256 - 1) for p in checks])
    for h in range(H):
        assert rel_rms(o[:, h].float().cpu(), ref["o"][:, h]) < BF16_OUT_TOL, h
        assert rel_rms(fin[0, h].cpu(), ref["final"][0, h]) < BF16_STATE_TOL, h
        for i, p in enumerate(checks):
            assert rel_rms(pool[p // 256 - 1, h].cpu(), ref["snaps"][i, h]) < BF16_STATE_TOL, (p, h)

    for p, exact in ((2 * SEG_TOKENS, True), (100096, False)):
        tail = {key: data[key][p:] for key in ("q", "k", "v", "alpha", "beta")}
        tail["cu_seqlens"] = torch.tensor([0, T - p], dtype=torch.int32)
        table2 = np.full((1, n_ord), -1, np.int32)
        table2[0, p // 256:] = n_ord + np.arange(n_ord - p // 256)
        o2, fin2 = run_gpu(kda, dev, tail, start_pos=[p], init_slot=[p // 256 - 1], pool=pool,
                           snap_table=table2)
        if exact:
            assert torch.equal(o2, o[p:])
            assert torch.equal(fin2, fin)
            assert torch.equal(pool[n_ord:2 * n_ord - p // 256], pool[p // 256:n_ord])
        else:
            for h in range(H):
                assert rel_rms(o2[:, h].float().cpu(), o[p:, h].float().cpu()) < BF16_OUT_TOL
                assert rel_rms(fin2[0, h].cpu(), fin[0, h].cpu()) < BF16_STATE_TOL


def test_split_chain_resumes_bit_exactly_inside_a_segment_when_the_gates_forget(kda, cuda_device):
    """The workloads' gates (decay about e^-140 per chunk): every segment boundary's
    two-chunk tail map is exactly zero, so a boundary state is the tail window run
    from zero in both the full run and a run resumed inside the previous segment.
    The resumed run then reproduces the full run bit for bit, outputs, snapshots
    and final states, although its first segment is shorter."""
    dev = cuda_device
    H, d, T = 2, 128, 1 << 18
    data = inputs.gen_prefill([T], H, d, d, 20271)
    n_ord = T // 256
    pool = torch.zeros((n_ord + n_ord, H, d, d), device=dev)
    table = np.arange(n_ord, dtype=np.int32)[None]
    o, fin = run_gpu(kda, dev, data, pool=pool, snap_table=table)
    assert not torch.isnan(o.float()).any() and not torch.isnan(fin).any()
    for p in (100096, 200192):
        tail = {key: data[key][p:] for key in ("q", "k", "v", "alpha", "beta")}
        tail["cu_seqlens"] = torch.tensor([0, T - p], dtype=torch.int32)
        table2 = np.full((1, n_ord), -1, np.int32)
        table2[0, p // 256:] = n_ord + np.arange(n_ord - p // 256)
        o2, fin2 = run_gpu(kda, dev, tail, start_pos=[p], init_slot=[p // 256 - 1], pool=pool,
                           snap_table=table2)
        assert torch.equal(o2, o[p:]), p
        assert torch.equal(fin2, fin), p
        assert torch.equal(pool[n_ord:2 * n_ord - p // 256], pool[p // 256:n_ord]), p


def test_split_and_plain_sequences_in_one_batch(kda, cuda_device):
    """A batch with a split chain beside plain ones: 140,000 tokens (split), a
    3,000-token sequence resumed at position 512 from a pool state, an empty
    sequence, and an empty sequence resumed at 256 from that pool state; 8
    heads, mild decay.  Every output, final state and snapshot against the
    oracle.  The final states start as NaN: an empty sequence's final state is
    its initial state, written even though it has no chunk."""
    dev = cuda_device
    H, d = 8, 128
    lens = [140000, 3000, 0, 0]
    data = inputs.gen_prefill(lens, H, d, d, 20269, decay="mild")
    starts = [0, 512, 0, 256]
    init_slot = [-1, 0, -1, 0]
    n = len(lens)
    init_state = inputs.gen_states(1, H, d, d, 20270, std=0.05)
    n_ord = [(s + L) // 256 for s, L in zip(starts, lens)]
    width = max(n_ord)
    table = np.full((n, width), -1, np.int32)
    slot = 1                                      # slot 0 holds the resumed sequences' initial state
    for i in range(n):
        for m in range(starts[i] // 256, n_ord[i]):
            table[i, m] = slot
            slot += 1
    pool = torch.zeros((slot, H, d, d), device=dev)
    pool[0] = init_state[0].to(dev)
    x = to_dev(data, dev)
    fin = torch.full((n, H, d, d), float("nan"), device=dev)
    o, fin = kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], data["cu_seqlens"].to(dev),
                         total_tokens=int(data["cu_seqlens"][-1]),
                         start_pos=torch.tensor(starts, dtype=torch.int32, device=dev),
                         init_slot=torch.tensor(init_slot, dtype=torch.int32, device=dev), pool=pool,
                         snap_table=torch.from_numpy(table).to(dev), final_state=fin)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    assert torch.equal(fin[2], torch.zeros_like(fin[2]))          # empty, zero start
    assert torch.equal(fin[3], pool[0])                           # empty, resumed: its initial state
    init64 = np.zeros((n, H, d, d))
    init64[1] = init64[3] = init_state[0].double().numpy()
    req = [(i, m) for i in range(n) for m in range(starts[i] // 256, n_ord[i]) if m % 37 == 0 or m == n_ord[i] - 1]
    ref = oracle.run(data["q"], data["k"], data["v"], data["alpha"], data["beta"], data["cu_seqlens"],
                     start_pos=starts, init_state=init64, snap_req=req)
    cu = data["cu_seqlens"].tolist()
    for i in range(n):
        for h in range(H):
            if lens[i]:
                assert rel_rms(o[cu[i]:cu[i + 1], h].float().cpu(), ref["o"][cu[i]:cu[i + 1], h]) < BF16_OUT_TOL, (i, h)
                assert rel_rms(fin[i, h].cpu(), ref["final"][i, h]) < BF16_STATE_TOL, (i, h)
            else:
                assert np.array_equal(fin[i, h].double().cpu().numpy(), ref["final"][i, h]), (i, h)
    for r, (i, m) in enumerate(req):
        for h in range(H):
            assert rel_rms(pool[table[i, m], h].cpu(), ref["snaps"][r, h]) < BF16_STATE_TOL, (i, m, h)


@pytest.mark.parametrize("dtype, d", [(torch.bfloat16, 128), (torch.float32, 128), (torch.bfloat16, 64)])
def test_all_empty_batch_writes_the_initial_states(kda, cuda_device, dtype, d):
    """Three empty sequences (total_tokens = 0) on the tensor-core stages (bf16,
    d = 128) and the SIMT stages (fp32, or d = 64): nothing to compute, but every
    final state is written: zeros without an initial slot, the slot's state when
    resumed."""
    dev = cuda_device
    H = 4
    data = inputs.gen_prefill([0, 0, 0], H, d, d, 20272, dtype=dtype)
    pool = inputs.gen_states(2, H, d, d, 20273, std=0.05).to(dev)
    before = pool.clone()
    o, fin = run_gpu(kda, dev, data, start_pos=[0, 256, 512], init_slot=[-1, 0, 1], pool=pool)
    assert o.shape[0] == 0
    assert torch.equal(fin[0], torch.zeros_like(fin[0]))
    assert torch.equal(fin[1], pool[0]) and torch.equal(fin[2], pool[1])
    assert torch.equal(pool, before)


def test_status_check_times_out_while_the_stream_is_busy(kda, cuda_device):
    """The host watchdog: kda_check_status with a time limit reports
    KDA_ERR_TIMEOUT while a stream still runs (20 back-to-back prefills), leaves
    the status word alone, and the next unlimited check drains cleanly."""
    dev = cuda_device
    data = inputs.gen_prefill([8192] * 4, 32, 128, 128, 20271)
    x = to_dev(data, dev)
    cu = data["cu_seqlens"].to(dev)
    torch.cuda.synchronize()
    for _ in range(20):
        kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], cu)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_check_status(timeout_ms=1)
    assert e.value.status == kda.KDA_ERR_TIMEOUT
    assert kda.kda_check_status() == 0
