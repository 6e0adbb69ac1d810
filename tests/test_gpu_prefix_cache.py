"""The prefix-cache index driving the chunked prefill on the GPU.

A seeded serving stream runs for three steps.  Requests share system-prompt
prefixes and continue earlier turns.  Token ids map to layer inputs through a
fixed table, so equal prefixes give equal inputs.  Each step runs as follows:
  * the C++ index plans every request (start_pos, init_slot, snap_table row);
  * one kda_prefill_chunked call runs the packed suffixes of the step;
  * the step is published, then its requests are released.
Every request is then checked against the float64 oracle run on its whole
prompt from the zero state:
  * outputs of the computed suffix;
  * final state;
  * each state the step saved.
The saved states are read right after their step, before a later step may
evict and reuse the slot.  The bf16 tolerances are those of the other prefill
tests.
"""
import random

import numpy as np
import pytest
import torch

import oracle
from hybrid_linear_attention_kda_gb300 import inputs
from hybrid_linear_attention_kda_gb300.prefix_cache import PrefixCache
from _helpers import BF16_OUT_TOL, BF16_STATE_TOL, rel_rms

pytestmark = pytest.mark.gpu

U = 256


def _stream(seed, vocab):
    rng = random.Random(seed)
    fams = [[rng.randrange(vocab) for _ in range(n)] for n in (1500, 2600)]
    steps = []
    done = []
    for step in range(3):
        reqs = []
        for i in range(5):
            if step > 0 and i == 0:                   # next turn of an earlier conversation
                base = done[rng.randrange(len(done))]
                reqs.append(base + [rng.randrange(vocab) for _ in range(rng.randrange(50, 600))])
            else:
                reqs.append(list(fams[i % 2]) + [rng.randrange(vocab) for _ in range(rng.randrange(1, 900))])
        steps.append(reqs)
        done.extend(reqs)
    return steps


@pytest.mark.parametrize("interval,second_hit,n_slots", [(0, True, 48), (512, False, 10)])
def test_prefix_cache_drives_prefill(kda, cuda_device, interval, second_hit, n_slots):
    """n_slots = 10 makes the index evict and reuse slots between steps."""
    dev = cuda_device
    H, d, vocab = 4, 128, 4096
    table = inputs.gen_token_table(vocab, H, d, d, seed=20265, decay="mild")
    pc = PrefixCache(n_slots, match_unit=U, retention_interval=interval, admit_on_second_hit=second_hit)
    pool = torch.zeros((n_slots, H, d, d), device=dev)

    checks = []       # (full tokens, start, o suffix, final, {ordinal: state})
    for reqs in _stream(7 + interval, vocab):
        plans = [pc.plan_request(t) for t in reqs]
        suffixes = [t[p["start_pos"]:] for t, p in zip(reqs, plans)]
        x = inputs.embed(table, suffixes)
        width = max(1, max(p["n_units"] for p in plans))
        snap = np.full((len(reqs), width), -1, np.int32)
        for i, p in enumerate(plans):
            snap[i, :p["n_units"]] = p["snap_row"]
        dx = {key: x[key].to(dev) for key in ("q", "k", "v", "alpha", "beta")}
        o, fin = kda.prefill(dx["q"], dx["k"], dx["v"], dx["alpha"], dx["beta"], x["cu_seqlens"].to(dev),
                             start_pos=torch.tensor([p["start_pos"] for p in plans], dtype=torch.int32, device=dev),
                             init_slot=torch.tensor([p["init_slot"] for p in plans], dtype=torch.int32, device=dev),
                             pool=pool, snap_table=torch.from_numpy(snap).to(dev))
        torch.cuda.synchronize()
        status = kda.kda_check_status()
        assert status == 0
        pc.end_step(status == 0)
        for p in plans:
            pc.release(p["request_id"])
        cu = x["cu_seqlens"].tolist()
        for i, (t, p) in enumerate(zip(reqs, plans)):
            saved = {o_: pool[s].cpu().clone() for o_, s in enumerate(p["snap_row"]) if s >= 0}
            checks.append((t, p["start_pos"], o[cu[i]:cu[i + 1]].float().cpu(), fin[i].cpu(), saved))

    st = pc.stats()
    resumed = [c for c in checks if c[1] > 0]
    assert st["hits"] == len(resumed) and len(resumed) >= 4
    assert any(c[4] for c in checks)
    if n_slots < 16:
        assert st["evictions"] > 0

    full = inputs.embed(table, [c[0] for c in checks])
    snap_req = [(i, o_) for i, c in enumerate(checks) for o_ in sorted(c[4])]
    ref = oracle.run(full["q"], full["k"], full["v"], full["alpha"], full["beta"], full["cu_seqlens"],
                     snap_req=snap_req)
    cu = full["cu_seqlens"].tolist()
    j = 0
    for i, (t, start, o_s, f, saved) in enumerate(checks):
        ref_o = ref["o"][cu[i] + start:cu[i + 1]]
        for h in range(H):
            assert rel_rms(o_s[:, h], ref_o[:, h]) < BF16_OUT_TOL, (i, h)
            assert rel_rms(f[h], ref["final"][i, h]) < BF16_STATE_TOL, (i, h)
        for o_ in sorted(saved):
            for h in range(H):
                assert rel_rms(saved[o_][h], ref["snaps"][j, h]) < BF16_STATE_TOL, (i, o_, h)
            j += 1
    assert j == len(snap_req)
