"""State transfer by logical id on one GPU ("Kimi K3 Tech Intro", section 2.4:
workers exchange logical prefix ids, not addresses; section 7: the tail of a
transfer is zeroed).

Worker A prefills a prompt, keeping a state every 256 tokens. It exports the
states of the prompt's chained hashes, plus two unknown ids, into a transfer
buffer larger than needed. Worker B, with its own index and a pool numbered
differently, imports them. A prefill on B that resumes from an imported state
must reproduce A's own resumed run bit for bit.
"""
import numpy as np
import pytest
import torch

from hybrid_linear_attention_kda_gb300 import inputs
from hybrid_linear_attention_kda_gb300.prefix_cache import PrefixCache, kda_pcache_unit_hashes

pytestmark = pytest.mark.gpu


def _prefill(kda, dev, table, tokens, plan, pool):
    x = inputs.embed(table, [tokens[plan["start_pos"]:]])
    width = max(1, plan["n_units"])
    snap = np.full((1, width), -1, np.int32)
    snap[0, :plan["n_units"]] = plan["snap_row"]
    dx = {key: x[key].to(dev) for key in ("q", "k", "v", "alpha", "beta")}
    o, fin = kda.prefill(dx["q"], dx["k"], dx["v"], dx["alpha"], dx["beta"], x["cu_seqlens"].to(dev),
                         start_pos=torch.tensor([plan["start_pos"]], dtype=torch.int32, device=dev),
                         init_slot=torch.tensor([plan["init_slot"]], dtype=torch.int32, device=dev),
                         pool=pool, snap_table=torch.from_numpy(snap).to(dev))
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    return o, fin


def test_export_import_by_logical_id(kda, cuda_device):
    dev = cuda_device
    H, d, vocab = 4, 128, 4096
    table = inputs.gen_token_table(vocab, H, d, d, seed=20267)
    rng = np.random.default_rng(3)
    prompt = rng.integers(0, vocab, size=1500).tolist()
    ids = kda_pcache_unit_hashes(prompt)                          # 5 units: 256 .. 1280

    A = PrefixCache(16, match_unit=256, retention_interval=256)
    pool_a = torch.zeros((16, H, d, d), device=dev)
    pa = A.plan_request(prompt)
    _prefill(kda, dev, table, prompt, pa, pool_a)
    A.end_step(True)
    A.release(pa["request_id"])

    unknown = [bytes([7] * 32), bytes([9] * 32)]
    send = ids + unknown
    cap = len(send) + 3
    buf = torch.full((cap, H, d, d), float("nan"), device=dev)
    scratch = torch.empty(cap, dtype=torch.int32, device=dev)
    pos = A.export_states(send, pool_a, buf, scratch)
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    assert list(pos) == [256 * (i + 1) for i in range(len(ids))] + [0, 0]
    for i, lid in enumerate(ids):
        slot, p = A.lookup(lid)
        assert torch.equal(buf[i], pool_a[slot])
    assert torch.count_nonzero(buf[len(ids):]) == 0          # unknown ids and the tail are zeros

    B = PrefixCache(16, slot_base=20, match_unit=256, retention_interval=256)
    pool_b = torch.full((40, H, d, d), float("nan"), device=dev)
    found = [i for i in range(len(send)) if pos[i] > 0]
    taken = B.import_states([send[i] for i in found], [int(pos[i]) for i in found], buf[found].contiguous(),
                            pool_b, torch.empty(len(found), dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert kda.kda_check_status() == 0
    assert all(s >= 20 for s in taken)
    assert B.lookup(ids[0]) == (-1, 0)                        # not matchable before the step ends
    B.end_step(True)
    for i in found:
        slot_b, p_b = B.lookup(send[i])
        slot_a, p_a = A.lookup(send[i])
        assert p_b == p_a and torch.equal(pool_b[slot_b], pool_a[slot_a])
    again = B.import_states(ids[:1], [256], buf[:1].contiguous(), pool_b,
                            torch.empty(1, dtype=torch.int32, device=dev))
    assert list(again) == [-1]                                # already registered: skipped

    # the next turn resumes from the transferred state on B as it does on A
    turn2 = prompt + rng.integers(0, vocab, size=300).tolist()
    pb2 = B.plan_request(turn2)
    pa2 = A.plan_request(turn2)
    assert pb2["start_pos"] == pa2["start_pos"] == 1280
    ob, fb = _prefill(kda, dev, table, turn2, pb2, pool_b)
    oa, fa = _prefill(kda, dev, table, turn2, pa2, pool_a)
    assert torch.equal(ob, oa) and torch.equal(fb, fa)
