"""Pins of the prefix-cache policy oracle against what the pages fix.

"Kimi K3 Tech Intro" (tim-wang blog):
* section 2.1 worked example: two requests share 4800 and 4900 tokens.  With
  matching on the 4096-token physical block they reuse 4096 tokens and recompute
  704 and 804.
* section 2.2: with a 256-token match unit they reuse the last multiple of 256.
* section 2.4: chained hashes, so equal last units under different prefixes do
  not collide; a state is reused only in the step after the one that wrote it.
* section 3.1: checkpoints every 32K tokens plus the prompt boundary, or only the
  prompt boundary when the interval is 0.
* section 3.2: a prefix is not cached on its first use; on its second use the
  state at the shared boundary is cached; the third use reuses it.
"""
import json
import os
import random

import pytest

import oracle
from oracle.prefix_cache import PrefixCacheIndex, block_hashes

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _tokens(rng, n):
    return [rng.randrange(0, 163840) for _ in range(n)]


def _saved_positions(plan, unit):
    return [unit * (o + 1) for o, s in enumerate(plan["snap_row"]) if s >= 0]


@pytest.mark.parametrize("unit", [4096, 256])
def test_worked_example_4800_4900(unit):
    """The index run on the section 2.1 example.  A first request keeps a state
    at every unit.  Two later requests share 4800 and 4900 tokens with it."""
    with open(os.path.join(GOLDEN, "prefix_match_example.json")) as f:
        g = json.load(f)
    rng = random.Random(7)
    base = _tokens(rng, 6000)
    idx = PrefixCacheIndex(unit=unit, interval=unit, n_slots=64)
    idx.plan(base)
    idx.end_step()
    reused = []
    for shared in g["shared_prefix_tokens"]:
        req = base[:shared] + _tokens(rng, 300)
        req[shared] = base[shared] + 1 if shared < len(base) else 0      # diverge right after the shared part
        plan = idx.plan(req)
        reused.append(plan["start_pos"])
        assert plan["init_slot"] >= 0
    if unit == g["physical_block"]:
        assert reused == g["reused_with_physical_block"]
        assert [s - r for s, r in zip(g["shared_prefix_tokens"], reused)] == g["recomputed_with_physical_block"]
    else:
        assert unit == g["match_unit"]
        assert reused == [oracle.reusable_prefix(s, 256) for s in g["shared_prefix_tokens"]] == [4608, 4864]


def test_chained_hash_separates_equal_tails():
    rng = random.Random(1)
    u1a, u1b, u2 = _tokens(rng, 256), _tokens(rng, 256), _tokens(rng, 256)
    ha, hb = block_hashes(u1a + u2), block_hashes(u1b + u2)
    assert ha[0] != hb[0] and ha[1] != hb[1]
    # the same last unit under different prefixes is not a match
    idx = PrefixCacheIndex(interval=256, n_slots=8)
    idx.plan(u1a + u2 + [5])
    idx.end_step()
    assert idx.plan(u1b + u2 + [5])["start_pos"] == 0
    # and the same prefix is
    assert idx.plan(u1a + u2 + [6])["start_pos"] == 512


def test_block_hashes_cover_full_units_only():
    rng = random.Random(2)
    t = _tokens(rng, 1000)
    h = block_hashes(t)
    assert len(h) == 3
    assert block_hashes(t[:768]) == h
    assert block_hashes(t[:767]) == h[:2]
    assert block_hashes(t[:255]) == []


@pytest.mark.parametrize("interval,expected", [
    (32768, [32768, 65536, 98304, 99840]),
    (0, [99840]),
])
def test_interval_retention(interval, expected):
    """Section 3.1's figure: a 100,000-token prompt."""
    rng = random.Random(3)
    idx = PrefixCacheIndex(interval=interval, n_slots=16)
    plan = idx.plan(_tokens(rng, 100000))
    assert _saved_positions(plan, 256) == expected
    assert plan["start_pos"] == 0 and plan["init_slot"] == -1


def test_second_hit_admission_three_requests():
    """Section 3.2: [system prompt][tools][question A / B / C]."""
    rng = random.Random(4)
    shared = _tokens(rng, 3000)
    reqs = [shared + _tokens(rng, 700 + 100 * i) for i in range(3)]
    idx = PrefixCacheIndex(interval=0, second_hit=True, n_slots=16)
    p1 = idx.plan(reqs[0])
    idx.end_step()
    assert p1["start_pos"] == 0
    assert _saved_positions(p1, 256) == [(len(reqs[0]) // 256) * 256]     # prompt boundary only
    p2 = idx.plan(reqs[1])
    idx.end_step()
    assert p2["start_pos"] == 0                                          # nothing cached for the prefix yet
    boundary = (3000 // 256) * 256
    assert _saved_positions(p2, 256) == [boundary, (len(reqs[1]) // 256) * 256]
    p3 = idx.plan(reqs[2])
    assert p3["start_pos"] == boundary
    assert p3["init_slot"] == p2["snap_row"][boundary // 256 - 1]
    # without second-hit admission the shared boundary is never kept
    idx = PrefixCacheIndex(interval=0, second_hit=False, n_slots=16)
    for r in reqs:
        p = idx.plan(r)
        idx.end_step()
    assert p["start_pos"] == 0


def test_reuse_waits_for_the_next_step():
    rng = random.Random(5)
    t = _tokens(rng, 1024 + 17)
    idx = PrefixCacheIndex(interval=256, n_slots=16)
    a = idx.plan(t)
    b = idx.plan(t)                         # same step: a's states are not written yet
    assert b["start_pos"] == 0 and b["init_slot"] == -1
    assert all(s == -1 for s in b["snap_row"])      # a registered them; b does not duplicate
    idx.end_step()
    c = idx.plan(t)
    assert c["start_pos"] == 1024 and c["init_slot"] == a["snap_row"][3]


def test_failed_step_discards_its_states():
    rng = random.Random(6)
    t = _tokens(rng, 600)
    idx = PrefixCacheIndex(interval=256, n_slots=4)
    a = idx.plan(t)
    assert _saved_positions(a, 256) == [256, 512]
    idx.end_step(succeeded=False)
    assert idx.free == [0, 1, 2, 3]
    assert idx.plan(t)["start_pos"] == 0


def test_match_leaves_one_token():
    rng = random.Random(8)
    t = _tokens(rng, 768)
    idx = PrefixCacheIndex(interval=256, n_slots=8)
    idx.plan(t)
    idx.end_step()
    p = idx.plan(t)                          # the whole prompt is cached: redo its last unit
    assert p["start_pos"] == 512
    assert all(s == -1 for s in p["snap_row"])      # 768 is already kept


def test_lru_eviction_and_pins():
    rng = random.Random(9)
    idx = PrefixCacheIndex(interval=0, n_slots=2, slot_base=10)
    ps = [_tokens(rng, 300) for _ in range(3)]
    a = idx.plan(ps[0] + [1])
    b = idx.plan(ps[1] + [1])
    assert (a["snap_row"], b["snap_row"]) == ([10], [11])
    idx.end_step()
    hit = idx.plan(ps[0] + [2])              # pins ps[0]'s state and makes it the most recent
    assert hit["start_pos"] == 256 and hit["init_slot"] == 10
    c = idx.plan(ps[2] + [1])                # evicts ps[1] (least recently used, unpinned)
    assert c["snap_row"] == [11] and idx.evictions == 1
    idx.end_step()
    d = idx.plan(_tokens(rng, 300))          # ps[0] pinned, ps[2] free to go
    assert d["snap_row"] == [11]
    idx.end_step()
    e = idx.plan(_tokens(rng, 300))          # ps[0] still pinned, the last entry is recent but not pinned
    assert e["snap_row"] == [11]
    idx.release(hit["request_id"])
    idx.end_step()
    f = idx.plan(_tokens(rng, 300))          # now ps[0] (last used before e's entry) goes
    assert f["snap_row"] == [10]


def test_no_slot_means_no_state():
    rng = random.Random(10)
    idx = PrefixCacheIndex(interval=256, n_slots=1)
    p = idx.plan(_tokens(rng, 800))
    assert _saved_positions(p, 256) == [256]          # the others find no free or evictable slot
    assert idx.dropped == 2


def test_bad_configuration():
    with pytest.raises(ValueError):
        PrefixCacheIndex(unit=256, interval=300)
    with pytest.raises(ValueError):
        PrefixCacheIndex(unit=0)
    with pytest.raises(ValueError):
        PrefixCacheIndex().plan([])
