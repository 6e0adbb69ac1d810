"""The library's C++ prefix-cache index against the policy oracle, on the host.

The index needs no GPU.  Every decision must equal the oracle's: the resume
point, the snap_table row, the evictions and the counters.  The inputs are
seeded request streams shaped like a serving workload: families of prompts
sharing a system prefix, multi-turn continuations, repeats, failed steps and
late releases.
"""
import random

import numpy as np
import pytest

from hybrid_linear_attention_kda_gb300 import KdaError, KDA_ERR_INVALID_ARG
from hybrid_linear_attention_kda_gb300.prefix_cache import PrefixCache, kda_pcache_unit_hashes
from oracle.prefix_cache import PrefixCacheIndex, block_hashes


@pytest.mark.parametrize("unit", list(range(1, 40)) + [64, 256])
def test_unit_hashes_match_sha256(unit):
    """Messages of 32 + 4 * unit bytes cover every padding case of SHA-256."""
    rng = random.Random(unit)
    t = [rng.randrange(-2 ** 31, 2 ** 31) for _ in range(unit * 3 + 1)]
    assert kda_pcache_unit_hashes(t, unit) == block_hashes(t, unit)


def test_unit_hashes_short_prompt():
    assert kda_pcache_unit_hashes([1, 2, 3], 256) == []
    assert kda_pcache_unit_hashes([], 256) == []


def _stream(rng, n_req, n_families, unit):
    """(tokens, step_end, succeeded, release_lag) per request."""
    fams = [[rng.randrange(0, 163840) for _ in range(rng.randrange(0, 12) * unit + rng.randrange(0, unit))]
            for _ in range(n_families)]
    history = []
    out = []
    for _ in range(n_req):
        r = rng.random()
        if history and r < 0.2:                     # multi-turn: extend an earlier prompt
            base = rng.choice(history)
            toks = base + [rng.randrange(0, 163840) for _ in range(rng.randrange(1, 3 * unit))]
        elif history and r < 0.3:                   # exact repeat
            toks = list(rng.choice(history))
        else:                                       # family prefix + own question
            toks = list(rng.choice(fams)) + [rng.randrange(0, 163840) for _ in range(rng.randrange(1, 4 * unit))]
        history.append(toks)
        out.append((toks, rng.random() < 0.4, rng.random() > 0.1, rng.randrange(0, 4)))
    return out


@pytest.mark.parametrize("interval,second_hit,n_slots,seed", [
    (0, True, 24, 1),
    (0, False, 24, 2),
    (256, False, 40, 3),
    (1024, True, 12, 4),
    (512, True, 6, 5),
    (0, True, 3, 6),
    (256, True, 200, 7),
])
def test_index_matches_oracle_on_request_streams(interval, second_hit, n_slots, seed):
    unit = 256
    rng = random.Random(seed)
    ref = PrefixCacheIndex(unit=unit, interval=interval, second_hit=second_hit, slot_base=5, n_slots=n_slots)
    pc = PrefixCache(n_slots, slot_base=5, match_unit=unit, retention_interval=interval,
                     admit_on_second_hit=second_hit)
    live = []          # (release at request index, request id)
    hits = 0
    for i, (toks, end, ok, lag) in enumerate(_stream(rng, 220, 5, unit)):
        a = ref.plan(toks)
        b = pc.plan_request(toks)
        assert b["request_id"] == a["request_id"]
        assert (b["start_pos"], b["init_slot"]) == (a["start_pos"], a["init_slot"]), i
        assert list(b["snap_row"]) == a["snap_row"], i
        assert b["n_units"] == a["n_blocks"]
        assert b["n_saved"] == sum(s >= 0 for s in a["snap_row"])
        hits += a["start_pos"] > 0
        live.append((i + lag, a["request_id"]))
        if end:
            ref.end_step(ok)
            pc.end_step(ok)
        for due, rid in [x for x in live if x[0] <= i]:
            ref.release(rid)
            pc.release(rid)
        live = [x for x in live if x[0] > i]
        s = pc.stats()
        assert (s["hits"], s["misses"], s["evictions"], s["dropped"]) == \
            (ref.hits, ref.misses, ref.evictions, ref.dropped), i
        assert s["entries"] == len(ref.entries)
        assert s["free_slots"] == len(ref.free)
        assert s["seen_units"] == len(ref.seen)
        assert s["published"] == sum(e.published for e in ref.entries.values())
        assert s["pinned"] == sum(e.published and e.pins > 0 for e in ref.entries.values())
    assert hits > 10                     # the stream exercised reuse
    if n_slots <= 12:
        assert ref.evictions > 0 or ref.dropped > 0


def test_lookup_and_import_match_oracle():
    rng = random.Random(11)
    ref = PrefixCacheIndex(interval=256, n_slots=4)
    pc = PrefixCache(4, retention_interval=256)
    t = [rng.randrange(0, 1000) for _ in range(700)]
    ids = kda_pcache_unit_hashes(t)
    ref.plan(t)
    pc.plan_request(t)
    assert pc.lookup(ids[0]) == ref.lookup(ids[0]) == (-1, 0)          # not published yet
    ref.end_step()
    pc.end_step()
    assert pc.lookup(ids[1]) == ref.lookup(ids[1]) == (1, 512)
    other = bytes(range(32))
    assert pc.import_state(other, 4096) == ref.import_state(other, 4096) == (2, True)
    assert pc.import_state(other, 4096) == ref.import_state(other, 4096) == (-1, False)
    assert pc.lookup(other) == (-1, 0)
    pc.end_step()
    ref.end_step()
    assert pc.lookup(other) == ref.lookup(other) == (2, 4096)
    # a full pool evicts the least recently used published state for an import
    more = bytes(reversed(range(32)))
    ref.import_state(bytes(32), 256)
    pc.import_state(bytes(32), 256)
    assert pc.import_state(more, 512) == ref.import_state(more, 512)
    assert pc.stats()["evictions"] == ref.evictions == 1


def test_argument_errors_leave_the_index_unchanged():
    pc = PrefixCache(4, retention_interval=256)
    before = pc.stats()
    with pytest.raises(KdaError) as e:
        pc.plan_request([])
    assert e.value.status == KDA_ERR_INVALID_ARG
    with pytest.raises(KdaError):
        pc.plan_request(list(range(600)), snap_row=np.zeros(1, dtype=np.int32))    # two units, room for one
    with pytest.raises(KdaError):
        pc.release(12345)
    with pytest.raises(KdaError):
        pc.import_state(bytes(32), 100)
    assert pc.stats() == before


@pytest.mark.parametrize("cfg", [
    dict(match_unit=0), dict(retention_interval=100), dict(retention_interval=-256),
    dict(slot_base=-1), dict(n_slots=-1), dict(slot_base=2 ** 31 - 2, n_slots=4),
])
def test_bad_configurations(cfg):
    args = dict(n_slots=4)
    args.update(cfg)
    n = args.pop("n_slots")
    with pytest.raises(KdaError) as e:
        PrefixCache(n, **args)
    assert e.value.status == KDA_ERR_INVALID_ARG


def test_long_prompt_plan_is_fast():
    """One 1M-token prompt: 4096 units hashed and planned on the host."""
    import time
    rng = np.random.default_rng(0)
    t = rng.integers(0, 163840, size=1 << 20, dtype=np.int32)
    pc = PrefixCache(64, retention_interval=32768)
    t0 = time.perf_counter()
    p = pc.plan_request(t)
    dt = time.perf_counter() - t0
    assert p["n_units"] == 4096 and p["n_saved"] == 32
    assert dt < 5.0


def test_state_transfer_argument_errors():
    """Export/import reject bad arguments on the host, before any copy."""
    pc = PrefixCache(4, retention_interval=256)
    fake = 0x10000          # never dereferenced: every call below fails first
    ids = bytes(64)
    lib = pc._lib
    assert lib.kda_state_export(None, ids, 2, 2, fake, 4, 2, 64, 64, fake, fake, None, None) == KDA_ERR_INVALID_ARG
    assert lib.kda_state_export(pc._h, ids, 3, 2, fake, 4, 2, 64, 64, fake, fake, None, None) == KDA_ERR_INVALID_ARG
    assert lib.kda_state_export(pc._h, None, 2, 2, fake, 4, 2, 64, 64, fake, fake, None, None) == KDA_ERR_INVALID_ARG
    from hybrid_linear_attention_kda_gb300 import KDA_ERR_UNSUPPORTED
    assert lib.kda_state_export(pc._h, ids, 2, 2, fake, 4, 2, 96, 96, fake, fake, None, None) == KDA_ERR_UNSUPPORTED
    pos = np.array([256, 100], dtype=np.int64)          # the second position is not a multiple of 256
    st = lib.kda_state_import(pc._h, ids, pos.ctypes.data, 2, fake, fake, 4, 2, 64, 64, fake, None, None)
    assert st == KDA_ERR_INVALID_ARG
    assert pc.stats()["entries"] == 1                   # the first id was registered before the error
    pc.end_step(False)                                   # the caller discards it
    assert pc.stats()["entries"] == 0
