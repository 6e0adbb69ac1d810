"""Python binding of the host prefix-cache index (``include/kda_prefix_cache.h``).

Argument marshalling only; the index itself is C++ inside libkda.so.  It decides
which saved KDA state a request resumes from and which of its states to keep
("Kimi K3 Tech Intro", sections 2.2-2.4 and 3).  A plan fills the prefill's
``start_pos``, ``init_slot`` and one ``snap_table`` row.
"""
import ctypes

import numpy as np


class PcacheConfig(ctypes.Structure):
    """Mirror of ``kda_pcache_config``."""
    _fields_ = [("match_unit", ctypes.c_int32), ("admit_on_second_hit", ctypes.c_int32),
                ("retention_interval", ctypes.c_int64), ("slot_base", ctypes.c_int64),
                ("n_slots", ctypes.c_int64)]


class PcachePlan(ctypes.Structure):
    """Mirror of ``kda_pcache_plan``."""
    _fields_ = [("request_id", ctypes.c_int64), ("start_pos", ctypes.c_int64), ("init_slot", ctypes.c_int32),
                ("n_units", ctypes.c_int32), ("n_saved", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class PcacheStats(ctypes.Structure):
    """Mirror of ``kda_pcache_stats``."""
    _fields_ = [(n, ctypes.c_int64) for n in ("entries", "published", "pinned", "free_slots", "seen_units",
                                              "requests", "hits", "misses", "evictions", "dropped")]


def declare(lib):
    """Set the ctypes signatures of the kda_pcache_* entry points."""
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    lib.kda_pcache_create.restype = ctypes.c_int
    lib.kda_pcache_create.argtypes = [P(PcacheConfig), P(vp)]
    lib.kda_pcache_destroy.restype = None
    lib.kda_pcache_destroy.argtypes = [vp]
    lib.kda_pcache_plan_request.restype = ctypes.c_int
    lib.kda_pcache_plan_request.argtypes = [vp, vp, i64, vp, i64, P(PcachePlan)]
    lib.kda_pcache_end_step.restype = ctypes.c_int
    lib.kda_pcache_end_step.argtypes = [vp, i32]
    lib.kda_pcache_release.restype = ctypes.c_int
    lib.kda_pcache_release.argtypes = [vp, i64]
    lib.kda_pcache_get_stats.restype = ctypes.c_int
    lib.kda_pcache_get_stats.argtypes = [vp, P(PcacheStats)]
    lib.kda_pcache_lookup.restype = ctypes.c_int
    lib.kda_pcache_lookup.argtypes = [vp, vp, P(i32), P(i64)]
    lib.kda_pcache_import.restype = ctypes.c_int
    lib.kda_pcache_import.argtypes = [vp, vp, i64, P(i32), P(i32)]
    lib.kda_pcache_unit_hashes.restype = ctypes.c_int
    lib.kda_pcache_unit_hashes.argtypes = [vp, i64, i32, vp, i64]
    lib.kda_state_export.restype = ctypes.c_int
    lib.kda_state_export.argtypes = [vp, vp, i32, i32, vp, i64, i32, i32, i32, vp, vp, vp, vp]
    lib.kda_state_import.restype = ctypes.c_int
    lib.kda_state_import.argtypes = [vp, vp, vp, i32, vp, vp, i64, i32, i32, i32, vp, vp, vp]


def _lib_and_check():
    from . import load, _check
    return load(), _check


def _tokens(tokens):
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    if t.ndim != 1:
        raise ValueError("tokens must be one-dimensional")
    return t


def kda_pcache_unit_hashes(tokens, match_unit=256):
    """Chained hashes (logical ids) of the prompt's full units, as a list of 32-byte strings."""
    lib, check = _lib_and_check()
    t = _tokens(tokens)
    m = len(t) // match_unit
    out = np.zeros(max(1, 32 * m), dtype=np.uint8)
    check(lib.kda_pcache_unit_hashes(t.ctypes.data if len(t) else None, len(t), match_unit,
                                     out.ctypes.data, 32 * m))
    return [bytes(out[32 * n:32 * (n + 1)]) for n in range(m)]


class PrefixCache:
    """One index (``kda_pcache_create``); methods map one-to-one to the C calls."""

    def __init__(self, n_slots, slot_base=0, match_unit=256, retention_interval=0, admit_on_second_hit=False):
        lib, check = _lib_and_check()
        self._lib, self._check = lib, check
        cfg = PcacheConfig(match_unit, 1 if admit_on_second_hit else 0, retention_interval, slot_base, n_slots)
        h = ctypes.c_void_p()
        check(lib.kda_pcache_create(ctypes.byref(cfg), ctypes.byref(h)))
        self._h = h
        self.match_unit = match_unit

    def close(self):
        if self._h:
            self._lib.kda_pcache_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def plan_request(self, tokens, snap_row=None):
        """``kda_pcache_plan_request``.  Returns a dict with request_id,
        start_pos, init_slot, n_units, n_saved and snap_row (an int32 array of
        n_units entries, or the caller's array, filled in place)."""
        t = _tokens(tokens)
        m = len(t) // self.match_unit
        row = np.full(max(1, m), -1, dtype=np.int32) if snap_row is None else snap_row
        if row.dtype != np.int32 or not row.flags["C_CONTIGUOUS"]:
            raise ValueError("snap_row must be a contiguous int32 array")
        out = PcachePlan()
        self._check(self._lib.kda_pcache_plan_request(self._h, t.ctypes.data if len(t) else None, len(t),
                                                      row.ctypes.data, len(row), ctypes.byref(out)))
        return {"request_id": out.request_id, "start_pos": out.start_pos, "init_slot": out.init_slot,
                "n_units": out.n_units, "n_saved": out.n_saved, "snap_row": row[:m] if snap_row is None else row}

    def end_step(self, succeeded=True):
        self._check(self._lib.kda_pcache_end_step(self._h, 1 if succeeded else 0))

    def release(self, request_id):
        self._check(self._lib.kda_pcache_release(self._h, int(request_id)))

    def stats(self):
        s = PcacheStats()
        self._check(self._lib.kda_pcache_get_stats(self._h, ctypes.byref(s)))
        return {n: getattr(s, n) for n, _ in PcacheStats._fields_}

    def lookup(self, logical_id: bytes):
        """(slot, position) of the published state with this logical id, or (-1, 0)."""
        if len(logical_id) != 32:
            raise ValueError("logical ids are 32 bytes")
        buf = ctypes.create_string_buffer(logical_id, 32)
        slot, pos = ctypes.c_int32(), ctypes.c_int64()
        self._check(self._lib.kda_pcache_lookup(self._h, buf, ctypes.byref(slot), ctypes.byref(pos)))
        return slot.value, pos.value

    def export_states(self, ids, pool, dst, slot_scratch, stream=None):
        """``kda_state_export``: the published states of `ids` (32-byte logical
        ids) into dst[0 .. len(ids)), the rest of dst zeroed.  Returns the
        positions (0 where an id was not found)."""
        import torch
        from . import _dev, _dims, _stream_handle
        n = len(ids)
        n_slots, H, d_k, d_v = _dims(pool, "pool", 4)
        cap = _dims(dst, "dst", 4)[0]
        pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v))
        dp = _dev(dst, "dst", torch.float32, (cap, H, d_k, d_v), pool.device)
        sp = _dev(slot_scratch, "slot_scratch", torch.int32, device=pool.device, min_numel=cap)
        buf = ctypes.create_string_buffer(b"".join(ids), max(1, 32 * n))
        pos = np.zeros(max(1, n), dtype=np.int64)
        self._check(self._lib.kda_state_export(self._h, buf, n, cap, pp, n_slots, H, d_k, d_v, dp, sp,
                                               pos.ctypes.data, _stream_handle(stream)))
        return pos[:n]

    def import_states(self, ids, positions, src, pool, slot_scratch, stream=None):
        """``kda_state_import``: register `ids` at `positions` and copy the new
        ones from src into their slots.  Returns the slots taken (-1 = skipped)."""
        import torch
        from . import _dev, _dims, _stream_handle
        n = len(ids)
        n_slots, H, d_k, d_v = _dims(pool, "pool", 4)
        pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v))
        srp = _dev(src, "src", torch.float32, (n, H, d_k, d_v), pool.device)
        sp = _dev(slot_scratch, "slot_scratch", torch.int32, device=pool.device, min_numel=n)
        buf = ctypes.create_string_buffer(b"".join(ids), max(1, 32 * n))
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        if pos.shape != (n,):
            raise ValueError(f"positions must hold one entry per id ({n}), got shape {pos.shape}")
        slots = np.full(max(1, n), -1, dtype=np.int32)
        self._check(self._lib.kda_state_import(self._h, buf, pos.ctypes.data if n else None, n, srp, pp, n_slots,
                                               H, d_k, d_v, sp, slots.ctypes.data, _stream_handle(stream)))
        return slots[:n]

    def import_state(self, logical_id: bytes, pos: int):
        """(slot, is_new) for a state that arrives from elsewhere."""
        if len(logical_id) != 32:
            raise ValueError("logical ids are 32 bytes")
        buf = ctypes.create_string_buffer(logical_id, 32)
        slot, new = ctypes.c_int32(), ctypes.c_int32()
        self._check(self._lib.kda_pcache_import(self._h, buf, int(pos), ctypes.byref(slot), ctypes.byref(new)))
        return slot.value, bool(new.value)
