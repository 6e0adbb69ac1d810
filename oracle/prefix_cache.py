"""Prefix-cache index for recurrent KDA states (test infrastructure).

TEST INFRASTRUCTURE: only ``tests/`` may use this module.  It is the plain
statement of the policy that the library's C++ index implements.  It shares no
code with that index.  The block hash here is ``hashlib.sha256``; the index
carries its own SHA-256.

What it follows ("Kimi K3 Tech Intro", tim-wang blog):

* section 2.2: prefixes are matched in units of 256 tokens, independently of the
  4096-token physical block.
* section 2.4, chained hash row: every full unit n of a prompt has the hash
      h_n = H(h_{n-1} || tokens of unit n),    h_0 = 32 zero bytes.
  A hash of the last unit alone would let different prefixes collide.
  Here H = SHA-256, and the tokens are 32-bit little-endian integers.
* section 2.3: a request that matches a saved state starts from it without
  writing it.  The prefill reads the shared snapshot as its initial state and
  writes only its own outputs.
* section 2.4, same-step reuse row: a state registered in one step becomes
  matchable only in the next step, after the copy that writes it has finished.
* section 3.1: interval retention keeps one state every ``interval`` tokens plus
  the state at the prompt boundary.  ``interval = 0`` keeps the prompt boundary
  only.
* section 3.2: Marconi-style admission.  A prefix seen for the first time keeps
  only its prompt-boundary state.  A request whose prefix was seen before also
  keeps the state at the boundary of the shared part.  A later request reuses
  that state.

Readings where the pages are silent:

* The prompt boundary is the last multiple of the unit that is <= the prompt
  length, because states exist only at unit boundaries.
* A match leaves at least one prompt token to compute, so that the request
  produces its next-token output.  The matched unit n therefore satisfies
  n * unit <= L - 1.
* The shared-prefix boundary is the deepest full unit whose chained hash some
  earlier request produced.
* The index owns a fixed range of pool slots.  A new state takes the lowest free
  slot.  When none is free it evicts the least recently used published,
  unpinned entry, breaking ties by the lower slot.  A state that finds no slot
  is not saved.
* A request that matched an entry pins it until the caller releases the
  request.  A pinned entry is never evicted.
* A step that failed discards the states it registered and frees their slots.
"""
import hashlib
import struct

ZERO_HASH = bytes(32)


def block_hashes(tokens, unit=256):
    """Chained hashes h_1..h_m of the m = len(tokens) // unit full units."""
    out = []
    h = ZERO_HASH
    for n in range(len(tokens) // unit):
        blk = tokens[n * unit:(n + 1) * unit]
        h = hashlib.sha256(h + struct.pack(f"<{unit}i", *blk)).digest()
        out.append(h)
    return out


class _Entry:
    __slots__ = ("slot", "pos", "last_use", "pins", "published")

    def __init__(self, slot, pos, last_use):
        self.slot = slot
        self.pos = pos
        self.last_use = last_use
        self.pins = 0
        self.published = False


class PrefixCacheIndex:
    """The index's decisions, one request at a time, in plain Python."""

    def __init__(self, unit=256, interval=0, second_hit=False, slot_base=0, n_slots=0):
        if unit <= 0 or interval < 0 or interval % unit != 0 or n_slots < 0 or slot_base < 0:
            raise ValueError("bad configuration")
        self.unit = unit
        self.interval = interval
        self.second_hit = second_hit
        self.free = list(range(slot_base, slot_base + n_slots))   # kept sorted
        self.entries = {}        # hash -> _Entry
        self.seen = set()        # every chained hash any planned request produced
        self.pending = []        # hashes registered in the current step
        self.clock = 0
        self.next_id = 0
        self.pinned_by = {}      # request id -> hash it pinned (or None)
        self.hits = self.misses = self.evictions = self.dropped = 0

    def _take_slot(self):
        if self.free:
            return self.free.pop(0)
        victims = [(e.last_use, e.slot, h) for h, e in self.entries.items() if e.published and e.pins == 0]
        if not victims:
            return None
        _, slot, h = min(victims)
        del self.entries[h]
        self.evictions += 1
        return slot

    def plan(self, tokens):
        """Plan one request's prefill.  Returns a dict with the request id,
        start_pos, init_slot and snap_row (slot per absolute ordinal p/unit - 1
        for p = unit .. m*unit, -1 where nothing is saved)."""
        L = len(tokens)
        if L <= 0:
            raise ValueError("empty prompt")
        U = self.unit
        self.clock += 1
        hashes = block_hashes(tokens, U)
        m = len(hashes)
        rid = self.next_id
        self.next_id += 1

        # deepest published state that leaves at least one token to compute
        start_pos, init_slot, pinned = 0, -1, None
        for n in range((L - 1) // U, 0, -1):
            e = self.entries.get(hashes[n - 1])
            if e is not None and e.published:
                e.pins += 1
                e.last_use = self.clock
                start_pos, init_slot, pinned = n * U, e.slot, hashes[n - 1]
                break
        if pinned is None:
            self.misses += 1
        else:
            self.hits += 1
        self.pinned_by[rid] = pinned

        # positions whose states this request keeps
        keep = set()
        if m >= 1:
            keep.add(m * U)                                    # prompt boundary
        if self.interval > 0:
            keep.update(range(self.interval, m * U + 1, self.interval))
        if self.second_hit:
            shared = 0
            for n in range(m, 0, -1):
                if hashes[n - 1] in self.seen:
                    shared = n
                    break
            if shared > 0:
                keep.add(shared * U)
        self.seen.update(hashes)

        snap_row = [-1] * m
        for p in sorted(x for x in keep if x > start_pos):
            h = hashes[p // U - 1]
            if h in self.entries:            # published or registered by another request
                continue
            slot = self._take_slot()
            if slot is None:
                self.dropped += 1
                continue
            self.entries[h] = _Entry(slot, p, self.clock)
            self.pending.append(h)
            snap_row[p // U - 1] = slot
        return {"request_id": rid, "start_pos": start_pos, "init_slot": init_slot, "snap_row": snap_row,
                "n_blocks": m}

    def end_step(self, succeeded=True):
        """Publish (or, after a failed step, discard) the states registered
        since the previous call."""
        for h in self.pending:
            e = self.entries.get(h)
            if e is None:
                continue
            if succeeded:
                e.published = True
            else:
                del self.entries[h]
                self.free.append(e.slot)
        self.free.sort()
        self.pending = []

    def release(self, rid):
        """The request no longer reads its matched state."""
        h = self.pinned_by.pop(rid)
        if h is not None and h in self.entries:
            self.entries[h].pins -= 1

    def lookup(self, h):
        """Published entry with chained hash (logical id) h: (slot, position), or (-1, 0)."""
        e = self.entries.get(h)
        if e is not None and e.published:
            return e.slot, e.pos
        return -1, 0

    def import_state(self, h, pos):
        """Register a state that arrives from elsewhere under logical id h at
        position pos.  Returns (slot, is_new): a new pending slot, or -1 when h is
        already registered or no slot can be had."""
        if pos < 1 or pos % self.unit != 0:
            raise ValueError("bad position")
        if h in self.entries:
            return -1, False
        self.clock += 1
        slot = self._take_slot()
        if slot is None:
            self.dropped += 1
            return -1, False
        self.entries[h] = _Entry(slot, pos, self.clock)
        self.pending.append(h)
        return slot, True
