// Host prefix-cache index for saved KDA states: which saved state a request
// resumes from, and which of its own states it keeps.  The policy follows
// "Kimi K3 Tech Intro" (tim-wang blog), sections 2.2-2.4 and 3.1-3.2.  The
// contract and the readings where the pages are silent are in
// include/kda_prefix_cache.h.
//
// Data structures (all host memory, one lock per index):
//   entries     chained hash -> {slot, position, last use, pins, published}
//   evictable   ordered (last use, slot) of published, unpinned entries; the
//               first element is the LRU victim
//   free        ordered free slots (lowest first)
//   seen        every chained hash an earlier request produced (second-hit
//               admission)
//   pending     hashes registered since the last end_step
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

#include "kda_prefix_cache.h"

namespace kda {
kda_status_t record_error(kda_status_t status, const char* message);
}

namespace {

// ------------------------------------------------------------------ SHA-256
// FIPS 180-4, section 6.2.  The round constants are the first 32 bits of the
// fractional parts of the cube roots of the first 64 primes, and the initial
// hash value the same for the square roots of the first 8 primes (section
// 4.2.2 and 5.3.3).  They are derived here from that definition with exact
// integer roots: floor(frac(p^(1/e)) * 2^32) = floor(root_e(p * 2^(32 e))) mod 2^32.
struct Sha256Consts {
    uint32_t k[64];
    uint32_t h0[8];
    Sha256Consts() {
        uint32_t primes[64];
        int n = 0;
        for (uint32_t c = 2; n < 64; ++c) {
            bool prime = true;
            for (uint32_t d = 2; d * d <= c; ++d)
                if (c % d == 0) {
                    prime = false;
                    break;
                }
            if (prime) primes[n++] = c;
        }
        for (int i = 0; i < 64; ++i) k[i] = frac_root(primes[i], 3);
        for (int i = 0; i < 8; ++i) h0[i] = frac_root(primes[i], 2);
    }
    // largest x with x^e <= p * 2^(32 e), reduced mod 2^32
    static uint32_t frac_root(uint32_t p, int e) {
        using u128 = unsigned __int128;
        const u128 target = (u128)p << (32 * e);
        uint64_t lo = 0, hi = (uint64_t)1 << 40;          // p < 2^9: the root is below 2^38
        while (lo < hi) {
            const uint64_t mid = lo + (hi - lo + 1) / 2;
            u128 pw = 1;
            for (int j = 0; j < e; ++j) pw *= (u128)mid;
            if (pw <= target) lo = mid;
            else hi = mid - 1;
        }
        return (uint32_t)(lo & 0xFFFFFFFFu);
    }
};

const Sha256Consts& sha_consts() {
    static const Sha256Consts c;
    return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

class Sha256 {
public:
    Sha256() : k_(sha_consts()) { std::memcpy(h_, k_.h0, sizeof h_); }
    void update(const uint8_t* data, size_t len) {
        total_ += len;
        while (len > 0) {
            const size_t take = len < 64 - fill_ ? len : 64 - fill_;
            std::memcpy(buf_ + fill_, data, take);
            fill_ += take;
            data += take;
            len -= take;
            if (fill_ == 64) {
                block(buf_);
                fill_ = 0;
            }
        }
    }
    void finish(uint8_t out[32]) {
        // padding (section 5.1.1): a 1 bit, zeros, then the message length in bits, big-endian
        const uint64_t bits = (uint64_t)total_ * 8u;
        uint8_t pad[72] = {0x80};
        const size_t zeros = (fill_ < 56) ? 56 - fill_ : 120 - fill_;
        for (int i = 0; i < 8; ++i) pad[zeros + i] = (uint8_t)(bits >> (56 - 8 * i));
        update(pad, zeros + 8);
        for (int i = 0; i < 8; ++i)
            for (int j = 0; j < 4; ++j) out[4 * i + j] = (uint8_t)(h_[i] >> (24 - 8 * j));
    }

private:
    void block(const uint8_t* m) {
        uint32_t w[64];
        for (int t = 0; t < 16; ++t)
            w[t] = ((uint32_t)m[4 * t] << 24) | ((uint32_t)m[4 * t + 1] << 16) | ((uint32_t)m[4 * t + 2] << 8) |
                   (uint32_t)m[4 * t + 3];
        for (int t = 16; t < 64; ++t) {
            const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
            const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
            w[t] = w[t - 16] + s0 + w[t - 7] + s1;
        }
        uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6], h = h_[7];
        for (int t = 0; t < 64; ++t) {
            const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
            const uint32_t ch = (e & f) ^ (~e & g);
            const uint32_t t1 = h + S1 + ch + k_.k[t] + w[t];
            const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
            const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
            const uint32_t t2 = S0 + maj;
            h = g;
            g = f;
            f = e;
            e = d + t1;
            d = c;
            c = b;
            b = a;
            a = t1 + t2;
        }
        h_[0] += a;
        h_[1] += b;
        h_[2] += c;
        h_[3] += d;
        h_[4] += e;
        h_[5] += f;
        h_[6] += g;
        h_[7] += h;
    }

    const Sha256Consts& k_;
    uint32_t h_[8];
    uint8_t buf_[64];
    size_t fill_ = 0;
    uint64_t total_ = 0;
};

struct Hash32 {
    uint8_t b[32];
    bool operator==(const Hash32& o) const { return std::memcmp(b, o.b, 32) == 0; }
};
struct Hash32Hasher {
    size_t operator()(const Hash32& h) const {
        uint64_t x;
        std::memcpy(&x, h.b, 8);
        return (size_t)x;
    }
};

// h_n = SHA-256(h_{n-1} || unit n as int32 little-endian), h_0 = 0 (32 bytes)
void unit_hashes(const int32_t* tokens, int64_t n_units, int32_t unit, Hash32* out) {
    std::vector<uint8_t> bytes((size_t)unit * 4);
    Hash32 prev;
    std::memset(prev.b, 0, 32);
    for (int64_t n = 0; n < n_units; ++n) {
        const int32_t* t = tokens + n * unit;
        for (int32_t i = 0; i < unit; ++i) {
            const uint32_t v = (uint32_t)t[i];
            bytes[4 * i] = (uint8_t)v;
            bytes[4 * i + 1] = (uint8_t)(v >> 8);
            bytes[4 * i + 2] = (uint8_t)(v >> 16);
            bytes[4 * i + 3] = (uint8_t)(v >> 24);
        }
        Sha256 s;
        s.update(prev.b, 32);
        s.update(bytes.data(), bytes.size());
        s.finish(out[n].b);
        prev = out[n];
    }
}

struct Entry {
    int64_t slot;
    int64_t pos;
    int64_t last_use;
    int32_t pins;
    bool published;
};

}  // namespace

struct kda_pcache {
    kda_pcache_config cfg;
    mutable std::mutex mu;
    std::unordered_map<Hash32, Entry, Hash32Hasher> entries;
    std::unordered_set<Hash32, Hash32Hasher> seen;
    std::vector<Hash32> pending;
    std::set<int64_t> free_slots;
    std::set<std::pair<int64_t, int64_t>> evictable;   // (last_use, slot)
    std::vector<Hash32> slot_owner;                      // by slot - slot_base
    std::unordered_map<int64_t, std::pair<bool, Hash32>> pinned_by;   // request -> (pinned?, hash)
    int64_t clock = 0, next_id = 0;
    int64_t hits = 0, misses = 0, evictions = 0, dropped = 0, n_pinned = 0, n_published = 0;

    // lowest free slot, else the LRU published unpinned entry's slot, else -1
    int64_t take_slot() {
        if (!free_slots.empty()) {
            const int64_t s = *free_slots.begin();
            free_slots.erase(free_slots.begin());
            return s;
        }
        if (evictable.empty()) return -1;
        const int64_t s = evictable.begin()->second;
        evictable.erase(evictable.begin());
        entries.erase(slot_owner[(size_t)(s - cfg.slot_base)]);
        n_published -= 1;
        evictions += 1;
        return s;
    }
    void add_pending(const Hash32& h, int64_t slot, int64_t pos) {
        entries.emplace(h, Entry{slot, pos, clock, 0, false});
        slot_owner[(size_t)(slot - cfg.slot_base)] = h;
        pending.push_back(h);
    }
    void pin(Entry& e) {
        if (e.pins == 0) {
            evictable.erase({e.last_use, e.slot});
            n_pinned += 1;
        }
        e.pins += 1;
        e.last_use = clock;
    }
    void unpin(Entry& e) {
        e.pins -= 1;
        if (e.pins == 0) {
            n_pinned -= 1;
            evictable.insert({e.last_use, e.slot});
        }
    }
};

extern "C" {

kda_status_t kda_pcache_create(const kda_pcache_config* cfg, kda_pcache** out) {
    if (!cfg || !out) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_create: cfg or out is NULL");
    if (cfg->match_unit < 1) return kda::record_error(KDA_ERR_INVALID_ARG, "match_unit must be >= 1");
    if (cfg->retention_interval < 0 || cfg->retention_interval % cfg->match_unit != 0)
        return kda::record_error(KDA_ERR_INVALID_ARG, "retention_interval must be 0 or a positive multiple of match_unit");
    if (cfg->slot_base < 0 || cfg->n_slots < 0 || cfg->slot_base + cfg->n_slots > ((int64_t)1 << 31))
        return kda::record_error(KDA_ERR_INVALID_ARG, "slot range outside [0, 2^31)");
    try {
        kda_pcache* pc = new kda_pcache;
        pc->cfg = *cfg;
        pc->slot_owner.resize((size_t)cfg->n_slots);
        for (int64_t s = 0; s < cfg->n_slots; ++s) pc->free_slots.insert(pc->free_slots.end(), cfg->slot_base + s);
        *out = pc;
        return KDA_OK;
    } catch (const std::bad_alloc&) {
        return kda::record_error(KDA_ERR_NO_MEMORY, "kda_pcache_create: host allocation failed");
    }
}

void kda_pcache_destroy(kda_pcache* pc) { delete pc; }

kda_status_t kda_pcache_plan_request(kda_pcache* pc, const int32_t* tokens, int64_t n_tokens, int32_t* snap_row,
                                     int64_t snap_row_len, kda_pcache_plan* out) {
    if (!pc || !tokens || !out)
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_plan_request: pc, tokens or out is NULL");
    if (n_tokens < 1) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_plan_request: empty prompt");
    const int64_t U = pc->cfg.match_unit;
    const int64_t m = n_tokens / U;
    if (m > ((int64_t)1 << 30)) return kda::record_error(KDA_ERR_INVALID_ARG, "prompt too long");
    if (m > 0 && (!snap_row || snap_row_len < m))
        return kda::record_error(KDA_ERR_INVALID_ARG, "snap_row shorter than the prompt's units");
    try {
        std::vector<Hash32> h((size_t)m);
        unit_hashes(tokens, m, (int32_t)U, h.data());
        std::vector<int64_t> keep;
        keep.reserve(8);
        std::lock_guard<std::mutex> lock(pc->mu);
        // reserve everything that can throw before the first change of state
        pc->pending.reserve(pc->pending.size() + (size_t)m + 2);
        pc->seen.reserve(pc->seen.size() + (size_t)m);
        pc->entries.reserve(pc->entries.size() + (size_t)m + 2);
        pc->pinned_by.reserve(pc->pinned_by.size() + 1);

        pc->clock += 1;
        const int64_t rid = pc->next_id++;
        // deepest published state with start_pos <= L - 1
        int64_t start_pos = 0, init_slot = -1;
        std::pair<bool, Hash32> pinned{false, Hash32{}};
        for (int64_t n = (n_tokens - 1) / U; n >= 1; --n) {
            auto it = pc->entries.find(h[(size_t)(n - 1)]);
            if (it != pc->entries.end() && it->second.published) {
                pc->pin(it->second);
                start_pos = n * U;
                init_slot = it->second.slot;
                pinned = {true, it->first};
                break;
            }
        }
        if (pinned.first) pc->hits += 1;
        else pc->misses += 1;
        pc->pinned_by.emplace(rid, pinned);

        // positions whose states this request keeps
        if (m >= 1) keep.push_back(m * U);
        if (pc->cfg.retention_interval > 0)
            for (int64_t p = pc->cfg.retention_interval; p <= m * U; p += pc->cfg.retention_interval) keep.push_back(p);
        if (pc->cfg.admit_on_second_hit) {
            for (int64_t n = m; n >= 1; --n)
                if (pc->seen.count(h[(size_t)(n - 1)])) {
                    keep.push_back(n * U);
                    break;
                }
        }
        for (const Hash32& x : h) pc->seen.insert(x);
        std::sort(keep.begin(), keep.end());
        keep.erase(std::unique(keep.begin(), keep.end()), keep.end());

        for (int64_t o = 0; o < m; ++o) snap_row[o] = -1;
        int32_t n_saved = 0;
        for (int64_t p : keep) {
            if (p <= start_pos) continue;
            const Hash32& x = h[(size_t)(p / U - 1)];
            if (pc->entries.count(x)) continue;       // published, or registered by another request
            const int64_t slot = pc->take_slot();
            if (slot < 0) {
                pc->dropped += 1;
                continue;
            }
            pc->add_pending(x, slot, p);
            snap_row[p / U - 1] = (int32_t)slot;
            n_saved += 1;
        }
        out->request_id = rid;
        out->start_pos = start_pos;
        out->init_slot = (int32_t)init_slot;
        out->n_units = (int32_t)m;
        out->n_saved = n_saved;
        out->reserved = 0;
        return KDA_OK;
    } catch (const std::bad_alloc&) {
        return kda::record_error(KDA_ERR_NO_MEMORY, "kda_pcache_plan_request: host allocation failed");
    }
}

kda_status_t kda_pcache_end_step(kda_pcache* pc, int32_t succeeded) {
    if (!pc) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_end_step: pc is NULL");
    std::lock_guard<std::mutex> lock(pc->mu);
    for (const Hash32& x : pc->pending) {
        auto it = pc->entries.find(x);
        if (it == pc->entries.end() || it->second.published) continue;
        Entry& e = it->second;
        if (succeeded) {
            e.published = true;
            pc->n_published += 1;
            if (e.pins == 0) pc->evictable.insert({e.last_use, e.slot});
        } else {
            pc->free_slots.insert(e.slot);
            pc->entries.erase(it);
        }
    }
    pc->pending.clear();
    return KDA_OK;
}

kda_status_t kda_pcache_release(kda_pcache* pc, int64_t request_id) {
    if (!pc) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_release: pc is NULL");
    std::lock_guard<std::mutex> lock(pc->mu);
    auto it = pc->pinned_by.find(request_id);
    if (it == pc->pinned_by.end())
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_release: unknown or released request id");
    if (it->second.first) {
        auto e = pc->entries.find(it->second.second);
        if (e != pc->entries.end()) pc->unpin(e->second);
    }
    pc->pinned_by.erase(it);
    return KDA_OK;
}

kda_status_t kda_pcache_get_stats(const kda_pcache* pc, kda_pcache_stats* out) {
    if (!pc || !out) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_get_stats: NULL argument");
    std::lock_guard<std::mutex> lock(pc->mu);
    out->entries = (int64_t)pc->entries.size();
    out->published = pc->n_published;
    out->pinned = pc->n_pinned;
    out->free_slots = (int64_t)pc->free_slots.size();
    out->seen_units = (int64_t)pc->seen.size();
    out->requests = pc->next_id;
    out->hits = pc->hits;
    out->misses = pc->misses;
    out->evictions = pc->evictions;
    out->dropped = pc->dropped;
    return KDA_OK;
}

kda_status_t kda_pcache_lookup(const kda_pcache* pc, const uint8_t* hash, int32_t* slot, int64_t* pos) {
    if (!pc || !hash || !slot || !pos) return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_lookup: NULL argument");
    Hash32 x;
    std::memcpy(x.b, hash, 32);
    std::lock_guard<std::mutex> lock(pc->mu);
    auto it = pc->entries.find(x);
    if (it != pc->entries.end() && it->second.published) {
        *slot = (int32_t)it->second.slot;
        *pos = it->second.pos;
    } else {
        *slot = -1;
        *pos = 0;
    }
    return KDA_OK;
}

kda_status_t kda_pcache_import(kda_pcache* pc, const uint8_t* hash, int64_t pos, int32_t* slot, int32_t* is_new) {
    if (!pc || !hash || !slot || !is_new)
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_import: NULL argument");
    if (pos < 1 || pos % pc->cfg.match_unit != 0)
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_import: pos must be a positive multiple of match_unit");
    Hash32 x;
    std::memcpy(x.b, hash, 32);
    try {
        std::lock_guard<std::mutex> lock(pc->mu);
        pc->pending.reserve(pc->pending.size() + 1);
        pc->entries.reserve(pc->entries.size() + 1);
        *slot = -1;
        *is_new = 0;
        if (pc->entries.count(x)) return KDA_OK;
        pc->clock += 1;
        const int64_t s = pc->take_slot();
        if (s < 0) {
            pc->dropped += 1;
            return KDA_OK;
        }
        pc->add_pending(x, s, pos);
        *slot = (int32_t)s;
        *is_new = 1;
        return KDA_OK;
    } catch (const std::bad_alloc&) {
        return kda::record_error(KDA_ERR_NO_MEMORY, "kda_pcache_import: host allocation failed");
    }
}

kda_status_t kda_pcache_unit_hashes(const int32_t* tokens, int64_t n_tokens, int32_t match_unit, uint8_t* out,
                                    int64_t out_len) {
    if (n_tokens < 0 || match_unit < 1 || (n_tokens > 0 && !tokens))
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_unit_hashes: bad tokens or match_unit");
    const int64_t m = n_tokens / match_unit;
    if (m > 0 && (!out || out_len < 32 * m))
        return kda::record_error(KDA_ERR_INVALID_ARG, "kda_pcache_unit_hashes: out shorter than 32 bytes per unit");
    try {
        std::vector<Hash32> h((size_t)m);
        unit_hashes(tokens, m, match_unit, h.data());
        for (int64_t n = 0; n < m; ++n) std::memcpy(out + 32 * n, h[(size_t)n].b, 32);
        return KDA_OK;
    } catch (const std::bad_alloc&) {
        return kda::record_error(KDA_ERR_NO_MEMORY, "kda_pcache_unit_hashes: host allocation failed");
    }
}

}  // extern "C"
