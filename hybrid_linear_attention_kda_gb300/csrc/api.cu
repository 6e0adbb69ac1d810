// C-ABI entry points of libkda.so: argument checks, the device status word, and
// dispatch to the kernels.  Declarations and the contract live in include/kda.h.
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "chunk_common.cuh"
#include "kda_prefix_cache.h"

namespace {

thread_local char g_last_error[512] = "";

kda_status_t fail(kda_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kda_status_t fail(kda_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kda_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One status word per device, in this library's own device memory.
__device__ uint32_t g_status_word;

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

// Device address of the current device's status word (looked up once per device).
kda_status_t status_ptr(uint32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KDA_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        g_status_ptr[dev] = static_cast<uint32_t*>(p);
    }
    *out = g_status_ptr[dev];
    return KDA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status_t check_dims(int32_t H, int32_t d_k, int32_t d_v, int32_t dtype) {
    if (H <= 0) return fail(KDA_ERR_INVALID_ARG, "n_heads must be >= 1 (got %d)", H);
    if (d_k != d_v || (d_k != 64 && d_k != 128))
        return fail(KDA_ERR_UNSUPPORTED, "d_k == d_v in {64, 128} required (got %d, %d)", d_k, d_v);
    if (dtype != KDA_BF16 && dtype != KDA_FP32)
        return fail(KDA_ERR_UNSUPPORTED, "dtype %d", dtype);
    return KDA_OK;
}

#define KDA_REQUIRE_PTR(p, name)                                                        \
    do {                                                                                \
        if (!(p)) return fail(KDA_ERR_INVALID_ARG, "%s is NULL", name);                 \
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

constexpr int64_t kMaxSeqs = 1 << 20;

kda_status_t validate_prefill(const kda_prefill_args* a) {
    if (!a) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    kda_status_t st = check_dims(a->n_heads, a->d_k, a->d_v, a->dtype);
    if (st != KDA_OK) return st;
    if (a->n_seqs < 0 || a->n_seqs > kMaxSeqs)
        return fail(KDA_ERR_INVALID_ARG, "n_seqs %d outside [0, %lld]", a->n_seqs, (long long)kMaxSeqs);
    if (a->chunk != 64) return fail(KDA_ERR_UNSUPPORTED, "chunk must be 64 (got %d)", a->chunk);
    if (a->snap_interval != 256)
        return fail(KDA_ERR_UNSUPPORTED, "snap_interval must be 256 (got %d)", a->snap_interval);
    if (a->total_tokens < 0 || a->total_tokens > (int64_t)INT32_MAX)
        return fail(KDA_ERR_INVALID_ARG, "total_tokens %lld outside [0, 2^31)", (long long)a->total_tokens);
    if (a->reserved0 != 0) return fail(KDA_ERR_INVALID_ARG, "reserved0 must be 0");
    if (a->n_slots < 0) return fail(KDA_ERR_INVALID_ARG, "n_slots < 0");
    if (a->n_seqs == 0) return KDA_OK;
    KDA_REQUIRE_PTR(a->cu_seqlens, "cu_seqlens");
    if (a->total_tokens > 0) {
        KDA_REQUIRE_PTR(a->q, "q");
        KDA_REQUIRE_PTR(a->k, "k");
        KDA_REQUIRE_PTR(a->v, "v");
        KDA_REQUIRE_PTR(a->alpha, "alpha");
        KDA_REQUIRE_PTR(a->beta, "beta");
        KDA_REQUIRE_PTR(a->o, "o");
    }
    if (a->start_pos && !aligned16(a->start_pos)) return fail(KDA_ERR_INVALID_ARG, "start_pos misaligned");
    if (a->init_slot || a->snap_table) {
        KDA_REQUIRE_PTR(a->pool, "pool (needed by init_slot / snap_table)");
        if (a->n_slots <= 0) return fail(KDA_ERR_INVALID_ARG, "n_slots must be > 0 with a pool");
    }
    if (a->init_slot && !aligned16(a->init_slot)) return fail(KDA_ERR_INVALID_ARG, "init_slot misaligned");
    if (a->snap_table) {
        if (!aligned16(a->snap_table)) return fail(KDA_ERR_INVALID_ARG, "snap_table misaligned");
        if (a->snap_table_stride <= 0)
            return fail(KDA_ERR_INVALID_ARG, "snap_table_stride must be > 0 with a snap_table");
    }
    if (a->final_state && !aligned16(a->final_state))
        return fail(KDA_ERR_INVALID_ARG, "final_state misaligned");
    return KDA_OK;
}

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// bf16 with d = 128 runs the tensor-core stages; fp32 q/k/v and d = 64 the same
// chunk algorithm in fp32 SIMT arithmetic (chunk_simt.cu).
bool use_tensor_cores(const kda_prefill_args* a) { return a->dtype == KDA_BF16 && a->d_k == 128; }

size_t record_bytes(const kda_prefill_args* a) {
    return use_tensor_cores(a) ? (size_t)kda::kRecBytes : kda::simt_record_bytes(a->d_k);
}

// Upper bound on the chunks of a batch: each sequence starts chunk-aligned
// (start_pos is a multiple of snap_interval), so it has at most one partial chunk.
int64_t max_chunks_for(const kda_prefill_args* a) {
    return a->total_tokens / kda::kC + a->n_seqs;
}

// Long sequences in a batch of few chains are split into segments that run in
// parallel (a chain of 16,384 chunks would otherwise keep one SM busy while the
// others idle): when the batch has fewer chains than half the SMs and at least
// two segments' worth of tokens.
bool split_for(const kda_prefill_args* a) {
    if (!use_tensor_cores(a) || a->total_tokens < 2 * kda::kSegTokens) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 1 << 20;                      // unknown: assume splitting pays
    return (int64_t)a->n_seqs * a->n_heads * 2 < sms;
}

// A split sequence of L tokens has at most L / kSegTokens + 2 segments.
int64_t max_segs_for(const kda_prefill_args* a) { return kda::max_segments(a->total_tokens, a->n_seqs); }
int64_t max_scratch_for(const kda_prefill_args* a) { return kda::max_segments(a->total_tokens, a->n_seqs); }

struct WorkspaceLayout {
    size_t chunk_base, exact_count, exact_items, chunk_info, records, seg_info, seg_count, seg_slow, seg_state, total;
    bool split;
};

WorkspaceLayout layout_for(const kda_prefill_args* a) {
    WorkspaceLayout w{};
    if (a->n_seqs == 0) return w;
    size_t off = 0;
    w.chunk_base = off;
    off = round_up(off + sizeof(int32_t) * ((size_t)a->n_seqs + 1), 256);
    w.exact_count = off;
    off = round_up(off + sizeof(uint32_t), 256);
    if (use_tensor_cores(a)) {
        w.exact_items = off;
        off = round_up(off + sizeof(int64_t) * (size_t)max_chunks_for(a) * a->n_heads, 256);
    }
    w.chunk_info = off;
    off = round_up(off + sizeof(int4) * (size_t)max_chunks_for(a), 256);
    w.records = off;
    off += (size_t)max_chunks_for(a) * a->n_heads * record_bytes(a);
    w.split = split_for(a);
    if (w.split) {
        off = round_up(off, 256);
        w.seg_info = off;
        off = round_up(off + sizeof(int4) * (size_t)max_segs_for(a), 256);
        w.seg_count = off;
        off = round_up(off + sizeof(int32_t) * ((size_t)a->n_seqs + 2), 256);
        w.seg_slow = off;
        off = round_up(off + sizeof(int32_t) * (size_t)max_scratch_for(a) * a->n_heads, 256);
        w.seg_state = off;
        off += (size_t)max_scratch_for(a) * a->n_heads * 3 * kda::kD * kda::kD * sizeof(float);
    }
    w.total = round_up(off, 256);
    return w;
}

// Workspace of the path the arguments select (bytes, 256-byte multiple).
size_t workspace_bytes_for(const kda_prefill_args* a) { return layout_for(a).total; }

std::atomic<uint64_t> g_launches{0};

}  // namespace

void kda::note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

kda_status_t kda::record_error(kda_status_t status, const char* message) { return fail(status, "%s", message); }

extern "C" {

uint64_t kda_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }


int32_t kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DEVICE_STATUS: return "KDA_ERR_DEVICE_STATUS";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_NO_MEMORY: return "KDA_ERR_NO_MEMORY";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error(void) { return g_last_error; }

size_t kda_prefill_workspace_size(const kda_prefill_args* a) {
    // the size checks of validate_prefill, without recording an error
    if (!a || a->n_seqs < 0 || a->n_seqs > kMaxSeqs || a->n_heads <= 0) return 0;
    if (a->d_k != a->d_v || (a->d_k != 64 && a->d_k != 128)) return 0;
    if (a->dtype != KDA_BF16 && a->dtype != KDA_FP32) return 0;
    if (a->chunk != kda::kC || a->snap_interval != 256) return 0;
    if (a->total_tokens < 0 || a->total_tokens > (int64_t)INT32_MAX) return 0;
    return workspace_bytes_for(a);
}

}  // extern "C"

namespace {

// Launch the prefill; when marks is non-null, record marks->ev[i] before the
// i-th kernel and one after the last.
struct Marks {
    void* const* ev;
    int32_t n_ev, n_rec;
    const char** names;
};

kda_status_t mark(Marks* m, cudaStream_t s, const char* name) {
    if (!m) return KDA_OK;
    if (m->n_rec >= m->n_ev) return fail(KDA_ERR_INVALID_ARG, "kda_prefill_chunked_events: need more events");
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(m->ev[m->n_rec]), s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if (m->names) m->names[m->n_rec] = name;
    m->n_rec += 1;
    return KDA_OK;
}

kda_status_t prefill_impl(const kda_prefill_args* a, void* stream, Marks* m) {
    kda_status_t st = validate_prefill(a);
    if (st != KDA_OK) return st;
    if (a->n_seqs == 0) return KDA_OK;
    const size_t need = workspace_bytes_for(a);
    if (need > 0 && (!a->workspace || a->workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(a->workspace) & 255u)))
        return fail(KDA_ERR_INVALID_ARG, "workspace must be >= %zu bytes and 256-byte aligned", need);
    uint32_t* status = nullptr;
    st = status_ptr(&status);
    if (st != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
#define KDA_MARK(name)                          \
    do {                                        \
        kda_status_t ms_ = mark(m, s, name);    \
        if (ms_ != KDA_OK) return ms_;          \
    } while (0)
    const WorkspaceLayout w = layout_for(a);
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    kda::ChunkLaunch c;
    c.a = *a;
    c.chunk_base = reinterpret_cast<int32_t*>(ws + w.chunk_base);
    c.chunk_info = reinterpret_cast<int4*>(ws + w.chunk_info);
    c.exact_count = reinterpret_cast<uint32_t*>(ws + w.exact_count);
    c.exact_items = use_tensor_cores(a) ? reinterpret_cast<int64_t*>(ws + w.exact_items) : nullptr;
    c.records = ws + w.records;
    c.max_chunks = max_chunks_for(a);
    c.status = status;
    c.split = w.split ? 1 : 0;
    c.mode = kda::kCarryPlain;
    c.seg_info = w.split ? reinterpret_cast<int4*>(ws + w.seg_info) : nullptr;
    c.seg_count = w.split ? reinterpret_cast<int32_t*>(ws + w.seg_count) : nullptr;
    c.seg_state = w.split ? reinterpret_cast<float*>(ws + w.seg_state) : nullptr;
    c.seg_slow = w.split ? reinterpret_cast<int32_t*>(ws + w.seg_slow) : nullptr;
    c.max_segs = w.split ? max_segs_for(a) : 0;
    KDA_MARK("chunk_meta");
    cudaError_t e = kda::launch_chunk_meta(c, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill meta launch");
    if (w.split) {
        e = kda::launch_segment_meta(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill segment table launch");
    }
    if (!use_tensor_cores(a)) {
        KDA_MARK("simt_local");
        e = kda::launch_simt_local(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill chunk-local (SIMT) launch");
        KDA_MARK("simt_recur");
        e = kda::launch_simt_recur(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill carry (SIMT) launch");
        KDA_MARK("end");
        return KDA_OK;
    }
    KDA_MARK("chunk_local");
    e = kda::launch_chunk_local(c, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill chunk-local launch");
    KDA_MARK("chunk_exact");
    e = kda::launch_chunk_exact(c, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill exact-item launch");
    if (w.split) {
        // the tail windows before the segment boundaries (a head whose windows
        // all forget their start state needs no segment map), the segment maps
        // A (identity start, U~ = 0) and offsets B (zero start), the scan of
        // the segments' start states, then every segment in parallel
        KDA_MARK("chunk_recur_tail");
        c.mode = kda::kCarryTailMap;
        e = kda::launch_chunk_recur(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill segment-tail launch");
        KDA_MARK("chunk_recur_map");
        c.mode = kda::kCarryMap;
        e = kda::launch_chunk_recur(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill segment-map launch");
        KDA_MARK("chunk_recur_offset");
        c.mode = kda::kCarryOffset;
        e = kda::launch_chunk_recur(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill segment-offset launch");
        KDA_MARK("segment_scan");
        e = kda::launch_segment_scan(c, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill segment-scan launch");
        c.mode = kda::kCarryFinal;
    }
    KDA_MARK("chunk_recur");
    e = kda::launch_chunk_recur(c, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill chunk-recurrence launch");
    KDA_MARK("end");
#undef KDA_MARK
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_prefill_chunked(const kda_prefill_args* a, void* stream) {
    return prefill_impl(a, stream, nullptr);
}

kda_status_t kda_prefill_chunked_events(const kda_prefill_args* a, void* stream, void* const* events,
                                        int32_t n_events, int32_t* n_recorded, const char** names) {
    if (n_recorded) *n_recorded = 0;
    if (!events || n_events <= 0) return fail(KDA_ERR_INVALID_ARG, "events array is empty");
    Marks m{events, n_events, 0, names};
    kda_status_t st = prefill_impl(a, stream, &m);
    if (n_recorded) *n_recorded = m.n_rec;
    return st;
}

kda_status_t kda_decode_step(int32_t n_seqs, int32_t n_heads, int32_t d_k, int32_t d_v,
                             int32_t dtype, const void* q, const void* k, const void* v,
                             const float* alpha, const float* beta, float* pool,
                             int64_t n_slots, const int32_t* state_slot, void* o,
                             float scale, void* stream) {
    kda_status_t st = check_dims(n_heads, d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (n_seqs < 0 || n_seqs > kMaxSeqs) return fail(KDA_ERR_INVALID_ARG, "n_seqs %d", n_seqs);
    if (n_slots < 0) return fail(KDA_ERR_INVALID_ARG, "n_slots < 0");
    if (n_seqs == 0) return KDA_OK;
    KDA_REQUIRE_PTR(q, "q");
    KDA_REQUIRE_PTR(k, "k");
    KDA_REQUIRE_PTR(v, "v");
    KDA_REQUIRE_PTR(alpha, "alpha");
    KDA_REQUIRE_PTR(beta, "beta");
    KDA_REQUIRE_PTR(pool, "pool");
    KDA_REQUIRE_PTR(state_slot, "state_slot");
    KDA_REQUIRE_PTR(o, "o");
    if (n_slots == 0) return fail(KDA_ERR_INVALID_ARG, "n_slots must be > 0");
    if ((int64_t)n_seqs * n_heads > (int64_t)INT32_MAX)
        return fail(KDA_ERR_INVALID_ARG, "n_seqs * n_heads too large");
    kda::DecodeLaunch p{n_seqs, n_heads, d_k, dtype, q, k, v, alpha, beta, pool, n_slots,
                        state_slot, o, scale, nullptr};
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_decode(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return KDA_OK;
}

kda_status_t kda_decode_fused(const kda_fused_decode_args* args, void* stream) {
    if (!args) return fail(KDA_ERR_INVALID_ARG, "args is NULL");
    const kda_fused_decode_args& a = *args;
    kda_status_t st = check_dims(a.n_heads, a.d, a.d, KDA_BF16);
    if (st != KDA_OK) return st;
    if (a.conv_size != 4) return fail(KDA_ERR_UNSUPPORTED, "conv_size must be 4 (got %d)", a.conv_size);
    if (a.reserved0 != 0) return fail(KDA_ERR_INVALID_ARG, "reserved0 must be 0");
    if (!(a.norm_eps >= 0.f)) return fail(KDA_ERR_INVALID_ARG, "norm_eps must be >= 0");
    if (a.n_seqs < 0 || a.n_seqs > kMaxSeqs) return fail(KDA_ERR_INVALID_ARG, "n_seqs %d", a.n_seqs);
    if (a.n_slots < 0) return fail(KDA_ERR_INVALID_ARG, "n_slots < 0");
    if (a.n_seqs == 0) return KDA_OK;
    if ((int64_t)a.n_seqs * a.n_heads > (int64_t)INT32_MAX) return fail(KDA_ERR_INVALID_ARG, "n_seqs * n_heads too large");
    KDA_REQUIRE_PTR(a.xq, "xq");
    KDA_REQUIRE_PTR(a.xk, "xk");
    KDA_REQUIRE_PTR(a.xv, "xv");
    KDA_REQUIRE_PTR(a.a, "a");
    KDA_REQUIRE_PTR(a.b, "b");
    KDA_REQUIRE_PTR(a.g, "g");
    KDA_REQUIRE_PTR(a.conv_w, "conv_w");
    KDA_REQUIRE_PTR(a.norm_w, "norm_w");
    KDA_REQUIRE_PTR(a.pool, "pool");
    KDA_REQUIRE_PTR(a.conv_state, "conv_state");
    KDA_REQUIRE_PTR(a.state_slot, "state_slot");
    KDA_REQUIRE_PTR(a.y, "y");
    if (a.n_slots == 0) return fail(KDA_ERR_INVALID_ARG, "n_slots must be > 0");
    kda::FusedDecodeLaunch L{a, nullptr};
    st = status_ptr(&L.status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_fused_decode(L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused decode launch");
    return KDA_OK;
}

static kda_status_t check_spec(int32_t n_seqs, int32_t n_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t dtype, int64_t n_slots) {
    kda_status_t st = check_dims(n_heads, d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (n_tokens < 1 || n_tokens > 16) return fail(KDA_ERR_UNSUPPORTED, "n_tokens must be in [1, 16] (got %d)", n_tokens);
    if (n_seqs < 0 || n_seqs > kMaxSeqs) return fail(KDA_ERR_INVALID_ARG, "n_seqs %d", n_seqs);
    if (n_slots < 0) return fail(KDA_ERR_INVALID_ARG, "n_slots < 0");
    if ((int64_t)n_seqs * n_heads > (int64_t)INT32_MAX) return fail(KDA_ERR_INVALID_ARG, "n_seqs * n_heads too large");
    return KDA_OK;
}

kda_status_t kda_decode_verify(int32_t n_seqs, int32_t n_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t dtype, const void* q, const void* k, const void* v,
                               const float* alpha, const float* beta, const float* pool,
                               int64_t n_slots, const int32_t* state_slot, void* o, float* u,
                               float scale, void* stream) {
    kda_status_t st = check_spec(n_seqs, n_tokens, n_heads, d_k, d_v, dtype, n_slots);
    if (st != KDA_OK) return st;
    if (n_seqs == 0) return KDA_OK;
    KDA_REQUIRE_PTR(q, "q");
    KDA_REQUIRE_PTR(k, "k");
    KDA_REQUIRE_PTR(v, "v");
    KDA_REQUIRE_PTR(alpha, "alpha");
    KDA_REQUIRE_PTR(beta, "beta");
    KDA_REQUIRE_PTR(pool, "pool");
    KDA_REQUIRE_PTR(state_slot, "state_slot");
    KDA_REQUIRE_PTR(o, "o");
    KDA_REQUIRE_PTR(u, "u");
    if (n_slots == 0) return fail(KDA_ERR_INVALID_ARG, "n_slots must be > 0");
    kda::SpecLaunch p{n_seqs, n_tokens, n_heads, d_k, dtype, q, k, v, alpha, beta, const_cast<float*>(pool),
                      n_slots, state_slot, o, u, nullptr, scale, nullptr};
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_verify(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "verify launch");
    return KDA_OK;
}

kda_status_t kda_decode_commit(int32_t n_seqs, int32_t n_tokens, int32_t n_heads, int32_t d_k, int32_t d_v,
                               int32_t dtype, const void* k, const float* alpha, const float* u,
                               const int32_t* n_accept, float* pool, int64_t n_slots,
                               const int32_t* state_slot, void* stream) {
    kda_status_t st = check_spec(n_seqs, n_tokens, n_heads, d_k, d_v, dtype, n_slots);
    if (st != KDA_OK) return st;
    if (n_seqs == 0) return KDA_OK;
    KDA_REQUIRE_PTR(k, "k");
    KDA_REQUIRE_PTR(alpha, "alpha");
    KDA_REQUIRE_PTR(u, "u");
    KDA_REQUIRE_PTR(n_accept, "n_accept");
    KDA_REQUIRE_PTR(pool, "pool");
    KDA_REQUIRE_PTR(state_slot, "state_slot");
    if (n_slots == 0) return fail(KDA_ERR_INVALID_ARG, "n_slots must be > 0");
    kda::SpecLaunch p{n_seqs, n_tokens, n_heads, d_k, dtype, nullptr, k, nullptr, alpha, nullptr, pool,
                      n_slots, state_slot, nullptr, const_cast<float*>(u), n_accept, 1.f, nullptr};
    st = status_ptr(&p.status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_commit(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "commit launch");
    return KDA_OK;
}

static kda_status_t check_copy(const void* a, const void* b, int64_t n_slots, const int32_t* slots,
                               int32_t n, int32_t H, int32_t d_k, int32_t d_v) {
    kda_status_t st = check_dims(H, d_k, d_v, KDA_FP32);
    if (st != KDA_OK) return st;
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "n < 0");
    if (n_slots < 0) return fail(KDA_ERR_INVALID_ARG, "n_slots < 0");
    if (n == 0) return KDA_OK;
    KDA_REQUIRE_PTR(a, "pool/src");
    KDA_REQUIRE_PTR(b, "dst/pool");
    KDA_REQUIRE_PTR(slots, "slots");
    return KDA_OK;
}

kda_status_t kda_snapshot_gather(const float* pool, int64_t n_slots, const int32_t* slots,
                                 int32_t n, int32_t n_heads, int32_t d_k, int32_t d_v,
                                 float* dst, void* stream) {
    kda_status_t st = check_copy(pool, dst, n_slots, slots, n, n_heads, d_k, d_v);
    if (st != KDA_OK || n == 0) return st;
    uint32_t* status = nullptr;
    st = status_ptr(&status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_gather(pool, n_slots, slots, n, (int64_t)n_heads * d_k * d_v, dst,
                                       status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    return KDA_OK;
}

kda_status_t kda_snapshot_restore(const float* src, float* pool, int64_t n_slots,
                                  const int32_t* slots, int32_t n, int32_t n_heads, int32_t d_k,
                                  int32_t d_v, void* stream) {
    kda_status_t st = check_copy(src, pool, n_slots, slots, n, n_heads, d_k, d_v);
    if (st != KDA_OK || n == 0) return st;
    uint32_t* status = nullptr;
    st = status_ptr(&status);
    if (st != KDA_OK) return st;
    cudaError_t e = kda::launch_restore(src, pool, n_slots, slots, n, (int64_t)n_heads * d_k * d_v,
                                        status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "restore launch");
    return KDA_OK;
}

kda_status_t kda_state_export(const kda_pcache* pc, const uint8_t* ids, int32_t n, int32_t capacity,
                              const float* pool, int64_t n_slots, int32_t n_heads, int32_t d_k, int32_t d_v,
                              float* dst, int32_t* slot_scratch, int64_t* pos_out, void* stream) {
    if (!pc) return fail(KDA_ERR_INVALID_ARG, "kda_state_export: pc is NULL");
    if (n < 0 || capacity < n) return fail(KDA_ERR_INVALID_ARG, "kda_state_export: need 0 <= n <= capacity");
    if (n > 0 && !ids) return fail(KDA_ERR_INVALID_ARG, "kda_state_export: ids is NULL");
    kda_status_t st = check_copy(pool, dst, n_slots, slot_scratch, capacity, n_heads, d_k, d_v);
    if (st != KDA_OK || capacity == 0) return st;
    std::vector<int32_t> slots((size_t)capacity, -1);      // the tail stays -1: zeroed by the gather
    for (int32_t i = 0; i < n; ++i) {
        int32_t slot = -1;
        int64_t pos = 0;
        st = kda_pcache_lookup(pc, ids + 32 * (size_t)i, &slot, &pos);
        if (st != KDA_OK) return st;
        if (slot >= 0 && (int64_t)slot >= n_slots) slot = -1;  // outside this pool: treated as absent
        slots[(size_t)i] = slot;
        if (pos_out) pos_out[i] = slot >= 0 ? pos : 0;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(slot_scratch, slots.data(), sizeof(int32_t) * (size_t)capacity,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "slot list copy");
    return kda_snapshot_gather(pool, n_slots, slot_scratch, capacity, n_heads, d_k, d_v, dst, stream);
}

kda_status_t kda_state_import(kda_pcache* pc, const uint8_t* ids, const int64_t* pos, int32_t n,
                              const float* src, float* pool, int64_t n_slots, int32_t n_heads, int32_t d_k,
                              int32_t d_v, int32_t* slot_scratch, int32_t* slots_out, void* stream) {
    if (!pc) return fail(KDA_ERR_INVALID_ARG, "kda_state_import: pc is NULL");
    if (n < 0) return fail(KDA_ERR_INVALID_ARG, "kda_state_import: n < 0");
    if (n > 0 && (!ids || !pos)) return fail(KDA_ERR_INVALID_ARG, "kda_state_import: ids or pos is NULL");
    kda_status_t st = check_copy(src, pool, n_slots, slot_scratch, n, n_heads, d_k, d_v);
    if (st != KDA_OK || n == 0) return st;
    std::vector<int32_t> slots((size_t)n, -1);
    for (int32_t i = 0; i < n; ++i) {
        int32_t slot = -1, is_new = 0;
        st = kda_pcache_import(pc, ids + 32 * (size_t)i, pos[i], &slot, &is_new);
        if (st != KDA_OK) return st;
        if (is_new && (int64_t)slot < n_slots) slots[(size_t)i] = slot;
        if (slots_out) slots_out[i] = slots[(size_t)i];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(slot_scratch, slots.data(), sizeof(int32_t) * (size_t)n,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "slot list copy");
    return kda_snapshot_restore(src, pool, n_slots, slot_scratch, n, n_heads, d_k, d_v, stream);
}

kda_status_t kda_check_status(void* stream, int32_t timeout_ms, uint32_t* bits_out) {
    if (bits_out) *bits_out = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) {
        cudaEventDestroy(ev);
        return cuda_fail(e, "cudaEventRecord");
    }
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        e = cudaEventQuery(ev);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) {
            cudaEventDestroy(ev);
            return cuda_fail(e, "stream drain");
        }
        if (timeout_ms > 0 &&
            std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms)) {
            cudaEventDestroy(ev);
            return fail(KDA_ERR_TIMEOUT, "stream did not drain within %d ms", timeout_ms);
        }
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    cudaEventDestroy(ev);
    uint32_t bits = 0;
    e = cudaMemcpyFromSymbol(&bits, g_status_word, sizeof bits);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (bits) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
        if (bits_out) *bits_out = bits;
        return fail(KDA_ERR_DEVICE_STATUS, "device status bits 0x%x", bits);
    }
    return KDA_OK;
}

}  // extern "C"
