// kvq_api.cu -- the C ABI of libkvq (include/kvq.h): argument checks, the host handle,
// the host mirror of the lengths and the launches.  No device memory is allocated here.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "kvq_internal.cuh"

struct kvq_cache {
    kvq_cache_desc desc;
    uint8_t *k_mem, *v_mem;
    int32_t *state;  // [len B][ticket][error][pad]
    size_t k_code_bytes, v_code_bytes;
    int32_t *h_len;  // host mirror
    int device;
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_pair(int32_t tk, int32_t tv) {
    return (kvq::is_base_type(tk) && kvq::is_base_type(tv)) || kvq::is_ext_pair(tk, tv);
}

kvq_status check_desc(const kvq_cache_desc *d) {
    if (!d) return KVQ_ERR_INVALID_ARG;
    if (d->batch < 1 || d->n_kv_heads < 1 || d->capacity < 1) return KVQ_ERR_INVALID_ARG;
    if (d->capacity % kvq::kTileRows != 0) return KVQ_ERR_INVALID_ARG;
    if (!valid_pair(d->type_k, d->type_v)) return KVQ_ERR_UNSUPPORTED;
    if (d->head_dim != 128 && d->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

// bytes of the codes region and of the whole plane for one type; false on overflow
bool plane_bytes(const kvq_cache_desc *d, int type, size_t *codes, size_t *total) {
    const unsigned long long tiles = static_cast<unsigned long long>(d->batch) * d->n_kv_heads * (d->capacity / 16);
    const unsigned long long ns = d->head_dim / kvq::kSlice;
    const unsigned long long per_tile_codes = ns * kvq::code_tile_bytes(type);
    const unsigned long long per_tile_scales = ns * kvq::scale_tile_bytes(type);
    if (tiles > (~0ull) / (per_tile_codes + per_tile_scales)) return false;
    *codes = static_cast<size_t>(tiles * per_tile_codes);
    *total = static_cast<size_t>(tiles * (per_tile_codes + per_tile_scales));
    return true;
}

size_t state_bytes_for(int32_t batch) { return ((static_cast<size_t>(batch) + 2) * 4 + 15) / 16 * 16; }

kvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// kvq_set_verify_path: 0 automatic, 1 register-operand MMA, 2 tensor-memory MMA
std::atomic<int> g_verify_path{0};

// Draft verify on the 128-row tensor-memory tile: base types, more than one group of 8 rows
// and at most 128 rows per (sequence, KV head), unless the caller chose a path.
// Automatic choice: the 128-row tile costs about the same for any row count, the groups of 8
// about one single-query pass each.  Measured crossovers: near 6 groups (48 rows) on the
// 65,536-position hybrid layers (D = 256) and near 4 groups (32 rows) on the 131,072-position
// dense layers (D = 128), so the tile is taken from 49 rows at D = 256 and from 33 at D = 128.
int verify_tc_min_rows(int head_dim) { return (head_dim == 2 * kvq::kSlice ? 6 : 4) * kvq::kMaxRowsPerGroup + 1; }

bool verify_on_tc(const kvq_cache *c, int32_t n_q_heads, int32_t n_q) {
    const int rows = n_q * (n_q_heads / c->desc.n_kv_heads);
    if (rows > kvq::kVerifyTileRows || !kvq::is_base_type(c->desc.type_k) || !kvq::is_base_type(c->desc.type_v))
        return false;
    const int path = g_verify_path.load(std::memory_order_relaxed);
    return path == 2 || (path == 0 && rows >= verify_tc_min_rows(c->desc.head_dim));
}

int auto_splits(const kvq_cache *c, int n_q_heads, int *out, int n_q = 1) {
    int ctas = 0, sms = 0;
    if (kvq::decode_occupancy(c->desc.type_k, c->desc.type_v, c->desc.head_dim, &ctas, &sms) != cudaSuccess)
        return -1;
    if (ctas < 1) ctas = 1;
    const int G = n_q_heads / c->desc.n_kv_heads;
    // the tensor-memory verify holds every query row of a (sequence, KV head) in one CTA, one
    // CTA per SM (its shared and tensor memory)
    const bool tc = n_q > 1 && verify_on_tc(c, n_q_heads, n_q);
    if (tc) ctas = 1;
    const int QG = tc ? 1 : (n_q * G + kvq::kMaxRowsPerGroup - 1) / kvq::kMaxRowsPerGroup;
    const long long units = static_cast<long long>(c->desc.batch) * c->desc.n_kv_heads * QG;
    // one full wave of CTAs, rounded down so that a unit count that does not divide the
    // wave does not spill into a partial second one; with several sequences (lengths may
    // differ) about four waves, rounded up, so that short sequences leave no SM idle (16
    // sequences of 8K-64K on the 48-layer shape: 64.6 / 68.2 / 69.4 / 69.7 / 64.3 % of the
    // copy peak with 2 / 3 / 4 / 6 / 8 waves)
    const long long target = static_cast<long long>(sms) * ctas * (c->desc.batch > 1 ? 4 : 1);
    long long s = c->desc.batch > 1 ? (target + units - 1) / units : target / units;
    const long long max_tiles = c->desc.capacity / kvq::kTileRows;
    if (s > max_tiles) s = max_tiles;
    if (s > kvq::kMaxSplits) s = kvq::kMaxSplits;
    if (s < 1) s = 1;
    *out = static_cast<int>(s);
    return 0;
}

kvq_status check_q_heads(const kvq_cache *c, int32_t n_q_heads, int32_t n_q = 1) {
    if (n_q_heads < 1 || n_q_heads % c->desc.n_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
    const long long G = n_q_heads / c->desc.n_kv_heads;
    const long long QG = (n_q * G + kvq::kMaxRowsPerGroup - 1) / kvq::kMaxRowsPerGroup;
    if (static_cast<long long>(c->desc.batch) * QG > 65535) return KVQ_ERR_UNSUPPORTED;
    if (c->desc.n_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

// kvq_set_wait_limit (0: the default of about two seconds)
std::atomic<long long> g_wait_cycles{kvq::kWaitCycles};

// kvq_set_launch_stamps: each decode launch takes the next slot of the caller's buffer
std::mutex g_stamp_mu;
unsigned long long *g_stamp_buf = nullptr;
int g_stamp_slots = 0, g_stamp_ctas = 0, g_stamp_next = 0;

void take_stamp_slot(kvq::DecodeParams &p) {
    std::lock_guard<std::mutex> lock(g_stamp_mu);
    if (!g_stamp_buf || g_stamp_slots < 1) return;
    p.stamps = g_stamp_buf + static_cast<size_t>(g_stamp_next) * g_stamp_ctas * 2;
    p.stamp_ctas = g_stamp_ctas;
    g_stamp_next = (g_stamp_next + 1) % g_stamp_slots;
}

kvq::DecodeParams base_params(const kvq_cache *c, const float *q, int32_t n_q_heads, float scale, int32_t splits,
                              int32_t n_q = 1) {
    kvq::DecodeParams p{};
    p.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
    p.k_codes = c->k_mem;
    p.k_scales = c->desc.type_k == KVQ_F16 ? nullptr : c->k_mem + c->k_code_bytes;
    p.v_codes = c->v_mem;
    p.v_scales = c->desc.type_v == KVQ_F16 ? nullptr : c->v_mem + c->v_code_bytes;
    p.len = c->state;
    p.err = c->state + c->desc.batch + 1;
    p.q = q;
    p.B = c->desc.batch;
    p.Hkv = c->desc.n_kv_heads;
    p.Hq = n_q_heads;
    p.G = n_q_heads / c->desc.n_kv_heads;
    p.QG = (n_q * p.G + kvq::kMaxRowsPerGroup - 1) / kvq::kMaxRowsPerGroup;
    p.n_q = n_q;
    p.D = c->desc.head_dim;
    p.cap_tiles = c->desc.capacity / kvq::kTileRows;
    p.n_splits = splits;
    p.part_stride = splits;
    p.part_base = 0;
    p.scale_log2 = scale * 1.44269504088896340736f;
    return p;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t counters, counters1, part_m, part_l, part_o, grp_m, grp_l, grp_o, total;
    int n_groups_max;
};

// The arrival counters come first and their places depend only on the unit count
// (sequences x KV heads x row groups), never on n_splits: a workspace zeroed once serves
// every split count of the same cache shape and query rows, since each completed decode
// leaves its arrival counts (the low 16 bits of each counter) at zero.  Split and group
// triples follow.
WsLayout ws_layout(const kvq_cache *c, int32_t n_q_heads, int32_t splits, int32_t n_q = 1) {
    WsLayout w{};
    const size_t G = n_q_heads / c->desc.n_kv_heads;
    const size_t QG = (n_q * G + kvq::kMaxRowsPerGroup - 1) / kvq::kMaxRowsPerGroup;
    const size_t rows = static_cast<size_t>(c->desc.batch) * n_q * n_q_heads;
    const size_t units = static_cast<size_t>(c->desc.batch) * c->desc.n_kv_heads * QG;
    const size_t ng = static_cast<size_t>(kvq::max_merge_groups(splits));
    w.n_groups_max = static_cast<int>(ng);
    w.counters = 0;
    w.counters1 = align256(units * 4);
    w.part_m = w.counters1 + align256(units * kvq::kGroupCounterStride * 4);
    w.part_l = w.part_m + align256(rows * splits * 4);
    w.part_o = w.part_l + align256(rows * splits * 4);
    w.grp_m = w.part_o + align256(rows * splits * c->desc.head_dim * 4);
    w.grp_l = w.grp_m + align256(rows * ng * 4);
    w.grp_o = w.grp_l + align256(rows * ng * 4);
    w.total = w.grp_o + align256(rows * ng * c->desc.head_dim * 4);
    return w;
}

// Decode parameters: the arrival counters, split triples and group triples in `ws`.
void set_workspace(kvq::DecodeParams &p, uint8_t *ws, const WsLayout &w) {
    take_stamp_slot(p);
    p.counters = reinterpret_cast<int32_t *>(ws + w.counters);
    p.counters1 = reinterpret_cast<int32_t *>(ws + w.counters1);
    p.grp_m = reinterpret_cast<float *>(ws + w.grp_m);
    p.grp_l = reinterpret_cast<float *>(ws + w.grp_l);
    p.grp_o = reinterpret_cast<float *>(ws + w.grp_o);
    p.n_groups_max = w.n_groups_max;
    p.part_m = reinterpret_cast<float *>(ws + w.part_m);
    p.part_l = reinterpret_cast<float *>(ws + w.part_l);
    p.part_o = reinterpret_cast<float *>(ws + w.part_o);
}

// ---- per-stream record of which cache each library launch writes ----
// A decode launch reads its cache's lengths and tiles before the previous kernel of the
// stream has finished (DecodeParams::early) unless the library's previous launch on that
// stream wrote the cache.  After kvq_cache_create only this library writes cache memory,
// so the record covers every writer.  A fixed table of streams; once an entry has been
// evicted, streams without an entry are treated as unknown (no early reads).
struct StreamRec {
    cudaStream_t stream;
    const kvq_cache *wrote[2];  // caches written by the latest library launch on the stream
};
constexpr int kTrackSlots = 64;
std::mutex g_track_mu;
StreamRec g_track[kTrackSlots];
int g_track_n = 0, g_track_next = 0;
bool g_track_lost = false;

// Called just before the library enqueues work on `stream` that reads cache `reads`
// (nullptr: none) and writes caches `w0`, `w1` (nullptr: none).  Returns whether the
// reads may start before the previous kernel of the stream completes.
bool track_launch(cudaStream_t stream, const kvq_cache *reads, const kvq_cache *w0,
                  const kvq_cache *w1 = nullptr, const kvq_cache *reads2 = nullptr) {
    std::lock_guard<std::mutex> lock(g_track_mu);
    int i = 0;
    while (i < g_track_n && g_track[i].stream != stream) ++i;
    bool early;
    if (i < g_track_n) {
        early = g_track[i].wrote[0] != reads && g_track[i].wrote[1] != reads &&
                (!reads2 || (g_track[i].wrote[0] != reads2 && g_track[i].wrote[1] != reads2));
    } else {
        early = !g_track_lost;
        if (g_track_n < kTrackSlots) {
            i = g_track_n++;
        } else {
            i = g_track_next;
            g_track_next = (g_track_next + 1) % kTrackSlots;
            g_track_lost = true;
        }
        g_track[i].stream = stream;
    }
    g_track[i].wrote[0] = w0;
    g_track[i].wrote[1] = w1;
    return early && reads != nullptr;
}

}  // namespace

extern "C" {

int32_t kvq_abi_version(void) { return KVQ_ABI_VERSION; }

kvq_status kvq_set_wait_limit(int64_t cycles) {
    if (cycles < 0) return KVQ_ERR_INVALID_ARG;
    g_wait_cycles.store(cycles == 0 ? kvq::kWaitCycles : static_cast<long long>(cycles), std::memory_order_relaxed);
    return KVQ_OK;
}

kvq_status kvq_set_launch_stamps(void *buf, int32_t n_slots, int32_t ctas_per_slot) {
    std::lock_guard<std::mutex> lock(g_stamp_mu);
    if (buf == nullptr) {
        g_stamp_buf = nullptr;
        g_stamp_slots = g_stamp_ctas = g_stamp_next = 0;
        return KVQ_OK;
    }
    if (n_slots < 1 || ctas_per_slot < 1 || !aligned16(buf)) return KVQ_ERR_INVALID_ARG;
    g_stamp_buf = static_cast<unsigned long long *>(buf);
    g_stamp_slots = n_slots;
    g_stamp_ctas = ctas_per_slot;
    g_stamp_next = 0;
    return KVQ_OK;
}

const char *kvq_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
        case KVQ_ERR_CAPACITY: return "append exceeds cache capacity";
        case KVQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case KVQ_ERR_CUDA: return "CUDA error";
        case KVQ_ERR_DEVICE: return "device error word set";
        case KVQ_ERR_SCRATCH: return "decode needs more scratch than the built-in no-allocation buffer holds";
    }
    return "unknown status";
}

int32_t kvq_block_bytes(kvq_type type) {
    switch (type) {
        case KVQ_F16: return 64;
        case KVQ_Q8_0: return 34;
        case KVQ_Q4_0: return 18;
        case KVQ_Q4_1: return 20;
        case KVQ_Q5_0: return 22;
        case KVQ_Q5_1: return 24;
    }
    return 0;
}

kvq_status kvq_select_tier(int64_t cells, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                           uint64_t budget_bytes, kvq_tier_choice *out) {
    if (!out || cells < 0 || n_layers < 1 || n_kv_heads < 1 || head_dim < 32 || head_dim % 32 != 0)
        return KVQ_ERR_INVALID_ARG;
    static const kvq_type ladder[4][2] = {
        {KVQ_F16, KVQ_F16}, {KVQ_Q8_0, KVQ_Q8_0}, {KVQ_Q8_0, KVQ_Q4_0}, {KVQ_Q5_1, KVQ_Q4_0}};
    // blocks per cell over all layers and heads, then bytes per rung (overflow-checked)
    const unsigned __int128 blocks = static_cast<unsigned __int128>(cells) * static_cast<uint64_t>(n_layers) *
                                     static_cast<uint64_t>(n_kv_heads) * static_cast<uint64_t>(head_dim / 32);
    for (int r = 0; r < 4; ++r) {
        const unsigned __int128 b =
            blocks * static_cast<uint64_t>(kvq_block_bytes(ladder[r][0]) + kvq_block_bytes(ladder[r][1]));
        if (b > static_cast<unsigned __int128>(~0ull)) return KVQ_ERR_INVALID_ARG;
        const bool fits = static_cast<uint64_t>(b) <= budget_bytes;
        if (fits || r == 3) {
            out->rung = r;
            out->type_k = ladder[r][0];
            out->type_v = ladder[r][1];
            out->fits = fits ? 1 : 0;
            out->bytes = static_cast<uint64_t>(b);
            return KVQ_OK;
        }
    }
    return KVQ_ERR_INVALID_ARG;  // not reached
}

kvq_status kvq_cache_size(const kvq_cache_desc *desc, size_t *k_bytes, size_t *v_bytes, size_t *state_bytes) {
    kvq_status st = check_desc(desc);
    if (st != KVQ_OK) return st;
    if (!k_bytes || !v_bytes || !state_bytes) return KVQ_ERR_INVALID_ARG;
    size_t kc, kt, vc, vt;
    if (!plane_bytes(desc, desc->type_k, &kc, &kt) || !plane_bytes(desc, desc->type_v, &vc, &vt))
        return KVQ_ERR_INVALID_ARG;
    *k_bytes = kt;
    *v_bytes = vt;
    *state_bytes = state_bytes_for(desc->batch);
    return KVQ_OK;
}

kvq_status kvq_cache_create(const kvq_cache_desc *desc, void *k_mem, void *v_mem, void *state, void *stream,
                            kvq_cache **out) {
    kvq_status st = check_desc(desc);
    if (st != KVQ_OK) return st;
    if (!k_mem || !v_mem || !state || !out) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_mem) || !aligned16(v_mem) || !aligned16(state)) return KVQ_ERR_ALIGNMENT;
    size_t kc, kt, vc, vt;
    if (!plane_bytes(desc, desc->type_k, &kc, &kt) || !plane_bytes(desc, desc->type_v, &vc, &vt))
        return KVQ_ERR_INVALID_ARG;
    kvq_cache *c = new (std::nothrow) kvq_cache;
    if (!c) return KVQ_ERR_INVALID_ARG;
    c->h_len = static_cast<int32_t *>(std::calloc(desc->batch, sizeof(int32_t)));
    if (!c->h_len) {
        delete c;
        return KVQ_ERR_INVALID_ARG;
    }
    c->desc = *desc;
    c->k_mem = static_cast<uint8_t *>(k_mem);
    c->v_mem = static_cast<uint8_t *>(v_mem);
    c->state = static_cast<int32_t *>(state);
    c->k_code_bytes = kc;
    c->v_code_bytes = vc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaMemcpyAsync(c->h_len, state, sizeof(int32_t) * desc->batch, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        std::free(c->h_len);
        delete c;
        return KVQ_ERR_CUDA;
    }
    for (int i = 0; i < desc->batch; ++i) {
        if (c->h_len[i] < 0 || c->h_len[i] > desc->capacity) {
            std::free(c->h_len);
            delete c;
            return KVQ_ERR_INVALID_ARG;
        }
    }
    track_launch(s, nullptr, c);
    *out = c;
    return KVQ_OK;
}

kvq_status kvq_cache_destroy(kvq_cache *cache) {
    if (!cache) return KVQ_ERR_INVALID_ARG;
    std::free(cache->h_len);
    delete cache;
    return KVQ_OK;
}

kvq_status kvq_cache_lengths(const kvq_cache *cache, int32_t *h_len) {
    if (!cache || !h_len) return KVQ_ERR_INVALID_ARG;
    std::memcpy(h_len, cache->h_len, sizeof(int32_t) * cache->desc.batch);
    return KVQ_OK;
}

kvq_status kvq_cache_set_lengths(kvq_cache *cache, const int32_t *h_len, void *stream) {
    if (!cache || !h_len) return KVQ_ERR_INVALID_ARG;
    for (int i = 0; i < cache->desc.batch; ++i)
        if (h_len[i] < 0 || h_len[i] > cache->desc.capacity) return KVQ_ERR_INVALID_ARG;
    std::memcpy(cache->h_len, h_len, sizeof(int32_t) * cache->desc.batch);
    // copy from the mirror (which outlives this call), not from the caller's buffer
    track_launch(static_cast<cudaStream_t>(stream), nullptr, cache);
    return cuda_status(cudaMemcpyAsync(cache->state, cache->h_len, sizeof(int32_t) * cache->desc.batch,
                                       cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_cache_sync_lengths(kvq_cache *cache, void *stream) {
    if (!cache) return KVQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(cache->h_len, cache->state, sizeof(int32_t) * cache->desc.batch,
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

kvq_status kvq_cache_read_error(kvq_cache *cache, void *stream, int32_t *h_err) {
    if (!cache || !h_err) return KVQ_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t *err = cache->state + cache->desc.batch + 1;
    cudaError_t e = cudaMemcpyAsync(h_err, err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

kvq_status kvq_quantize_append(kvq_cache *cache, const float *k, const float *v, int32_t b0, int32_t nb,
                               int32_t n_new, void *stream) {
    if (!cache) return KVQ_ERR_INVALID_ARG;
    if (nb < 0 || n_new < 0 || b0 < 0) return KVQ_ERR_INVALID_ARG;
    if (nb == 0 || n_new == 0) return KVQ_OK;
    if (b0 + static_cast<long long>(nb) > cache->desc.batch) return KVQ_ERR_INVALID_ARG;
    if (!k || !v) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v)) return KVQ_ERR_ALIGNMENT;
    for (int i = 0; i < nb; ++i)
        if (static_cast<long long>(cache->h_len[b0 + i]) + n_new > cache->desc.capacity) return KVQ_ERR_CAPACITY;
    const long long warps = static_cast<long long>(nb) * cache->desc.n_kv_heads * n_new * (cache->desc.head_dim / 128);
    if (warps > (1ll << 31) - 256) return KVQ_ERR_INVALID_ARG;
    kvq::AppendParams p{};
    p.k_codes = cache->k_mem;
    p.k_scales = cache->desc.type_k == KVQ_F16 ? nullptr : cache->k_mem + cache->k_code_bytes;
    p.v_codes = cache->v_mem;
    p.v_scales = cache->desc.type_v == KVQ_F16 ? nullptr : cache->v_mem + cache->v_code_bytes;
    p.len = cache->state;
    p.ticket = cache->state + cache->desc.batch;
    p.err = cache->state + cache->desc.batch + 1;
    p.k = k;
    p.v = v;
    p.b0 = b0;
    p.nb = nb;
    p.n_new = n_new;
    p.Hkv = cache->desc.n_kv_heads;
    p.D = cache->desc.head_dim;
    p.cap = cache->desc.capacity;
    p.cap_tiles = cache->desc.capacity / kvq::kTileRows;
    p.total_warps = static_cast<int>(warps);
    track_launch(static_cast<cudaStream_t>(stream), nullptr, cache);
    cudaError_t e = kvq::launch_append(cache->desc.type_k, cache->desc.type_v, p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    for (int i = 0; i < nb; ++i) cache->h_len[b0 + i] += n_new;
    return KVQ_OK;
}

kvq_status kvq_decode_auto_splits(const kvq_cache *cache, int32_t n_q_heads, int32_t *n_splits) {
    if (!cache || !n_splits) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    int s = 0;
    if (auto_splits(cache, n_q_heads, &s) != 0) return KVQ_ERR_CUDA;
    *n_splits = s;
    return KVQ_OK;
}

kvq_status kvq_decode_workspace_size(const kvq_cache *cache, int32_t n_q_heads, int32_t n_splits, size_t *bytes) {
    if (!cache || !bytes) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s) != 0) return KVQ_ERR_CUDA;
    *bytes = ws_layout(cache, n_q_heads, s).total;
    return KVQ_OK;
}

kvq_status kvq_decode_attention(const kvq_cache *cache, const float *q, int32_t n_q_heads, float scale,
                                int32_t n_splits, void *workspace, float *out, float *lse, void *stream) {
    if (!cache || !q || !workspace || !out) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || (lse && !aligned16(lse)))
        return KVQ_ERR_ALIGNMENT;
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s) != 0) return KVQ_ERR_CUDA;
    const WsLayout w = ws_layout(cache, n_q_heads, s);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    kvq::DecodeParams p = base_params(cache, q, n_q_heads, scale, s);
    p.out = out;
    p.lse = lse;
    set_workspace(p, ws, w);
    p.early = track_launch(static_cast<cudaStream_t>(stream), cache, nullptr) ? 1 : 0;
    return cuda_status(
        kvq::launch_decode(cache->desc.type_k, cache->desc.type_v, p, true, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_append_decode(kvq_cache *cache, const float *k_new, const float *v_new, const float *q,
                             int32_t n_q_heads, float scale, int32_t n_splits, void *workspace, float *out, float *lse,
                             void *stream) {
    if (!cache || !k_new || !v_new || !q || !workspace || !out) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
        (lse && !aligned16(lse)))
        return KVQ_ERR_ALIGNMENT;
    for (int i = 0; i < cache->desc.batch; ++i)
        if (static_cast<long long>(cache->h_len[i]) + 1 > cache->desc.capacity) return KVQ_ERR_CAPACITY;
    const int G = n_q_heads / cache->desc.n_kv_heads;
    if (G > kvq::kMaxRowsPerGroup) {
        // several CTAs per KV head would read the new row: write it first, then attend
        st = kvq_quantize_append(cache, k_new, v_new, 0, cache->desc.batch, 1, stream);
        if (st != KVQ_OK) return st;
        return kvq_decode_attention(cache, q, n_q_heads, scale, n_splits, workspace, out, lse, stream);
    }
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s) != 0) return KVQ_ERR_CUDA;
    const WsLayout w = ws_layout(cache, n_q_heads, s);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    kvq::DecodeParams p = base_params(cache, q, n_q_heads, scale, s);
    p.out = out;
    p.lse = lse;
    set_workspace(p, ws, w);
    p.k_new = k_new;
    p.v_new = v_new;
    p.ticket = cache->state + cache->desc.batch;
    p.early = track_launch(static_cast<cudaStream_t>(stream), cache, cache) ? 1 : 0;
    cudaError_t e =
        kvq::launch_decode(cache->desc.type_k, cache->desc.type_v, p, true, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    for (int i = 0; i < cache->desc.batch; ++i) cache->h_len[i] += 1;
    return KVQ_OK;
}

kvq_status kvq_decode_partials(const kvq_cache *cache, const float *q, int32_t n_q_heads, float scale,
                               int32_t n_splits, float *part_o, float *part_m, float *part_l, void *stream) {
    if (!cache || !q || !part_o || !part_m || !part_l) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    if (n_splits < 1 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(part_o)) return KVQ_ERR_ALIGNMENT;
    kvq::DecodeParams p = base_params(cache, q, n_q_heads, scale, n_splits);
    p.part_o = part_o;
    p.part_m = part_m;
    p.part_l = part_l;
    take_stamp_slot(p);
    p.early = track_launch(static_cast<cudaStream_t>(stream), cache, nullptr) ? 1 : 0;
    return cuda_status(
        kvq::launch_decode(cache->desc.type_k, cache->desc.type_v, p, false, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_combine(const float *part_o, const float *part_m, const float *part_l, int32_t rows,
                       int32_t n_splits, int32_t head_dim, float *out, float *lse, void *stream) {
    if (!part_o || !part_m || !part_l || !out) return KVQ_ERR_INVALID_ARG;
    if (rows < 0 || n_splits < 1 || n_splits > 8192 || head_dim < 4 || head_dim % 4 != 0) return KVQ_ERR_INVALID_ARG;
    if (rows == 0) return KVQ_OK;
    if (!aligned16(part_o) || !aligned16(out)) return KVQ_ERR_ALIGNMENT;
    kvq::CombineParams p{part_o, part_m, part_l, out, lse, rows, n_splits, head_dim};
    track_launch(static_cast<cudaStream_t>(stream), nullptr, nullptr);
    return cuda_status(kvq::launch_combine(p, static_cast<cudaStream_t>(stream)));
}

// ---- draft verify: several queries per sequence, causal within the draft ----
kvq_status kvq_verify_workspace_size(const kvq_cache *cache, int32_t n_q, int32_t n_q_heads, int32_t n_splits,
                                     size_t *bytes) {
    if (!cache || !bytes || n_q < 1 || n_q > KVQ_MAX_VERIFY_QUERIES) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads, n_q);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s, n_q) != 0) return KVQ_ERR_CUDA;
    *bytes = ws_layout(cache, n_q_heads, s, n_q).total;
    return KVQ_OK;
}

kvq_status kvq_decode_verify(const kvq_cache *cache, const float *q, int32_t n_q, int32_t n_q_heads, float scale,
                             int32_t n_splits, void *workspace, float *out, float *lse, void *stream) {
    if (!cache || !q || !workspace || !out || n_q < 1 || n_q > KVQ_MAX_VERIFY_QUERIES) return KVQ_ERR_INVALID_ARG;
    if (!kvq::is_base_type(cache->desc.type_k) || !kvq::is_base_type(cache->desc.type_v)) return KVQ_ERR_UNSUPPORTED;
    kvq_status st = check_q_heads(cache, n_q_heads, n_q);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || (lse && !aligned16(lse)))
        return KVQ_ERR_ALIGNMENT;
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s, n_q) != 0) return KVQ_ERR_CUDA;
    const WsLayout w = ws_layout(cache, n_q_heads, s, n_q);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    kvq::DecodeParams p = base_params(cache, q, n_q_heads, scale, s, n_q);
    p.out = out;
    p.lse = lse;
    set_workspace(p, ws, w);
    p.early = track_launch(static_cast<cudaStream_t>(stream), cache, nullptr) ? 1 : 0;
    if (verify_on_tc(cache, n_q_heads, n_q)) {
        p.QG = 1;
        return cuda_status(
            kvq::launch_verify_tc(cache->desc.type_k, cache->desc.type_v, p, static_cast<cudaStream_t>(stream)));
    }
    return cuda_status(kvq::launch_verify(cache->desc.type_k, cache->desc.type_v, p, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_set_verify_path(int32_t path) {
    if (path < 0 || path > 2) return KVQ_ERR_INVALID_ARG;
    g_verify_path.store(path, std::memory_order_relaxed);
    return KVQ_OK;
}

// ---- rolling f16 window + quantised tail ----
static kvq_status check_window_pair(const kvq_cache *window, const kvq_cache *tail) {
    if (!window || !tail || window == tail) return KVQ_ERR_INVALID_ARG;
    if (window->desc.type_k != KVQ_F16 || window->desc.type_v != KVQ_F16) return KVQ_ERR_UNSUPPORTED;
    if (!kvq::is_base_type(tail->desc.type_k) || !kvq::is_base_type(tail->desc.type_v)) return KVQ_ERR_UNSUPPORTED;
    if (window->desc.batch != tail->desc.batch || window->desc.n_kv_heads != tail->desc.n_kv_heads ||
        window->desc.head_dim != tail->desc.head_dim)
        return KVQ_ERR_INVALID_ARG;
    return KVQ_OK;
}

kvq_status kvq_window_append(kvq_cache *window, kvq_cache *tail, const float *k, const float *v, void *stream) {
    kvq_status st = check_window_pair(window, tail);
    if (st != KVQ_OK) return st;
    if (!k || !v) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v)) return KVQ_ERR_ALIGNMENT;
    const int W = window->desc.capacity;
    for (int b = 0; b < window->desc.batch; ++b)
        if (window->h_len[b] >= W && static_cast<long long>(tail->h_len[b]) + 1 > tail->desc.capacity)
            return KVQ_ERR_CAPACITY;
    kvq::WindowParams p{};
    p.w_k = window->k_mem;
    p.w_v = window->v_mem;
    p.t_kc = tail->k_mem;
    p.t_ks = tail->desc.type_k == KVQ_F16 ? nullptr : tail->k_mem + tail->k_code_bytes;
    p.t_vc = tail->v_mem;
    p.t_vs = tail->desc.type_v == KVQ_F16 ? nullptr : tail->v_mem + tail->v_code_bytes;
    p.w_len = window->state;
    p.ticket = window->state + window->desc.batch;
    p.w_err = window->state + window->desc.batch + 1;
    p.t_len = tail->state;
    p.t_err = tail->state + tail->desc.batch + 1;
    p.k = k;
    p.v = v;
    p.B = window->desc.batch;
    p.Hkv = window->desc.n_kv_heads;
    p.D = window->desc.head_dim;
    p.w_cap = W;
    p.w_cap_tiles = W / kvq::kTileRows;
    p.t_cap = tail->desc.capacity;
    p.t_cap_tiles = tail->desc.capacity / kvq::kTileRows;
    p.total_warps = p.B * p.Hkv * (p.D / kvq::kSlice);
    track_launch(static_cast<cudaStream_t>(stream), nullptr, window, tail);
    if (kvq::launch_window_append(tail->desc.type_k, tail->desc.type_v, p, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    for (int b = 0; b < window->desc.batch; ++b) {
        if (window->h_len[b] < W)
            window->h_len[b] += 1;
        else
            tail->h_len[b] += 1;
    }
    return KVQ_OK;
}

static kvq_status window_splits(const kvq_cache *window, const kvq_cache *tail, int32_t n_q_heads, int *sw, int *stl) {
    kvq_status st = check_window_pair(window, tail);
    if (st != KVQ_OK) return st;
    st = check_q_heads(window, n_q_heads);
    if (st != KVQ_OK) return st;
    if (auto_splits(window, n_q_heads, sw) != 0 || auto_splits(tail, n_q_heads, stl) != 0) return KVQ_ERR_CUDA;
    return KVQ_OK;
}

// One launch over both regions: the tail's automatic split count S is shared between the
// regions in proportion to their capacity bytes (window bytes weighted, below), at least
// one each.
static bool dual_splits(const kvq_cache *window, const kvq_cache *tail, int32_t n_q_heads, int *nw, int *S) {
    if (window->desc.head_dim != kvq::kSlice && window->desc.head_dim != 2 * kvq::kSlice) return false;
    int s = 0;
    if (auto_splits(tail, n_q_heads, &s) != 0 || s < 2) return false;
    auto row_bytes = [](const kvq_cache *c) {
        const int NS = c->desc.head_dim / kvq::kSlice;
        return static_cast<double>(NS) *
               (kvq::code_tile_bytes(c->desc.type_k) + kvq::code_tile_bytes(c->desc.type_v) +
                kvq::scale_tile_bytes(c->desc.type_k) + kvq::scale_tile_bytes(c->desc.type_v)) /
               kvq::kTileRows;
    };
    // a window byte weighs more than a tail byte: the f16 body runs with the tail's
    // tile-warp count and reads twice the bytes per value, and the two bodies share the
    // instruction cache.  Weights 1.0 / 1.25 / 1.5 / 1.75 / 2.0 / 2.5 measured 42.8 / 44.9 /
    // 45.4 / 45.9 / 46.2 / 45.2 % of the copy peak with 256-wide heads and 68.5 / 70.3 /
    // 70.4 / 70.4 / 67.4 / 67.4 % with 128-wide heads.
    const double weight = window->desc.head_dim == 2 * kvq::kSlice ? 2.0 : 1.75;
    const double bw = weight * row_bytes(window) * window->desc.capacity;
    const double bt = row_bytes(tail) * tail->desc.capacity;
    int w = static_cast<int>(s * bw / (bw + bt) + 0.5);
    w = w < 1 ? 1 : (w > s - 1 ? s - 1 : w);
    *nw = w;
    *S = s;
    return true;
}

// Workspace of a window + tail decode: one decode workspace, used by the window's decode
// and then by the tail's (each leaves its counters at zero), and the window's result at
// *res_off; or, for the one-launch form, one decode workspace over the splits of both
// regions, whichever is larger.  Then the eviction flags of kvq_window_append_decode
// ([B][Hkv] int32, left at zero) at *flag_off.
static size_t window_ws(const kvq_cache *window, const kvq_cache *tail, int32_t n_q_heads, int sw, int stl,
                        size_t *res_off, size_t *flag_off = nullptr) {
    const size_t wsz = ws_layout(window, n_q_heads, sw).total, tsz = ws_layout(tail, n_q_heads, stl).total;
    const size_t rows = static_cast<size_t>(window->desc.batch) * n_q_heads;
    *res_off = align256(wsz > tsz ? wsz : tsz);
    size_t total = *res_off + align256(rows * window->desc.head_dim * 4) + align256(rows * 4);
    int nw = 0, S = 0;
    if (dual_splits(window, tail, n_q_heads, &nw, &S)) {
        const size_t d = ws_layout(tail, n_q_heads, S).total;
        if (d > total) total = d;
    }
    total = align256(total);
    if (flag_off) *flag_off = total;
    return total + align256(static_cast<size_t>(window->desc.batch) * window->desc.n_kv_heads * 4);
}

kvq_status kvq_window_workspace_size(const kvq_cache *window, const kvq_cache *tail, int32_t n_q_heads,
                                     size_t *bytes) {
    if (!bytes) return KVQ_ERR_INVALID_ARG;
    int sw = 0, stl = 0;
    kvq_status st = window_splits(window, tail, n_q_heads, &sw, &stl);
    if (st != KVQ_OK) return st;
    size_t off = 0;
    *bytes = window_ws(window, tail, n_q_heads, sw, stl, &off);
    return KVQ_OK;
}

kvq_status kvq_window_decode(const kvq_cache *window, const kvq_cache *tail, const float *q, int32_t n_q_heads,
                             float scale, void *workspace, float *out, float *lse, void *stream) {
    if (!q || !workspace || !out) return KVQ_ERR_INVALID_ARG;
    int sw = 0, stl = 0;
    kvq_status st = window_splits(window, tail, n_q_heads, &sw, &stl);
    if (st != KVQ_OK) return st;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || (lse && !aligned16(lse)))
        return KVQ_ERR_ALIGNMENT;
    size_t res_off = 0;
    window_ws(window, tail, n_q_heads, sw, stl, &res_off);
    const size_t rows = static_cast<size_t>(window->desc.batch) * n_q_heads;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *w_out = reinterpret_cast<float *>(ws + res_off);
    float *w_lse = reinterpret_cast<float *>(ws + res_off + align256(rows * window->desc.head_dim * 4));
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int nw = 0, S = 0;
    if (dual_splits(window, tail, n_q_heads, &nw, &S)) {
        // one launch: splits [0, nw) over the window, [nw, S) over the tail, one merge
        const WsLayout w = ws_layout(tail, n_q_heads, S);
        kvq::DecodeParams pr[2] = {base_params(window, q, n_q_heads, scale, nw),
                                   base_params(tail, q, n_q_heads, scale, S - nw)};
        for (int r = 0; r < 2; ++r) {
            kvq::DecodeParams &p = pr[r];
            p.out = out;
            p.lse = lse;
            set_workspace(p, ws, w);
            p.part_stride = S;
            p.part_base = r == 0 ? 0 : nw;
            p.merge_slots = S;
        }
        pr[0].early = pr[1].early = track_launch(cs, window, nullptr, nullptr, tail) ? 1 : 0;
        return cuda_status(kvq::launch_window_dual(tail->desc.type_k, tail->desc.type_v, window->desc.head_dim, pr[0],
                                                   pr[1], nw, cs));
    }
    // each region in its own typed decode (the window's first, into the workspace); the
    // tail's final merge takes the window's result as one more triple
    const kvq_cache *region[2] = {window, tail};
    const int splits[2] = {sw, stl};
    for (int r = 0; r < 2; ++r) {
        const WsLayout w = ws_layout(region[r], n_q_heads, splits[r]);
        kvq::DecodeParams p = base_params(region[r], q, n_q_heads, scale, splits[r]);
        p.out = r == 0 ? w_out : out;
        p.lse = r == 0 ? w_lse : lse;
        set_workspace(p, ws, w);
        if (r == 1) {
            p.ext_out = w_out;
            p.ext_lse = w_lse;
        }
        p.early = track_launch(cs, region[r], nullptr) ? 1 : 0;
        if (kvq::launch_decode(region[r]->desc.type_k, region[r]->desc.type_v, p, true, cs) != cudaSuccess)
            return KVQ_ERR_CUDA;
    }
    return KVQ_OK;
}

kvq_status kvq_window_append_decode(kvq_cache *window, kvq_cache *tail, const float *k, const float *v,
                                    const float *q, int32_t n_q_heads, float scale, void *workspace, float *out,
                                    float *lse, void *stream) {
    kvq_status st = check_window_pair(window, tail);
    if (st != KVQ_OK) return st;
    if (!k || !v || !q || !workspace || !out) return KVQ_ERR_INVALID_ARG;
    int sw = 0, stl = 0;
    st = window_splits(window, tail, n_q_heads, &sw, &stl);
    if (st != KVQ_OK) return st;
    if (!aligned16(k) || !aligned16(v) || !aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
        (lse && !aligned16(lse)))
        return KVQ_ERR_ALIGNMENT;
    const int W = window->desc.capacity;
    for (int b = 0; b < window->desc.batch; ++b)
        if (window->h_len[b] >= W && static_cast<long long>(tail->h_len[b]) + 1 > tail->desc.capacity)
            return KVQ_ERR_CAPACITY;
    auto two_launches = [&]() {
        kvq_status s2 = kvq_window_append(window, tail, k, v, stream);
        if (s2 != KVQ_OK) return s2;
        return kvq_window_decode(window, tail, q, n_q_heads, scale, workspace, out, lse, stream);
    };
    int nw = 0, S = 0;
    // one launch needs one CTA per (split, KV head, sequence): at most 8 query heads per KV head
    if (n_q_heads / window->desc.n_kv_heads > kvq::kMaxRowsPerGroup || !dual_splits(window, tail, n_q_heads, &nw, &S))
        return two_launches();
    size_t res_off = 0, flag_off = 0;
    window_ws(window, tail, n_q_heads, sw, stl, &res_off, &flag_off);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const WsLayout w = ws_layout(tail, n_q_heads, S);
    kvq::DecodeParams pr[2] = {base_params(window, q, n_q_heads, scale, nw), base_params(tail, q, n_q_heads, scale, S - nw)};
    for (int r = 0; r < 2; ++r) {
        kvq::DecodeParams &p = pr[r];
        p.out = out;
        p.lse = lse;
        set_workspace(p, ws, w);
        p.part_stride = S;
        p.part_base = r == 0 ? 0 : nw;
        p.merge_slots = S;
        p.win = r + 1;
        p.wl_len = window->state;
        p.tl_len = tail->state;
        p.wl_err = window->state + window->desc.batch + 1;
        p.tl_err = tail->state + tail->desc.batch + 1;
        p.wl_cap = W;
        p.tl_cap = tail->desc.capacity;
        p.win_k = window->k_mem;
        p.win_v = window->v_mem;
        p.evict = reinterpret_cast<int32_t *>(ws + flag_off);
        p.ticket = window->state + window->desc.batch;  // one ticket for the whole grid
    }
    pr[0].k_new = k;
    pr[0].v_new = v;
    pr[0].early = pr[1].early = track_launch(cs, window, window, tail, tail) ? 1 : 0;
    const cudaError_t e =
        kvq::launch_window_dual(tail->desc.type_k, tail->desc.type_v, window->desc.head_dim, pr[0], pr[1], nw, cs);
    if (e == cudaErrorCooperativeLaunchTooLarge) return two_launches();  // not resident at once: nothing launched
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    for (int b = 0; b < window->desc.batch; ++b) {
        if (window->h_len[b] < W)
            window->h_len[b] += 1;
        else
            tail->h_len[b] += 1;
    }
    return KVQ_OK;
}

// ---- decode without a caller workspace: scratch compiled into the library ----
namespace {
// Shared by every call of kvq_decode_attention_noalloc on a device; see include/kvq.h.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];
constexpr int kNoAllocDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kNoAllocDevices] = {};
// Bytes at the front of the array that hold zero once the last call's kernel has finished:
// the counter region of that call (its split triples lie beyond it).
size_t g_noalloc_zero[kNoAllocDevices] = {};

// Device address of the scratch array for device `dev`, looked up once per device (the
// caller holds g_noalloc_mutex and has made `dev` current).
kvq_status noalloc_scratch(int dev, void **addr) {
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
        g_noalloc_addr[dev] = p;
        g_noalloc_zero[dev] = 0;  // contents unknown until the first clear
    }
    *addr = g_noalloc_addr[dev];
    return KVQ_OK;
}
}  // namespace

kvq_status kvq_decode_attention_noalloc(const kvq_cache *cache, const float *q, int32_t n_q_heads, float scale,
                                        int32_t n_splits, float *out, float *lse, void *stream) {
    if (!cache || !q || !out) return KVQ_ERR_INVALID_ARG;
    kvq_status st = check_q_heads(cache, n_q_heads);
    if (st != KVQ_OK) return st;
    if (n_splits < 0 || n_splits > kvq::kMaxSplits) return KVQ_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || (lse && !aligned16(lse))) return KVQ_ERR_ALIGNMENT;
    int s = n_splits;
    if (s == 0 && auto_splits(cache, n_q_heads, &s) != 0) return KVQ_ERR_CUDA;
    const WsLayout w = ws_layout(cache, n_q_heads, s);
    if (w.total > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_SCRATCH;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocDevices) return KVQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    void *base = nullptr;
    st = noalloc_scratch(dev, &base);
    if (st != KVQ_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(base);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // The arrival counts of both merge levels must start at zero; the rest is
    // overwritten.  Every finished decode leaves them at zero, so the clear is
    // needed only when this call's counter region reaches past the previous call's (whose
    // split triples lie beyond it); skipping it keeps the programmatic launch overlap.
    if (w.part_m > g_noalloc_zero[dev]) {
        g_noalloc_zero[dev] = 0;
        if (cudaMemsetAsync(ws, 0, w.part_m, cs) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    g_noalloc_zero[dev] = w.part_m;
    kvq::DecodeParams p = base_params(cache, q, n_q_heads, scale, s);
    p.out = out;
    p.lse = lse;
    set_workspace(p, ws, w);
    p.early = track_launch(cs, cache, nullptr) ? 1 : 0;
    return cuda_status(kvq::launch_decode(cache->desc.type_k, cache->desc.type_v, p, true, cs));
}

}  // extern "C"
