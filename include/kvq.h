/*
 * kvq.h -- C ABI of libkvq: a block-quantised KV cache with quantise-on-append and
 * split-K single-token decode attention for one NVIDIA GB300 (sm_103a).
 *
 * The operation: for each sequence b and
 * query head hq, with G = Hq / Hkv query heads sharing KV head h = hq / G,
 *
 *     s_t   = scale * <q[b,hq,:], k_hat[b,h,t,:]>          for t < len[b]
 *     out   = sum_t exp(s_t - M) v_hat[b,h,t,:] / sum_t exp(s_t - M),  M = max_t s_t
 *     lse   = M + log(sum_t exp(s_t - M))
 *
 * where k_hat, v_hat are the dequantised cache rows.  Exact softmax attention is what
 * the pages require a quantised reader to reproduce ("logit-identical", real_frac = 0:
 * "HAL #582 -- per-layer KV compression study", section 3b finding 2 and section 5 P0).
 * Storage types are GGML-style blocks of 32 values along the head dimension with one
 * f16 scale: q8_0 (34 bytes / 32 values), q4_0 (18 bytes / 32 values), and the f16
 * control arm (same study, section 1 size model: 102 / 54 / 192 KiB per token for the
 * 48-layer, 8-KV-head, D=128 model).  Asymmetric pairs (q8_0 K / q4_0 V, the study's
 * default tier, section 4) and symmetric pairs are supported; any (K type, V type)
 * combination of the three is accepted.
 *
 * Quantiser rules (fp32, one rounding per operation):
 *   q8_0: d = amax/127; q_j = round_half_away(x_j * (1/d)) (0 if d == 0); scale = f16_rne(d)
 *   q4_0: m = x_k with the largest |x_k| (lowest k on ties); d = m/-8;
 *         c_j = min(15, trunc(x_j * (1/d) + 8.5)); scale = f16_rne(d);
 *         a 32-value block packs byte i = c_i | c_{i+16} << 4   (GGML nibble order)
 *   f16 : x -> binary16, round to nearest even.
 *   Dequantised values: q8_0 f16(d)*q, q4_0 f16(d)*(c-8), f16 as stored.
 *
 * Further scalar types (the study's section 5 P0 note lists q8/q5, q5/q5, q5_1/q5_1,
 * q4_1/q4_1 among the typed readers; section 5 P1 floors its ladder at q5_1 K / q4_0 V).
 * The pages name these GGML-style formats without defining them; the plain reading is:
 *   q4_1: lo = min x, hi = max x, d = (hi - lo)/15, c_j = min(15, trunc((x_j - lo)*(1/d)
 *         + 0.5)); scales f16(d), f16(lo); x_hat = f16(d)*c + f16(lo)
 *   q5_0: as q4_0 with d = m/-16, c_j = min(31, trunc(x_j*(1/d) + 16.5)); x_hat = f16(d)*(c-16)
 *   q5_1: as q4_1 with d = (hi - lo)/31 and codes up to 31
 * Caches accept the pairs of f16/q8_0/q4_0 and the pairs (q8_0, q5_0), (q5_0, q5_0),
 * (q5_1, q5_1), (q4_1, q4_1), (q5_1, q4_0); draft verify and the window + tail cache
 * accept f16/q8_0/q4_0 only (KVQ_ERR_UNSUPPORTED otherwise).
 *
 * ---------------------------------------------------------------------------------
 * Memory ownership.  The library allocates NO device memory.  The caller allocates
 * (with any allocator) the K plane, the V plane, the state block and the decode
 * workspace, sized by kvq_cache_size / kvq_decode_workspace_size, and keeps them alive
 * while the cache handle exists.  A handle holds host metadata only (including a host
 * mirror of the lengths used for capacity checks).  Handles are not thread-safe; all
 * calls on one cache must be issued to one stream (or externally ordered).
 *
 * Asynchrony.  Every call that takes a stream enqueues work on it and returns without
 * synchronising, except kvq_cache_create, kvq_cache_sync_lengths and
 * kvq_cache_read_error, which synchronise their stream as documented.  Device pointers must point to
 * memory of the current CUDA device.  `stream` is a cudaStream_t (NULL = legacy default).
 *
 * Early reads.  The decode kernels are launched with programmatic dependent launch: a
 * launch may start while the previous kernel of its stream is still finishing.  Queries,
 * new rows, outputs and the workspace are touched only once that kernel has completed.
 * The cache's lengths and tiles are read before then whenever the library's own record
 * shows that the previous library launch on the stream did not write this cache (the
 * library notes, per stream, which cache each of its launches writes).  So after
 * kvq_cache_create the K plane, V plane and state block must be written only through
 * this library; a kernel of the caller's that writes them breaks that record.
 *
 * Errors.  Every entry point returns a kvq_status; nothing aborts, traps or throws.
 * Argument errors are detected on the host before any launch and leave device memory
 * untouched.  A launch failure returns KVQ_ERR_CUDA (the CUDA error is not cleared from
 * the context if it is sticky).  Conditions only the device can see (an append past
 * capacity after lengths changed behind the host mirror, e.g. in a CUDA-graph replay)
 * set the state block's error word; kvq_cache_read_error reports it.
 *
 * ---------------------------------------------------------------------------------
 * Cache layout ("fragment-native" tiles).  Rows of one (sequence b, KV head h) are
 * grouped in tiles of 16 consecutive positions; capacity must be a multiple of 16.
 * D = 128 * NS (NS = 1 or 2 slices).  Each plane (K and V separately) is
 *
 *     [codes region : B][Hkv][capacity/16][NS][code_tile_bytes]
 *     [scales region: B][Hkv][capacity/16][NS][128]             (absent for f16)
 *
 * with code_tile_bytes = 2048 (q8_0), 1024 (q4_0), 4096 (f16) per 16 rows x 128 values,
 * so the plane size equals the GGML block footprint exactly (bits/value 8.5, 4.5, 16;
 * 5, 5.5, 6 for q4_1, q5_0, q5_1).
 * Inside a tile, for row kt in [0,16) and value index dd in [0,128) of the slice, with
 *     n = kt % 8, st = kt / 8, and for "pair" order A/B/C/D:
 *         kt < 8 : j = kt/2,      pos = kt%2 ? 1 (B) : 0 (A)
 *         kt >= 8: j = (kt-8)/2,  pos = kt%2 ? 3 (D) : 2 (C)
 * byte offsets are (b = dd/32, i = dd%32):
 *   K, q8_0 : b*512 + (4n + (dd%16)/4)*16 + (2st + (i/16))*4 + dd%4
 *   K, q4_0 : (b/2)*512 + (4n + (i%16)/4)*16 + (2(b%2) + st)*4 + (i%16)%4,
 *             value in the low nibble if i < 16, else the high nibble
 *   K, f16  : (2b + st)*512 + (4n + (dd%16)/4)*16 + (i/16)*8 + P(dd%4)*2,
 *             P(0)=0, P(2)=1, P(1)=2, P(3)=3
 *   V rows use the pair order; with r = i%16, hv = i/16, n' = r/2:
 *   V, q8_0 : b*512 + (4n' + j)*16 + ((r%2) + 2hv)*4 + Q(pos),      Q(A,B,C,D) = 0,2,1,3
 *   V, q4_0 : (b/2)*512 + (4n' + j)*16 + (2(b%2) + r%2)*4 + Q(pos),
 *             value in the low nibble if i < 16, else the high nibble
 *   V, f16  : (2b + hv)*512 + (4n' + j)*16 + (r%2)*8 + pos*2
 *   K/V, q4_1, q5_0, q5_1: the low 4 bits of each code at the q4_0 nibble place; for q5_0
 *             and q5_1 the fifth bits follow the 1024 nibble bytes: for a nibble at byte
 *             offset o, the 32-bit word at 1024 + (o/512)*128 + ((o%512)/16)*4 holds it at
 *             bit 8e + 4 + w (low nibble) or 8e + w (high nibble), e = o%4, w = (o%16)/4
 *             (code_tile_bytes 1024 for q4_1, 1280 for q5_0 and q5_1)
 *   scales (K or V), for block b of the slice: j*32 + b*8 + pos*2   (f16 bits); q4_1 and
 *             q5_1 hold lo at 128 + the same offset (scale region 256 bytes per tile slice)
 * The codes and scales are the GGML q8_0/q4_0 values above; only their placement
 * differs from GGML's array-of-blocks order, and a q8_0 code q is stored as a
 * sign-magnitude byte (q < 0 ? 0x80 | -q : q), which a permute and a mask turn into the
 * f16 subnormal q * 2^-24 that the decode kernel feeds to the tensor cores.
 *
 * State block (int32, 16-byte multiple): [len[B]][append ticket][error word][pad].
 * Zero it (or set lengths with kvq_cache_set_lengths) before kvq_cache_create.
 * ---------------------------------------------------------------------------------
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_ABI_VERSION 4

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

typedef enum {
    KVQ_F16 = 0,
    KVQ_Q8_0 = 1,
    KVQ_Q4_0 = 2,
    KVQ_Q4_1 = 3, /* see "Further scalar types" below */
    KVQ_Q5_0 = 4,
    KVQ_Q5_1 = 5
} kvq_type;

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad descriptor, sizes overflow       */
    KVQ_ERR_UNSUPPORTED = 2, /* head_dim not 128/256, unknown type, no suitable GPU           */
    KVQ_ERR_CAPACITY = 3,    /* append would exceed capacity (nothing is written)             */
    KVQ_ERR_ALIGNMENT = 4,   /* a pointer is not 16-byte aligned                              */
    KVQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed                          */
    KVQ_ERR_DEVICE = 6,      /* the device error word was set (see kvq_cache_read_error)      */
    KVQ_ERR_SCRATCH = 7      /* kvq_decode_attention_noalloc: the call needs more scratch than
                                the library's built-in buffer (KVQ_NOALLOC_SCRATCH_BYTES) has  */
} kvq_status;

/* Device error word bits (kvq_cache_read_error). */
#define KVQ_DEVERR_CAPACITY 0x1 /* an append found len + n_new > capacity on the device     */
#define KVQ_DEVERR_TIMEOUT 0x2  /* a pipeline or merge wait in a kernel took longer than its
                                   limit (kvq_set_wait_limit) or gave up: the outputs of that
                                   launch are undefined (the workspace counters are still
                                   left at zero)                                             */

typedef struct {
    int32_t batch;      /* B: sequences held by the cache (>= 1)                       */
    int32_t n_kv_heads; /* Hkv (>= 1)                                                  */
    int32_t head_dim;   /* D: 128 or 256                                               */
    int32_t capacity;   /* rows per (sequence, KV head); a positive multiple of 16     */
    int32_t type_k;     /* kvq_type of the K plane                                     */
    int32_t type_v;     /* kvq_type of the V plane                                     */
} kvq_cache_desc;

typedef struct kvq_cache kvq_cache; /* opaque host handle */

/* Bytes the caller must allocate for the K plane, the V plane and the state block.
 * Pure host arithmetic; no CUDA call. */
KVQ_API kvq_status kvq_cache_size(const kvq_cache_desc *desc, size_t *k_bytes, size_t *v_bytes,
                          size_t *state_bytes);

/* Create a handle over caller-owned device memory (all three pointers 16-byte aligned).
 * Reads the lengths from `state` once to seed the host mirror: the copy is queued on
 * `stream` (so it follows whatever the caller queued there, e.g. the zero-fill of the
 * state block) and the call synchronises that stream.  Fails with KVQ_ERR_INVALID_ARG
 * if a length is outside [0, capacity]. */
KVQ_API kvq_status kvq_cache_create(const kvq_cache_desc *desc, void *k_mem, void *v_mem, void *state,
                                    void *stream, kvq_cache **out);
KVQ_API kvq_status kvq_cache_destroy(kvq_cache *cache);

/* Host mirror of the lengths (B int32).  Exact unless appends ran in a replayed graph. */
KVQ_API kvq_status kvq_cache_lengths(const kvq_cache *cache, int32_t *h_len);
/* Set lengths (B int32 host array, each in [0, capacity]); async copy on `stream`. */
KVQ_API kvq_status kvq_cache_set_lengths(kvq_cache *cache, const int32_t *h_len, void *stream);
/* Re-read the lengths from the device into the mirror (synchronises `stream`). */
KVQ_API kvq_status kvq_cache_sync_lengths(kvq_cache *cache, void *stream);
/* Read and clear the device error word (synchronises `stream`).  *h_err = KVQ_DEVERR_* bits. */
KVQ_API kvq_status kvq_cache_read_error(kvq_cache *cache, void *stream, int32_t *h_err);

/*
 * Quantise-on-append (the write path of "HAL #582", section 5 P2: new tokens are
 * quantised once when they are written).  k and v are fp32 device arrays
 * [nb][Hkv][n_new][D] (row-major); rows go to positions len[b0+i] .. len[b0+i]+n_new-1
 * of sequence b0+i, after which len[b0+i] += n_new on the device (in the same launch,
 * so append + decode can be captured in a CUDA graph).  Positions are read from the
 * device lengths, not the host mirror.  Returns KVQ_ERR_CAPACITY (nothing written) if
 * the mirror shows an overflow; an overflow seen only on the device skips that
 * sequence and sets KVQ_DEVERR_CAPACITY.  n_new == 0 or nb == 0 is a no-op.
 */
KVQ_API kvq_status kvq_quantize_append(kvq_cache *cache, const float *k, const float *v, int32_t b0,
                               int32_t nb, int32_t n_new, void *stream);

/* Number of key splits the decode uses when n_splits == 0 (depends on the GPU, the
 * cache shape and n_q_heads; not on the lengths, so it is stable under graph replay). */
KVQ_API kvq_status kvq_decode_auto_splits(const kvq_cache *cache, int32_t n_q_heads, int32_t *n_splits);

/* Workspace bytes for kvq_decode_attention with this n_splits (0 = auto).  The workspace
 * holds per-(sequence, KV head, group of 8 query rows) arrival counters at its front,
 * then split and group partials.  Zero it once before its first use; every completed
 * decode leaves the arrival counts at zero (the low 16 bits of each counter: the one-level
 * column merge keeps a launch epoch in the bits above), including one whose waits timed
 * out (a CTA that gives up still arrives).  The counters' places depend on the cache's batch
 * and n_kv_heads and on n_q_heads (and n_q for draft verify) but not on n_splits, so one
 * zeroed workspace serves every split count of those shapes; zero it again before using
 * it for another shape. */
KVQ_API kvq_status kvq_decode_workspace_size(const kvq_cache *cache, int32_t n_q_heads, int32_t n_splits,
                                     size_t *bytes);

/*
 * Split-K decode attention over the whole cache (all B sequences, lengths read on the
 * device).  q: fp32 [B][Hq][D]; out: fp32 [B][Hq][D]; lse: fp32 [B][Hq] natural log, or
 * NULL.  scale multiplies q.k (e.g. 1/sqrt(D)).  Hq must be a multiple of Hkv.  Keys are
 * split into n_splits contiguous ranges per (sequence, KV head) (0 = auto, else 1..1024);
 * each range is attended with an online softmax in fp32, and the last range to finish
 * merges all ranges exactly (HAL #582 section 5 P2: softmax partials of ranges combine
 * without loss).  len == 0
 * gives out = 0 and lse = -inf.  One kernel launch.
 */
KVQ_API kvq_status kvq_decode_attention(const kvq_cache *cache, const float *q, int32_t n_q_heads,
                                float scale, int32_t n_splits, void *workspace, float *out,
                                float *lse, void *stream);

/*
 * One decode step of the hot path in one launch: quantise-on-append of one new K/V row per
 * sequence (k_new, v_new: fp32 [B][Hkv][D]) at position len[b], then split-K decode
 * attention over len[b] + 1 rows (the new row included), then len[b] += 1 on the device.
 * Arguments and workspace as kvq_decode_attention.  The CTA whose key range holds the new
 * row quantises it (same rules and layout as kvq_quantize_append) before reading that
 * tile, so the row is written exactly once; when more than 8 query heads share a KV head
 * the call falls back to kvq_quantize_append followed by kvq_decode_attention.  Returns
 * KVQ_ERR_CAPACITY (nothing launched) if the host mirror shows a full sequence; a full
 * sequence seen only on the device is attended without the new row, not advanced, and
 * sets KVQ_DEVERR_CAPACITY.
 */
KVQ_API kvq_status kvq_append_decode(kvq_cache *cache, const float *k_new, const float *v_new, const float *q,
                                     int32_t n_q_heads, float scale, int32_t n_splits, void *workspace,
                                     float *out, float *lse, void *stream);

/*
 * Same split attention, but writes the unnormalised split triples instead of merging
 * them: part_o fp32 [B][Hq][n_splits][D] = sum_t exp(s_t - m) v_hat_t over the split,
 * part_m [B][Hq][n_splits] = max_t s_t (natural units), part_l = sum_t exp(s_t - m).
 * Empty splits give (o, m, l) = (0, -inf, 0).  n_splits must be given (>= 1).  Split s
 * of a sequence with T = ceil(len/16) tiles covers tiles [s*c, min(T, (s+1)*c)),
 * c = ceil(T / min(n_splits, T)).  For merging several caches or key regions, or shards
 * of one context held on several GPUs, with kvq_combine.
 */
KVQ_API kvq_status kvq_decode_partials(const kvq_cache *cache, const float *q, int32_t n_q_heads,
                               float scale, int32_t n_splits, float *part_o, float *part_m,
                               float *part_l, void *stream);

/*
 * Merge split triples: for each of `rows` rows, M = max_s m_s, w_s = exp(m_s - M),
 * out = sum_s w_s o_s / sum_s w_s l_s, lse = M + log(sum_s w_s l_s) (lse may be NULL).
 * part_o fp32 [rows][n_splits][head_dim], part_m / part_l fp32 [rows][n_splits],
 * out fp32 [rows][head_dim].  head_dim a positive multiple of 4; rows with every split
 * empty give out = 0, lse = -inf.
 */
KVQ_API kvq_status kvq_combine(const float *part_o, const float *part_m, const float *part_l,
                       int32_t rows, int32_t n_splits, int32_t head_dim, float *out, float *lse,
                       void *stream);

/*
 * Draft verify: decode attention for n_q (1..KVQ_MAX_VERIFY_QUERIES) queries per sequence,
 * the last n_q cache rows being the draft tokens (appended before, e.g. with
 * kvq_quantize_append).  Query i (0-based) of sequence b attends causally to positions
 * [0, len[b] - n_q + i] -- positions past the length or before 0 are not attended (a query
 * that sees no position gets out = 0, lse = -inf).  "HAL #582 -- per-layer KV compression
 * study", section 5 P0: the quantised MMA reader serves decode batches of up to 16 query
 * rows (draft verify) in the same typed kernels.
 *   q    : fp32 [B][n_q][n_q_heads][D];   out : fp32 [B][n_q][n_q_heads][D]
 *   lse  : fp32 [B][n_q][n_q_heads] or NULL
 *   workspace: kvq_verify_workspace_size bytes, zeroed once before first use (as for
 *   kvq_decode_attention).  Each group of 8 of the n_q * G query rows of a KV head runs
 *   in its own CTAs, which read the same tiles at the same time (L2 serves the repeats).
 */
#define KVQ_MAX_VERIFY_QUERIES 16
KVQ_API kvq_status kvq_verify_workspace_size(const kvq_cache *cache, int32_t n_q, int32_t n_q_heads,
                                             int32_t n_splits, size_t *bytes);
KVQ_API kvq_status kvq_decode_verify(const kvq_cache *cache, const float *q, int32_t n_q, int32_t n_q_heads,
                                     float scale, int32_t n_splits, void *workspace, float *out, float *lse,
                                     void *stream);

/*
 * Kernel choice of kvq_decode_verify (process-wide; the result is the same exact attention
 * either way, within the same tolerance).  0 (default): when a (sequence, KV head) has 49
 * (D = 256) or 33 (D = 128) to 128 query rows (n_q * Hq / Hkv), all of them form one
 * 128-row tile on the tensor cores with accumulators in tensor memory (tcgen05): each key
 * chunk is dequantised once for all rows; otherwise groups of 8 rows run the
 * register-operand MMA kernel of kvq_decode_attention.  1: always the groups of 8.  2: the 128-row tile whenever the rows
 * fit it.  Workspace sizes and automatic split counts follow the choice
 * in force when they are computed: size the workspace after choosing.
 * KVQ_ERR_INVALID_ARG for another value.
 */
KVQ_API kvq_status kvq_set_verify_path(int32_t path);

/*
 * Position-axis mixed cache: an f16 window of the most recent tokens in front of a
 * quantised tail, "HAL #582 -- per-layer KV compression study", section 5 P2.  Two caches
 * of one shape (batch, n_kv_heads, head_dim) make the pair: `window` must be f16/f16, its
 * capacity W is the window length; `tail` has any K/V types and holds the older tokens.
 *
 * kvq_window_append: one new row per sequence, k and v fp32 [B][Hkv][D] (device, 16-byte
 * aligned).  The window is a ring (attention does not depend on key order): the new row
 * goes to slot (tail_len + window_len) mod W.  While the window is filling, window_len
 * grows; once it is full, the row in that slot is the oldest one: it is read back from
 * the window, quantised once into the tail at tail_len (the write path's
 * quantise-on-eviction; the tail quantises the window's f16 values), and then
 * overwritten, and tail_len grows.  Both lengths advance on the device, so the call can
 * be captured in a CUDA graph; the host mirrors advance too.  KVQ_ERR_CAPACITY (nothing
 * written) when a full window would evict into a full tail; KVQ_ERR_UNSUPPORTED when the
 * window is not f16/f16; KVQ_ERR_INVALID_ARG for mismatched shapes or the same cache twice.
 *
 * kvq_window_decode: decode attention of q [B][Hq][D] over the union of both regions
 * (window_len + tail_len rows per sequence), written like kvq_decode_attention.  Each
 * region is read by its own typed decode (the read path of section 5 P2) and the output is
 * the exact merge of both regions.  Normally one launch: its first splits read the window,
 * the rest the tail (the split count shared in proportion to the regions' capacity bytes,
 * a window byte weighted 2 with 256-wide heads and 1.75 with 128-wide ones), and all split
 * triples are merged as one set.  Where the tail's split count is below two,
 * two launches: the window's decode writes its normalised result into `workspace`, and the
 * tail's final merge takes that result as one more split triple.  `workspace`:
 * kvq_window_workspace_size bytes, zeroed once before its first use (as for
 * kvq_decode_attention); it also holds the eviction flags of kvq_window_append_decode
 * (one int32 per sequence and KV head, at its end).
 */
KVQ_API kvq_status kvq_window_append(kvq_cache *window, kvq_cache *tail, const float *k, const float *v,
                                     void *stream);
KVQ_API kvq_status kvq_window_workspace_size(const kvq_cache *window, const kvq_cache *tail, int32_t n_q_heads,
                                             size_t *bytes);
KVQ_API kvq_status kvq_window_decode(const kvq_cache *window, const kvq_cache *tail, const float *q,
                                     int32_t n_q_heads, float scale, void *workspace, float *out, float *lse,
                                     void *stream);

/*
 * One decode step of the window + tail pair: kvq_window_append of k, v followed by
 * kvq_window_decode of q, with the same arguments, results and errors, in one launch where
 * the two-region grid is resident at once (one CTA per SM: splits x Hkv x B <= the SM
 * count), a KV head has at most 8 query heads and the tail has at least two splits (as
 * chosen by kvq_decode_auto_splits) -- the read path's two regions then also take the write
 * path: the window's CTA that holds the new row's ring slot writes it there before reading
 * that tile, and, once the window is full, the tail's CTA that holds tail position tail_len
 * first moves the slot's old row there (quantised from its f16 value) and sets a flag in
 * `workspace` that the window's CTA waits for (bounded) before it overwrites the slot.
 * Otherwise the two calls run one after the other. `workspace`: kvq_window_workspace_size
 * bytes, zeroed once (the flags are left at zero; zero it again after a wait gave up, i.e.
 * after KVQ_DEVERR_TIMEOUT from a wait of about two seconds). Same section 5 P2 as above.
 */
KVQ_API kvq_status kvq_window_append_decode(kvq_cache *window, kvq_cache *tail, const float *k, const float *v,
                                            const float *q, int32_t n_q_heads, float scale, void *workspace,
                                            float *out, float *lse, void *stream);

/*
 * kvq_decode_attention without a caller-provided workspace.  (The pages have no
 * counterpart: this entry point exists for callers, not for the method.)
 *
 * Some callers cannot allocate device memory at the point where they decode: a plugin
 * whose host framework hands it only input and output pointers, a serving loop whose
 * allocator has already reserved every byte of HBM for cache pages, or code that must
 * not allocate while a CUDA graph is being captured.  This variant takes the same
 * arguments as kvq_decode_attention minus `workspace`, and uses instead a scratch array
 * compiled into the library as a file-scope __device__ variable of
 * KVQ_NOALLOC_SCRATCH_BYTES (8 MiB).  Every GPU on which the library's module is loaded
 * holds that array until the process exits.  The call itself performs no cudaMalloc,
 * cudaFree or other allocating call; the caller still passes q, out and lse.
 *
 * - The scratch needed is the kvq_decode_workspace_size of the same arguments; larger
 *   requests return KVQ_ERR_SCRATCH and launch nothing.
 * - The first call on a device looks up the array's device address for that device
 *   (cudaGetSymbolAddress, with that device current); make that first call before any
 *   stream capture.  Later calls only enqueue work.
 * - All calls share the one array, which keeps the contents of the last call.  The arrival
 *   counters at its front must start at zero: a call clears them (an asynchronous memset
 *   on `stream`, before its kernel) when its counter region reaches past the previous
 *   call's, whose split partials lie beyond that region; otherwise their arrival counts
 *   are zero already, since every finished decode leaves them at zero, and the call skips
 *   the clear.
 *   Calls that overlap on the GPU (different streams without ordering, or several host
 *   threads) race on the array and give wrong results.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)
KVQ_API kvq_status kvq_decode_attention_noalloc(const kvq_cache *cache, const float *q, int32_t n_q_heads,
                                                float scale, int32_t n_splits, float *out, float *lse,
                                                void *stream);

/*
 * Storage cost of one 32-value block of a type, in bytes: f16 64, q8_0 34, q4_0 18,
 * q4_1 20, q5_0 22, q5_1 24.  0 for an unknown type.
 * "HAL #582 -- per-layer KV compression study", section 1 and section 5 P1 (the P1
 * validation prices q5_1 K + q4_0 V at 2016 MiB for 32768 cells of the 14B shape).
 */
KVQ_API int32_t kvq_block_bytes(kvq_type type);

/*
 * Automatic KV tier at start-up, "HAL #582 -- per-layer KV compression study", section 5
 * P1: given the number of cache cells (all sequences), the model shape and the byte
 * budget for the KV cache, walk the ladder
 *     rung 0 f16/f16,  1 q8_0/q8_0,  2 q8_0 K/q4_0 V,  3 q5_1 K/q4_0 V (floor)
 * and choose the first (least compressing) rung whose whole cache,
 *     cells * n_layers * n_kv_heads * head_dim / 32 * (block_bytes(K) + block_bytes(V)),
 * is at most the budget; when none is, choose the floor and report fits = 0 (the caller
 * then spills or shortens the context).  The budget arithmetic itself (free memory,
 * memory already resident, reserve) is the caller's.  Host-only; no GPU call.
 * Errors: KVQ_ERR_INVALID_ARG for a null out, cells < 0, a non-positive shape, a
 * head_dim not a multiple of 32, or a size that overflows 64 bits.
 */
typedef struct {
    int32_t rung;     /* 0..3 as above                                             */
    kvq_type type_k;  /* chosen K type                                             */
    kvq_type type_v;  /* chosen V type                                             */
    int32_t fits;     /* 1 if bytes <= budget_bytes                                */
    uint64_t bytes;   /* whole-cache bytes of the chosen rung                      */
} kvq_tier_choice;
KVQ_API kvq_status kvq_select_tier(int64_t cells, int32_t n_layers, int32_t n_kv_heads, int32_t head_dim,
                                   uint64_t budget_bytes, kvq_tier_choice *out);

/*
 * Wait limit of the kernels' pipeline and merge waits, in SM clock cycles, for launches
 * enqueued after this call (process-wide).  0 restores the default (4e9 cycles, about two
 * seconds).  In the split-K decode kernels (decode, append-decode, partials, window + tail,
 * the 8-row verify groups) a wait that takes longer than the limit sets KVQ_DEVERR_TIMEOUT
 * in the cache's error word and goes on waiting; it gives up only at the default bound,
 * after which its CTA publishes an empty split triple, still takes its merge arrivals and
 * returns.  The 128-row verify tile gives up at the limit itself (its copies in flight land
 * first).  Either way the outputs of that launch are undefined, the workspace's arrival
 * counts end at zero and a later call on the same workspace is correct again.  For failure handling
 * and its tests: a short limit makes the error word report slow waits on a healthy GPU.
 * KVQ_ERR_INVALID_ARG for a negative value.
 */
KVQ_API kvq_status kvq_set_wait_limit(int64_t cycles);

/*
 * Launch timing for measurement (process-wide).  With buf non-NULL (device memory,
 * 16-byte aligned, n_slots * ctas_per_slot * 2 uint64), every split-K decode launch
 * enqueued afterwards (decode, fused append + decode, partials, 8-row verify groups,
 * no-alloc decode) takes the next of n_slots slots in turn, and CTA c of the launch
 * (linear index x + X * (y + Y * z), only c < ctas_per_slot) writes the GPU's global
 * nanosecond timer to buf[slot][c][0] when it starts and to buf[slot][c][1] when it exits.
 * Window + tail launches and the 128-row verify tile take a slot but write nothing.  A CUDA
 * graph keeps the slots assigned at capture.  buf NULL stops the stamps.
 * KVQ_ERR_INVALID_ARG for bad sizes or alignment.
 */
KVQ_API kvq_status kvq_set_launch_stamps(void *buf, int32_t n_slots, int32_t ctas_per_slot);

KVQ_API const char *kvq_status_string(kvq_status status);
KVQ_API int32_t kvq_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
