// kvq_append.cu -- quantise-on-append: fp32 K/V rows -> q8_0 / q4_0 / f16 cache tiles.
//
// The write path of "HAL #582 -- per-layer KV compression study", section 5 P2: each new
// token is quantised once, when it is written, by a GPU kernel.  One warp handles one
// (sequence, KV head, row, 128-value slice) for both K and V: lane l owns values
// 4l..4l+3, so a quantisation block of 32 values is 8 lanes and its max-abs is an
// 8-lane shuffle reduction.  Codes are then stored at their fragment-native places
// (include/kvq.h).  The last CTA to finish advances len[b] on the device, so the
// launch can be replayed inside a CUDA graph.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

// Items (row, KV head, slice) per warp and round: their fp32 values are all loaded before
// any is quantised, so that several rows' loads are in flight per warp.
constexpr int kAppendBatch = 8;
constexpr int kAppendWarps = 8;  // warps per CTA

template <int KT, int VT>
__global__ void __launch_bounds__(32 * kAppendWarps) append_kernel(const AppendParams p) {
    __shared__ int s_last;
    const int lane = threadIdx.x & 31;
    const int NS = p.D / kSlice;
    const int n_warps = gridDim.x * kAppendWarps;  // grid-stride over the items
    for (int base = blockIdx.x * kAppendWarps + (threadIdx.x >> 5); base < p.total_warps;
         base += kAppendBatch * n_warps) {
        float4 xk[kAppendBatch], xv[kAppendBatch];
        size_t tile_slice[kAppendBatch];
        int kt[kAppendBatch];
        bool ok[kAppendBatch];
#pragma unroll
        for (int u = 0; u < kAppendBatch; ++u) {
            const int item = base + u * n_warps;
            ok[u] = false;
            if (item < p.total_warps) {
                const int sl = item % NS;
                int rest = item / NS;
                const int row = rest % p.n_new;
                rest /= p.n_new;
                const int h = rest % p.Hkv;
                const int bl = rest / p.Hkv;
                const int bseq = p.b0 + bl;
                const int L = __ldcg(p.len + bseq);
                if (L >= 0 && L + p.n_new <= p.cap) {
                    const int pos = L + row;
                    tile_slice[u] = ((static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles + (pos >> 4)) * NS + sl;
                    kt[u] = pos & 15;
                    const size_t src =
                        ((static_cast<size_t>(bl) * p.Hkv + h) * p.n_new + row) * p.D + sl * kSlice + 4 * lane;
                    xk[u] = __ldcs(reinterpret_cast<const float4 *>(p.k + src));
                    xv[u] = __ldcs(reinterpret_cast<const float4 *>(p.v + src));
                    ok[u] = true;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kAppendBatch; ++u) {
            if (!ok[u]) continue;  // warp-uniform: every lane has the same item
            quantize_store_vals<KT, false>(xk[u], p.k_codes + tile_slice[u] * code_tile_bytes(KT),
                                           p.k_scales + tile_slice[u] * scale_tile_bytes(KT), kt[u], lane);
            quantize_store_vals<VT, true>(xv[u], p.v_codes + tile_slice[u] * code_tile_bytes(VT),
                                          p.v_scales + tile_slice[u] * scale_tile_bytes(VT), kt[u], lane);
        }
    }
    // the last CTA (all others have read len[] by now) advances the lengths
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int t = atomicAdd(p.ticket, 1);
        s_last = (t == static_cast<int>(gridDim.x) - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int i = threadIdx.x; i < p.nb; i += blockDim.x) {
            const int bseq = p.b0 + i;
            const int L = __ldcg(p.len + bseq);
            if (L >= 0 && L + p.n_new <= p.cap)
                p.len[bseq] = L + p.n_new;
            else
                atomicOr(p.err, KVQ_DEVERR_CAPACITY);
        }
        if (threadIdx.x == 0) *p.ticket = 0;
    }
}

// Bulk appends (n_new >= 16 rows): whole 16-row tile slices are assembled in shared
// memory and written out with 16-byte stores.  In the fragment-native layout the codes of
// one row are interleaved with those of other rows of its tile (a V word holds four rows),
// so writing row by row means byte stores scattered over the tile; assembling the tile
// first turns them into coalesced stores.  One item = (sequence, KV head, slice, tile of
// the append); a tile that the append covers only in part is first read back, so the rows
// already in it are kept.  One thread quantises one 32-value block (of K or of V) of one
// row: its maximum search and its two divisions are done once per block, with no shuffles.
// The arithmetic is that of quantize_store_vals, operation for operation.
template <int T, bool IS_V>
__device__ __forceinline__ void quantize_block_store(const float (&x)[kBlock], uint8_t *codes, uint8_t *scales,
                                                     int kt, int b) {
    const int n = kt & 7, st = kt >> 3;
    int j, pos;
    pair_slot(kt, j, pos);
    if constexpr (T == KVQ_F16) {
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
            const __half h0 = __float2half_rn(x[4 * g4]), h1 = __float2half_rn(x[4 * g4 + 1]);
            const __half h2 = __float2half_rn(x[4 * g4 + 2]), h3 = __float2half_rn(x[4 * g4 + 3]);
            if constexpr (!IS_V) {
                const uint2 w = make_uint2(h2_as_u32(__halves2half2(h0, h2)), h2_as_u32(__halves2half2(h1, h3)));
                *reinterpret_cast<uint2 *>(codes + (2 * b + st) * 512 + (4 * n + (g4 & 3)) * 16 + (g4 >> 2) * 8) = w;
            } else {
                const __half hv[4] = {h0, h1, h2, h3};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 4 * g4 + e, r = i & 15, hh = i >> 4, n2 = r >> 1;
                    *reinterpret_cast<__half *>(codes + (2 * b + hh) * 512 + (4 * n2 + j) * 16 + (r & 1) * 8 + pos * 2) =
                        hv[e];
                }
            }
        }
        return;
    }
    if constexpr (T == KVQ_Q8_0) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kBlock; ++i) amax = fmaxf(amax, fabsf(x[i]));
        const float d = __fdiv_rn(amax, 127.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        uint32_t c[kBlock];
#pragma unroll
        for (int i = 0; i < kBlock; ++i) {  // stored as a sign-magnitude byte
            const int q = static_cast<int>(round_half_away(__fmul_rn(x[i], id)));
            c[i] = static_cast<uint32_t>(q < 0 ? (0x80 | -q) : q) & 0xffu;
        }
        if constexpr (!IS_V) {
#pragma unroll
            for (int g4 = 0; g4 < 8; ++g4)
                *reinterpret_cast<uint32_t *>(codes + b * 512 + (4 * n + (g4 & 3)) * 16 + (2 * st + (g4 >> 2)) * 4) =
                    c[4 * g4] | (c[4 * g4 + 1] << 8) | (c[4 * g4 + 2] << 16) | (c[4 * g4 + 3] << 24);
        } else {
            const int vb = vword_byte(pos);
#pragma unroll
            for (int i = 0; i < kBlock; ++i) {
                const int r = i & 15, hv = i >> 4, n2 = r >> 1;
                codes[b * 512 + (4 * n2 + j) * 16 + ((r & 1) + 2 * hv) * 4 + vb] = static_cast<uint8_t>(c[i]);
            }
        }
        *reinterpret_cast<__half *>(scales + j * 32 + b * 8 + pos * 2) = __float2half_rn(d);
        return;
    }
    if constexpr (is_nibble_type(T)) {
        int c[kBlock];
        float d, lo = 0.f;
        if constexpr (!has_min(T)) {
            // value of largest magnitude, the lowest index on ties; d = m / -K; codes
            // min(2K - 1, trunc(x / d + K + 1/2)) with K = 8 (q4_0) or 16 (q5_0)
            constexpr float K = T == KVQ_Q4_0 ? 8.0f : 16.0f;
            constexpr int cmax = T == KVQ_Q4_0 ? 15 : 31;
            float best = x[0], ba = fabsf(x[0]);
#pragma unroll
            for (int i = 1; i < kBlock; ++i) {
                const float a = fabsf(x[i]);
                if (a > ba) {
                    ba = a;
                    best = x[i];
                }
            }
            d = __fdiv_rn(best, -K);
            const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
            for (int i = 0; i < kBlock; ++i) {
                const int t = static_cast<int>(__fadd_rn(__fmul_rn(x[i], id), K + 0.5f));  // truncation
                c[i] = t < cmax ? t : cmax;
            }
        } else {
            // lo = min, hi = max, d = (hi - lo) / L, codes min(L, trunc((x - lo) / d + 1/2))
            constexpr int L = T == KVQ_Q4_1 ? 15 : 31;
            float hi = x[0];
            lo = x[0];
#pragma unroll
            for (int i = 1; i < kBlock; ++i) {
                lo = fminf(lo, x[i]);
                hi = fmaxf(hi, x[i]);
            }
            d = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(L));
            const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
            for (int i = 0; i < kBlock; ++i) {
                const int t = static_cast<int>(__fadd_rn(__fmul_rn(__fsub_rn(x[i], lo), id), 0.5f));
                c[i] = t < L ? t : L;
            }
        }
        // low 4 bits in the nibble bytes (value i in the low nibble, i + 16 in the high one);
        // for 5-bit types the fifth bits in the plane after the nibbles (bit positions as in
        // quantize_store_vals; other rows' bits of a word are kept)
        uint32_t *hb_chunk = reinterpret_cast<uint32_t *>(codes + kNibbleBytes + (b >> 1) * 128);
        if constexpr (!IS_V) {
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                uint32_t w = 0, mask = 0, bits = 0;
                const int wi = 2 * (b & 1) + st;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int lo_c = c[4 * g4 + e], hi_c = c[4 * g4 + 16 + e];
                    w |= (uint32_t(lo_c & 15) | (uint32_t(hi_c & 15) << 4)) << (8 * e);
                    mask |= (1u << (8 * e + 4 + wi)) | (1u << (8 * e + wi));
                    bits |= (uint32_t(lo_c >> 4) << (8 * e + 4 + wi)) | (uint32_t(hi_c >> 4) << (8 * e + wi));
                }
                *reinterpret_cast<uint32_t *>(codes + (b >> 1) * 512 + (4 * n + g4) * 16 + (2 * (b & 1) + st) * 4) = w;
                if constexpr (has_fifth_bit(T)) {
                    atomicAnd(hb_chunk + (4 * n + g4), ~mask);
                    atomicOr(hb_chunk + (4 * n + g4), bits);
                }
            }
        } else {
            const int vb = vword_byte(pos);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int n2 = i >> 1, qq = i & 1;
                codes[(b >> 1) * 512 + (4 * n2 + j) * 16 + (2 * (b & 1) + qq) * 4 + vb] =
                    static_cast<uint8_t>(uint32_t(c[i] & 15) | (uint32_t(c[i + 16] & 15) << 4));
                if constexpr (has_fifth_bit(T)) {
                    const int wi = 2 * (b & 1) + qq;
                    const uint32_t mask = (1u << (8 * vb + 4 + wi)) | (1u << (8 * vb + wi));
                    const uint32_t bits = (uint32_t(c[i] >> 4) << (8 * vb + 4 + wi)) | (uint32_t(c[i + 16] >> 4) << (8 * vb + wi));
                    atomicAnd(hb_chunk + (4 * n2 + j), ~mask);
                    atomicOr(hb_chunk + (4 * n2 + j), bits);
                }
            }
        }
        *reinterpret_cast<__half *>(scales + j * 32 + b * 8 + pos * 2) = __float2half_rn(d);
        if constexpr (has_min(T)) *reinterpret_cast<__half *>(scales + kScaleTile + j * 32 + b * 8 + pos * 2) = __float2half_rn(lo);
        return;
    }
}

// threads of a tile CTA: one per (K or V, row, block): 2 x 16 x 4
constexpr int kTileThreads = 2 * kTileRows * (kSlice / kBlock);

// CTAs of the tile kernel per SM: each loops over items; every thread copies its 32 input
// values of the next item into its own shared-memory slot (asynchronous 16-byte copies)
// while it quantises the current one, so that every CTA keeps a load in flight without
// holding it in registers
constexpr int kTileCtasPerSm = 6;

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <int KT, int VT>
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm) append_tiles_kernel(const AppendParams p,
                                                                                    const int tiles_per_seq) {
    constexpr int KC = code_tile_bytes(KT), VC = code_tile_bytes(VT);
    constexpr int KS = scale_tile_bytes(KT), VS = scale_tile_bytes(VT);
    constexpr int BYTES = KC + VC + KS + VS;
    __shared__ __align__(16) uint8_t img[BYTES];
    // each thread's 8 input chunks of 16 bytes, chunk i at place i ^ (thread mod 8), so that
    // the 8 threads of a 128-bit shared access touch 8 different bank groups
    __shared__ __align__(16) float4 stage[kTileThreads * (kBlock / 4)];
    __shared__ int s_last;
    const bool is_v = threadIdx.x >= kTileThreads / 2;  // warp-uniform
    const int rb = threadIdx.x % (kTileThreads / 2);
    const int kt = rb >> 2, b = rb & 3;                 // row of the tile, block of the slice
    const int NS = p.D / kSlice;
    const long long items = static_cast<long long>(p.nb) * p.Hkv * NS * tiles_per_seq;
    float4 *slot = stage + threadIdx.x * (kBlock / 4);
    const int swz = threadIdx.x & 7;
    // An item's tile slice (ts), its first position r0, the sequence's length L and this
    // thread's 32 input values (src: nullptr where its row is not appended); false for an
    // item with nothing to write (past the append, or a sequence without room, which the
    // last CTA reports).
    struct Item {
        size_t ts;
        int r0, L;
        const float4 *src;
    };
    auto locate = [&](long long it, Item &m) -> bool {
        const int ti = static_cast<int>(it % tiles_per_seq);
        long long rest = it / tiles_per_seq;
        const int sl = static_cast<int>(rest % NS);
        rest /= NS;
        const int h = static_cast<int>(rest % p.Hkv);
        const int bl = static_cast<int>(rest / p.Hkv);
        const int bseq = p.b0 + bl;
        m.L = __ldcg(p.len + bseq);
        if (m.L < 0 || m.L + p.n_new > p.cap) return false;
        const int tile = (m.L >> 4) + ti;
        m.r0 = tile * kTileRows;
        if (m.r0 >= m.L + p.n_new) return false;
        m.ts = ((static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles + tile) * NS + sl;
        const int pos = m.r0 + kt;
        m.src = nullptr;
        if (pos >= m.L && pos < m.L + p.n_new)
            m.src = reinterpret_cast<const float4 *>(
                (is_v ? p.v : p.k) +
                ((static_cast<size_t>(bl) * p.Hkv + h) * p.n_new + (pos - m.L)) * p.D + sl * kSlice + kBlock * b);
        return true;
    };
    auto prefetch = [&](const float4 *src) {
#pragma unroll
        for (int i = 0; i < kBlock / 4; ++i) cp_async16(slot + (i ^ swz), src + i);
        cp_async_commit();
    };
    long long it = blockIdx.x;
    Item cur{};
    bool live = it < items && locate(it, cur);
    if (live && cur.src) prefetch(cur.src);
    while (it < items) {
        float x[kBlock];
        if (live && cur.src) {  // this thread's own slot only: no barrier needed
            cp_async_wait_all();
#pragma unroll
            for (int i = 0; i < kBlock / 4; ++i) {
                const float4 v = slot[i ^ swz];
                x[4 * i] = v.x;
                x[4 * i + 1] = v.y;
                x[4 * i + 2] = v.z;
                x[4 * i + 3] = v.w;
            }
        }
        // the next item's values are requested before this one is quantised
        const long long nx = it + gridDim.x;
        Item nxt{};
        const bool live_n = nx < items && locate(nx, nxt);
        if (live_n && nxt.src) prefetch(nxt.src);
        if (live) {  // block-uniform
            uint8_t *gk = p.k_codes + cur.ts * KC, *gv = p.v_codes + cur.ts * VC;
            uint8_t *gks = KS ? p.k_scales + cur.ts * KS : nullptr, *gvs = VS ? p.v_scales + cur.ts * VS : nullptr;
            auto region = [&](int o, uint8_t *&g, int &off) {  // global place of image byte o
                if (o < KC) { g = gk; off = o; }
                else if (o < KC + VC) { g = gv; off = o - KC; }
                else if (o < KC + VC + KS) { g = gks; off = o - KC - VC; }
                else { g = gvs; off = o - KC - VC - KS; }
            };
            const bool partial = cur.r0 < cur.L || cur.r0 + kTileRows > cur.L + p.n_new;
            __syncthreads();  // the previous item's image has been written out
            if (partial) {    // keep the rows of the tile that this append does not write
                for (int o = threadIdx.x * 16; o < BYTES; o += blockDim.x * 16) {
                    uint8_t *g;
                    int off;
                    region(o, g, off);
                    *reinterpret_cast<uint4 *>(img + o) = __ldcg(reinterpret_cast<const uint4 *>(g + off));
                }
                __syncthreads();
            }
            if (cur.src) {
                if (!is_v)
                    quantize_block_store<KT, false>(x, img, img + KC + VC, kt, b);
                else
                    quantize_block_store<VT, true>(x, img + KC, img + KC + VC + KS, kt, b);
            }
            __syncthreads();
            for (int o = threadIdx.x * 16; o < BYTES; o += blockDim.x * 16) {
                uint8_t *g;
                int off;
                region(o, g, off);
                *reinterpret_cast<uint4 *>(g + off) = *reinterpret_cast<const uint4 *>(img + o);
            }
        }
        it = nx;
        live = live_n;
        cur = nxt;
    }
    // the last CTA (all others have read len[] by now) advances the lengths
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int t = atomicAdd(p.ticket, 1);
        s_last = (t == static_cast<int>(gridDim.x) - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int i = threadIdx.x; i < p.nb; i += blockDim.x) {
            const int bseq = p.b0 + i;
            const int L = __ldcg(p.len + bseq);
            if (L >= 0 && L + p.n_new <= p.cap)
                p.len[bseq] = L + p.n_new;
            else
                atomicOr(p.err, KVQ_DEVERR_CAPACITY);
        }
        if (threadIdx.x == 0) *p.ticket = 0;
    }
}

template <int KT, int VT>
cudaError_t launch_append_t(const AppendParams &p, cudaStream_t stream) {
    if (p.n_new >= kTileRows) {
        // rows [L, L + n_new) cover (L % 16 + n_new - 1) / 16 + 1 tiles of a sequence, at
        // most (n_new + 14) / 16 + 1 (L % 16 = 15); items past the append return at once
        const int tiles_per_seq = (p.n_new + kTileRows - 2) / kTileRows + 1;
        const long long items = static_cast<long long>(p.nb) * p.Hkv * (p.D / kSlice) * tiles_per_seq;
        const long long blocks = items < kTileCtasPerSm * 152 ? items : kTileCtasPerSm * 152;
        append_tiles_kernel<KT, VT><<<static_cast<unsigned>(blocks), kTileThreads, 0, stream>>>(p, tiles_per_seq);
        return cudaGetLastError();
    }
    // enough CTAs for about two rounds of batches on 152 SMs; small appends get one
    // batch per warp (a one-row decode-step append is one CTA)
    const long long per_cta = static_cast<long long>(kAppendWarps) * kAppendBatch;
    long long blocks = (p.total_warps + per_cta - 1) / per_cta;
    if (blocks > 8 * 152) blocks = 8 * 152;
    if (blocks < 1) blocks = 1;
    append_kernel<KT, VT><<<static_cast<unsigned>(blocks), 32 * kAppendWarps, 0, stream>>>(p);
    return cudaGetLastError();
}

// Rolling f16 window + quantised tail ("HAL #582 -- per-layer KV compression study",
// section 5 P2 write path): one new row per sequence.  The window is a ring of w_cap rows
// (attention does not depend on key order); the row written now goes to slot
// (tail_len + window_len) mod w_cap.  When the window is full, the row in that slot is the
// oldest: it is read back from the window, quantised once into the tail at tail_len, and
// only then overwritten.  One warp per (sequence, KV head, slice); the last CTA advances
// the lengths (window_len up to w_cap, then tail_len).
template <int TK, int TV>
__global__ void __launch_bounds__(256) window_append_kernel(const WindowParams p) {
    __shared__ int s_last;
    // Programmatic dependent launch: everything below reads what the previous kernel of the
    // stream may write, so wait for it first; the next kernel (the window's decode) may then
    // start its own pre-wait part, which reads nothing this kernel writes.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int wg = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int NS = p.D / kSlice;
    if (wg < p.total_warps) {
        const int sl = wg % NS;
        const int rest = wg / NS;
        const int h = rest % p.Hkv, b = rest / p.Hkv;
        const int Lw = __ldcg(p.w_len + b), Lt = __ldcg(p.t_len + b);
        const bool full = Lw >= p.w_cap;
        if (Lw >= 0 && Lw <= p.w_cap && Lt >= 0 && (!full || Lt + 1 <= p.t_cap)) {
            const int slot = static_cast<int>((static_cast<long long>(Lt) + Lw) % p.w_cap);
            const size_t wtile = (static_cast<size_t>(b) * p.Hkv + h) * p.w_cap_tiles + (slot >> 4);
            const int wkt = slot & 15;
            uint8_t *wk = p.w_k + (wtile * NS + sl) * code_tile_bytes(KVQ_F16);
            uint8_t *wv = p.w_v + (wtile * NS + sl) * code_tile_bytes(KVQ_F16);
            if (full) {
                const float4 xk = load_f16_row<false>(wk, wkt, lane);
                const float4 xv = load_f16_row<true>(wv, wkt, lane);
                const size_t ttile = (static_cast<size_t>(b) * p.Hkv + h) * p.t_cap_tiles + (Lt >> 4);
                const int tkt = Lt & 15;
                quantize_store_vals<TK, false>(xk, p.t_kc + (ttile * NS + sl) * code_tile_bytes(TK),
                                               p.t_ks + (ttile * NS + sl) * scale_tile_bytes(TK), tkt, lane);
                quantize_store_vals<TV, true>(xv, p.t_vc + (ttile * NS + sl) * code_tile_bytes(TV),
                                              p.t_vs + (ttile * NS + sl) * scale_tile_bytes(TV), tkt, lane);
            }
            const size_t src = (static_cast<size_t>(b) * p.Hkv + h) * p.D + sl * kSlice + 4 * lane;
            quantize_store<KVQ_F16, false>(p.k + src, wk, nullptr, wkt, lane);
            quantize_store<KVQ_F16, true>(p.v + src, wv, nullptr, wkt, lane);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int t = atomicAdd(p.ticket, 1);
        s_last = (t == static_cast<int>(gridDim.x) - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
            const int Lw = __ldcg(p.w_len + b), Lt = __ldcg(p.t_len + b);
            if (Lw < 0 || Lw > p.w_cap || Lt < 0) {
                atomicOr(p.w_err, KVQ_DEVERR_CAPACITY);
            } else if (Lw < p.w_cap) {
                p.w_len[b] = Lw + 1;
            } else if (Lt + 1 <= p.t_cap) {
                p.t_len[b] = Lt + 1;
            } else {
                atomicOr(p.t_err, KVQ_DEVERR_CAPACITY);
            }
        }
        if (threadIdx.x == 0) *p.ticket = 0;
    }
}

template <int TK, int TV>
cudaError_t launch_window_t(const WindowParams &p, cudaStream_t stream) {
    const int warps_per_block = 8;
    const int blocks = (p.total_warps + warps_per_block - 1) / warps_per_block;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(32 * warps_per_block);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, window_append_kernel<TK, TV>, p);
}

}  // namespace

cudaError_t launch_window_append(int tail_k, int tail_v, const WindowParams &p, cudaStream_t stream) {
#define KVQ_WINDOW_CASE(KT, VT) \
    if (tail_k == KT && tail_v == VT) return launch_window_t<KT, VT>(p, stream);
    KVQ_WINDOW_CASE(KVQ_F16, KVQ_F16)
    KVQ_WINDOW_CASE(KVQ_F16, KVQ_Q8_0)
    KVQ_WINDOW_CASE(KVQ_F16, KVQ_Q4_0)
    KVQ_WINDOW_CASE(KVQ_Q8_0, KVQ_F16)
    KVQ_WINDOW_CASE(KVQ_Q8_0, KVQ_Q8_0)
    KVQ_WINDOW_CASE(KVQ_Q8_0, KVQ_Q4_0)
    KVQ_WINDOW_CASE(KVQ_Q4_0, KVQ_F16)
    KVQ_WINDOW_CASE(KVQ_Q4_0, KVQ_Q8_0)
    KVQ_WINDOW_CASE(KVQ_Q4_0, KVQ_Q4_0)
#undef KVQ_WINDOW_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_append(int type_k, int type_v, const AppendParams &p, cudaStream_t stream) {
#define KVQ_APPEND_CASE(KT, VT) \
    if (type_k == KT && type_v == VT) return launch_append_t<KT, VT>(p, stream);
    KVQ_APPEND_CASE(KVQ_F16, KVQ_F16)
    KVQ_APPEND_CASE(KVQ_F16, KVQ_Q8_0)
    KVQ_APPEND_CASE(KVQ_F16, KVQ_Q4_0)
    KVQ_APPEND_CASE(KVQ_Q8_0, KVQ_F16)
    KVQ_APPEND_CASE(KVQ_Q8_0, KVQ_Q8_0)
    KVQ_APPEND_CASE(KVQ_Q8_0, KVQ_Q4_0)
    KVQ_APPEND_CASE(KVQ_Q4_0, KVQ_F16)
    KVQ_APPEND_CASE(KVQ_Q4_0, KVQ_Q8_0)
    KVQ_APPEND_CASE(KVQ_Q4_0, KVQ_Q4_0)
    KVQ_APPEND_CASE(KVQ_Q8_0, KVQ_Q5_0)
    KVQ_APPEND_CASE(KVQ_Q5_0, KVQ_Q5_0)
    KVQ_APPEND_CASE(KVQ_Q5_1, KVQ_Q5_1)
    KVQ_APPEND_CASE(KVQ_Q4_1, KVQ_Q4_1)
    KVQ_APPEND_CASE(KVQ_Q5_1, KVQ_Q4_0)
#undef KVQ_APPEND_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvq
