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
// already in it are kept.  One warp per row of the tile.
constexpr int kTileWarps = kTileRows;

template <int KT, int VT>
__global__ void __launch_bounds__(32 * kTileWarps) append_tiles_kernel(const AppendParams p, const int tiles_per_seq) {
    constexpr int KC = code_tile_bytes(KT), VC = code_tile_bytes(VT);
    constexpr int KS = scale_tile_bytes(KT), VS = scale_tile_bytes(VT);
    constexpr int BYTES = KC + VC + KS + VS;
    __shared__ __align__(16) uint8_t img[BYTES];
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, kt = threadIdx.x >> 5;
    const int NS = p.D / kSlice;
    const long long items = static_cast<long long>(p.nb) * p.Hkv * NS * tiles_per_seq;
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const int ti = static_cast<int>(it % tiles_per_seq);
        long long rest = it / tiles_per_seq;
        const int sl = static_cast<int>(rest % NS);
        rest /= NS;
        const int h = static_cast<int>(rest % p.Hkv);
        const int bl = static_cast<int>(rest / p.Hkv);
        const int bseq = p.b0 + bl;
        const int L = __ldcg(p.len + bseq);
        if (L < 0 || L + p.n_new > p.cap) continue;  // block-uniform: the last CTA reports it
        const int tile = (L >> 4) + ti;
        const int r0 = tile * kTileRows;               // first position of the tile
        if (r0 >= L + p.n_new) continue;               // past the append
        const size_t ts = ((static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles + tile) * NS + sl;
        uint8_t *gk = p.k_codes + ts * KC, *gv = p.v_codes + ts * VC;
        uint8_t *gks = KS ? p.k_scales + ts * KS : nullptr, *gvs = VS ? p.v_scales + ts * VS : nullptr;
        auto region = [&](int o, uint8_t *&g, int &off) {  // global place of image byte o
            if (o < KC) { g = gk; off = o; }
            else if (o < KC + VC) { g = gv; off = o - KC; }
            else if (o < KC + VC + KS) { g = gks; off = o - KC - VC; }
            else { g = gvs; off = o - KC - VC - KS; }
        };
        const bool partial = r0 < L || r0 + kTileRows > L + p.n_new;
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
        const int pos = r0 + kt;
        if (pos >= L && pos < L + p.n_new) {
            const size_t src = ((static_cast<size_t>(bl) * p.Hkv + h) * p.n_new + (pos - L)) * p.D + sl * kSlice + 4 * lane;
            const float4 xk = __ldcs(reinterpret_cast<const float4 *>(p.k + src));
            const float4 xv = __ldcs(reinterpret_cast<const float4 *>(p.v + src));
            quantize_store_vals<KT, false>(xk, img, img + KC + VC, kt, lane);
            quantize_store_vals<VT, true>(xv, img + KC, img + KC + VC + KS, kt, lane);
        }
        __syncthreads();
        for (int o = threadIdx.x * 16; o < BYTES; o += blockDim.x * 16) {
            uint8_t *g;
            int off;
            region(o, g, off);
            *reinterpret_cast<uint4 *>(g + off) = *reinterpret_cast<const uint4 *>(img + o);
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

template <int KT, int VT>
cudaError_t launch_append_t(const AppendParams &p, cudaStream_t stream) {
    if (p.n_new >= kTileRows) {
        // rows [L, L + n_new) cover (L % 16 + n_new - 1) / 16 + 1 tiles of a sequence, at
        // most (n_new + 14) / 16 + 1 (L % 16 = 15); items past the append return at once
        const int tiles_per_seq = (p.n_new + kTileRows - 2) / kTileRows + 1;
        const long long items = static_cast<long long>(p.nb) * p.Hkv * (p.D / kSlice) * tiles_per_seq;
        const long long blocks = items < 4 * 152 ? items : 4 * 152;
        append_tiles_kernel<KT, VT><<<static_cast<unsigned>(blocks), 32 * kTileWarps, 0, stream>>>(p, tiles_per_seq);
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
