// kvq_internal.cuh -- shared definitions of the CUDA path: tile geometry, the
// fragment-native placement of codes/scales, launch parameter blocks and PTX helpers.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"  // include/ is on the include path

namespace kvq {

constexpr int kTileRows = 16;    // positions per tile
constexpr int kSlice = 128;      // head-dim values per slice
constexpr int kBlock = 32;       // values per quantisation block
constexpr int kScaleTile = 128;  // scale bytes per (tile, slice): 16 rows x 4 blocks x 2 B
constexpr int kMaxSplits = 1024;

// groups of the two-level split merge: at most ceil(sqrt(n_splits)) groups
__host__ __device__ constexpr int max_merge_groups(int n_splits) {
    int g = 1;
    while (g * g < n_splits) ++g;
    return g + 1;
}
// first-level arrival counters per (sequence, KV head, row group): room for the largest
// split count, so that the counter region of a workspace does not move with n_splits
constexpr int kGroupCounterStride = max_merge_groups(kMaxSplits);
constexpr int kMaxRowsPerGroup = 8;  // query heads of one KV head handled per CTA

// per 16-row x 128-value tile slice: nibble types keep the q4_0 nibble layout (1024 B),
// 5-bit types add a 256-B plane of fifth bits; types with a minimum keep (d, lo) scales
__host__ __device__ constexpr bool has_fifth_bit(int type) { return type == KVQ_Q5_0 || type == KVQ_Q5_1; }
__host__ __device__ constexpr bool has_min(int type) { return type == KVQ_Q4_1 || type == KVQ_Q5_1; }
__host__ __device__ constexpr bool is_nibble_type(int type) {
    return type == KVQ_Q4_0 || type == KVQ_Q4_1 || type == KVQ_Q5_0 || type == KVQ_Q5_1;
}
constexpr int kNibbleBytes = 1024, kFifthBitBytes = 256;
__host__ __device__ constexpr int code_tile_bytes(int type) {
    return type == KVQ_Q8_0 ? 2048
                            : (type == KVQ_F16 ? 4096 : kNibbleBytes + (has_fifth_bit(type) ? kFifthBitBytes : 0));
}
__host__ __device__ constexpr int scale_tile_bytes(int type) {
    return type == KVQ_F16 ? 0 : (has_min(type) ? 2 * kScaleTile : kScaleTile);
}

// ---- placement inside one (tile, slice); see include/kvq.h for the contract ----
// pair order of a row inside the 16-row tile: j in [0,4), pos in {A=0,B=1,C=2,D=3}
__host__ __device__ inline void pair_slot(int kt, int &j, int &pos) {
    if (kt < 8) {
        j = kt >> 1;
        pos = kt & 1;
    } else {
        j = (kt - 8) >> 1;
        pos = 2 + (kt & 1);
    }
}
// byte position of pair member A,B,C,D inside a 4-byte V word (A,C,B,D order)
__host__ __device__ inline int vword_byte(int pos) { return pos == 0 ? 0 : (pos == 1 ? 2 : (pos == 2 ? 1 : 3)); }

// ---- decode launch parameters ----
struct DecodeParams {
    const uint8_t *k_codes, *k_scales, *v_codes, *v_scales;
    const int32_t *len;   // [B]
    int32_t *err;         // device error word
    const float *q;       // [B][Hq][D]
    float *out, *lse;     // [B][Hq][D], [B][Hq] or nullptr
    float *part_o, *part_m, *part_l;  // [B][Hq][part_stride][D], [B][Hq][part_stride]
    int part_stride, part_base;       // triples per row; slot of this launch's split 0
    int32_t *counters;    // [B][Hkv][QG] (fused mode) or nullptr (partials mode)
    int32_t *counters1;   // [B][Hkv][QG][kGroupCounterStride]: first-level group arrivals
    float *grp_o, *grp_m, *grp_l;  // [B][Hq][n_groups_max][D], [B][Hq][n_groups_max]
    int n_groups_max;
    int B, Hkv, Hq, G, QG, D;
    // queries per sequence: 1 for decode; up to 16 for a draft verify, query i of sequence b
    // attending to positions [0, len[b] - n_q + i] (causal within the draft).  The rows of a
    // (sequence, KV head) are ordered r = i * G + g and grouped 8 per CTA (QG groups).
    int n_q;
    // optional: a normalised result (out, natural-log lse per query row) over other keys,
    // merged exactly into this decode's output (the window of a window + tail cache)
    const float *ext_out, *ext_lse;
    int cap_tiles;
    int n_splits;
    float scale_log2;     // scale * log2(e)
    // fused quantise-on-append of one row per sequence (nullptr: attend only)
    const float *k_new, *v_new;  // [B][Hkv][D]
    int32_t *ticket;             // grid arrival ticket (state block); the last CTA advances len[]
    // 1: the previous kernel of the stream does not write this cache, so lengths and tiles
    // may be read before the programmatic-launch wait (set by the host, see kvq_api.cu)
    int early;
    // 1: the whole grid is resident at once (one wave), so the last CTAs of a row group may
    // wait for the others and share the merge of its splits (set at launch)
    int wide;
    // 0: the merge covers this launch's splits.  > 0: this launch is one region of a grid
    // whose merge_slots splits all publish a triple (empty ones too) at part_base + split of
    // part_stride slots per row, merged as one set.
    int merge_slots;
    // SM clock cycles after which a pipeline or merge wait reports KVQ_DEVERR_TIMEOUT
    // (kWaitCycles unless the caller set a limit with kvq_set_wait_limit)
    long long wait_cycles;
    // optional launch timing: CTA c (linear index < stamp_ctas) writes its %globaltimer at
    // its start and exit to stamps[2c], stamps[2c + 1]; nullptr: no stamps
    unsigned long long *stamps;
    int stamp_ctas;
    // Window + tail append in the two-region launch (kvq_window_append_decode).  win: 1 in
    // the window region's parameters, 2 in the tail's, 0 otherwise.  wl_len / tl_len and
    // wl_err / tl_err: the window's and the tail's lengths and error words; wl_cap / tl_cap
    // their capacities (rows); win_k / win_v: the window planes, where the tail region reads
    // the row it evicts; evict: [B][Hkv] flags in the workspace, set by the tail CTA that
    // has written an evicted row and cleared by the window CTA that then overwrites its slot.
    // ticket: the window's arrival ticket, shared by both regions.
    int win;
    int32_t *wl_len, *tl_len, *wl_err, *tl_err;
    int wl_cap, tl_cap;
    const uint8_t *win_k, *win_v;
    int32_t *evict;
};

struct AppendParams {
    uint8_t *k_codes, *k_scales, *v_codes, *v_scales;
    int32_t *len;     // [B]
    int32_t *ticket;  // one int
    int32_t *err;
    const float *k, *v;  // [nb][Hkv][n_new][D]
    int b0, nb, n_new, Hkv, D, cap, cap_tiles;
    int total_warps;
};

// rolling f16 window + quantised tail: one new row per sequence (kvq_window_append)
struct WindowParams {
    uint8_t *w_k, *w_v;                              // window planes (f16: codes only)
    uint8_t *t_kc, *t_ks, *t_vc, *t_vs;              // tail planes
    int32_t *w_len, *t_len, *ticket, *w_err, *t_err;
    const float *k, *v;                              // [B][Hkv][D]
    int B, Hkv, D, w_cap, w_cap_tiles, t_cap, t_cap_tiles;
    int total_warps;
};

struct CombineParams {
    const float *part_o, *part_m, *part_l;
    float *out, *lse;
    int rows, S, D;
};

// ---- PTX helpers ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d = A * B (accumulator input zero)
__device__ __forceinline__ void mma_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    const float z = 0.f;
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` SM clock cycles (default ~2 s) and returns false.
// Limits below kPollWaitCycles (failure-handling tests) poll with the non-suspending test,
// so that the give-up point does not depend on how long a suspended try_wait sleeps.
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz
constexpr long long kPollWaitCycles = 1000000LL;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit = kWaitCycles) {
    if (mbar_test_wait(bar, parity)) return true;
    const long long t0 = clock64();
    const bool poll = limit < kPollWaitCycles;
    while (true) {
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}

// Wait of the split-K decode kernels: 0 when the phase completed within `report` SM cycles,
// 1 when it completed later (the caller reports it), 2 when it did not complete within
// kWaitCycles (the caller gives up).  A short `report` limit thus flags a slow wait without
// abandoning it, so no copy is ever left in flight by a reported wait.
__device__ __forceinline__ int mbar_wait_timed(uint64_t *bar, uint32_t parity, long long report) {
    if (mbar_test_wait(bar, parity)) return 0;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return clock64() - t0 > report ? 1 : 0;
        if (clock64() - t0 > kWaitCycles) return 2;
    }
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Hint: pull [src, src + bytes) into L2 (bytes % 16 == 0, src 16-byte aligned).  No data
// reaches the SM and nothing waits on it; L2 stays coherent with later writes.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}


// 16-byte shared-memory load (ordinary load: the mbarrier waits carry memory clobbers)
__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// ---- block quantisers (one warp: 32 lanes x 4 values = one 128-value slice of a row) ----
// round half away from zero, written from the definition (|y - trunc(y)| is exact in fp32)
__device__ __forceinline__ float round_half_away(float y) {
    float t = truncf(y);
    float r = y - t;
    if (fabsf(r) >= 0.5f) t += copysignf(1.0f, y);
    return t;
}

// One row of one 128-value slice, lane l holding values 4l..4l+3 (v4), quantised and
// stored at row kt of the slice's tile (codes, scales: the slice's tile regions).
template <int T, bool IS_V>
__device__ __forceinline__ void quantize_store_vals(const float4 v4, uint8_t *codes, uint8_t *scales, int kt,
                                                    int lane) {
    const float xs[4] = {v4.x, v4.y, v4.z, v4.w};
    const int dd0 = 4 * lane;   // first value index of this lane inside the slice
    const int b = lane >> 3;    // quantisation block inside the slice
    const int i0 = dd0 & 31;    // index of the first value inside its block
    const int n = kt & 7, st = kt >> 3;
    int j, pos;
    pair_slot(kt, j, pos);

    if constexpr (T == KVQ_F16) {
        __half h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __float2half_rn(xs[e]);
        if constexpr (!IS_V) {
            const int jd = (dd0 & 15) >> 2, hd = i0 >> 4;
            // halves in the order (e0, e2, e1, e3): the two mma k-pairs of this lane
            __half2 p0 = __halves2half2(h[0], h[2]);
            __half2 p1 = __halves2half2(h[1], h[3]);
            uint2 w = make_uint2(h2_as_u32(p0), h2_as_u32(p1));
            *reinterpret_cast<uint2 *>(codes + (2 * b + st) * 512 + (4 * n + jd) * 16 + hd * 8) = w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = i0 + e, r = i & 15, hv = i >> 4, n2 = r >> 1;
                *reinterpret_cast<__half *>(codes + (2 * b + hv) * 512 + (4 * n2 + j) * 16 + (r & 1) * 8 + pos * 2) =
                    h[e];
            }
        }
        return;
    }

    if constexpr (T == KVQ_Q8_0) {
        float amax = fmaxf(fmaxf(fabsf(xs[0]), fabsf(xs[1])), fmaxf(fabsf(xs[2]), fabsf(xs[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const float d = __fdiv_rn(amax, 127.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        int c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // stored as a sign-magnitude byte
            const int q = static_cast<int>(round_half_away(__fmul_rn(xs[e], id)));
            c[e] = q < 0 ? (0x80 | -q) : q;
        }
        if constexpr (!IS_V) {
            const int jd = (dd0 & 15) >> 2, hd = i0 >> 4;
            const uint32_t w = (uint32_t(c[0]) & 0xffu) | ((uint32_t(c[1]) & 0xffu) << 8) |
                               ((uint32_t(c[2]) & 0xffu) << 16) | ((uint32_t(c[3]) & 0xffu) << 24);
            *reinterpret_cast<uint32_t *>(codes + b * 512 + (4 * n + jd) * 16 + (2 * st + hd) * 4) = w;
        } else {
            const int vb = vword_byte(pos);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = i0 + e, r = i & 15, hv = i >> 4, n2 = r >> 1;
                codes[b * 512 + (4 * n2 + j) * 16 + ((r & 1) + 2 * hv) * 4 + vb] = static_cast<uint8_t>(c[e] & 0xff);
            }
        }
        if ((lane & 7) == 0)
            *reinterpret_cast<__half *>(scales + j * 32 + b * 8 + pos * 2) = __float2half_rn(d);
        return;
    }

    if constexpr (is_nibble_type(T)) {
        int c[4];
        float d, lo = 0.f;
        if constexpr (!has_min(T)) {
            // q4_0 / q5_0: value of largest magnitude (the lowest index wins a tie), d = m / -K,
            // codes min(2K - 1, trunc(x / d + K + 1/2)) with K = 8 or 16
            constexpr float K = T == KVQ_Q4_0 ? 8.0f : 16.0f;
            constexpr int cmax = T == KVQ_Q4_0 ? 15 : 31;
            float best = xs[0], ba = fabsf(xs[0]);
            int bi = dd0;
#pragma unroll
            for (int e = 1; e < 4; ++e) {
                const float a = fabsf(xs[e]);
                if (a > ba) {
                    ba = a;
                    best = xs[e];
                    bi = dd0 + e;
                }
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                const float oba = __shfl_xor_sync(0xffffffffu, ba, off);
                const float obest = __shfl_xor_sync(0xffffffffu, best, off);
                const int obi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (oba > ba || (oba == ba && obi < bi)) {
                    ba = oba;
                    best = obest;
                    bi = obi;
                }
            }
            d = __fdiv_rn(best, -K);
            const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = static_cast<int>(__fadd_rn(__fmul_rn(xs[e], id), K + 0.5f));  // truncation
                c[e] = t < cmax ? t : cmax;
            }
        } else {
            // q4_1 / q5_1: lo = min, hi = max, d = (hi - lo) / L, codes min(L, trunc((x - lo) / d + 1/2))
            constexpr int L = T == KVQ_Q4_1 ? 15 : 31;
            lo = fminf(fminf(xs[0], xs[1]), fminf(xs[2], xs[3]));
            float hi = fmaxf(fmaxf(xs[0], xs[1]), fmaxf(xs[2], xs[3]));
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
                hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
            }
            d = __fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(L));
            const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = static_cast<int>(__fadd_rn(__fmul_rn(__fsub_rn(xs[e], lo), id), 0.5f));
                c[e] = t < L ? t : L;
            }
        }
        int chi[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) chi[e] = __shfl_down_sync(0xffffffffu, c[e], 4);
        if ((lane & 7) < 4) {
            // this lane holds values i0..i0+3 (< 16) and, from lane+4, values i0+16..i0+19:
            // low 4 bits in the nibbles; for 5-bit types the fifth bits go to the plane after
            // the nibbles: lane L's word of chunk b/2 holds, for nibble word wi of that lane,
            // byte e's low-nibble code at bit 8e + 4 + wi and its high-nibble code at bit 8e + wi
            uint32_t byte[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) byte[e] = uint32_t(c[e] & 15) | (uint32_t(chi[e] & 15) << 4);
            uint32_t *hb_chunk = reinterpret_cast<uint32_t *>(codes + kNibbleBytes + (b >> 1) * 128);
            if constexpr (!IS_V) {
                const int jb = lane & 7;  // bytes 4jb..4jb+3 of the block
                const uint32_t w = byte[0] | (byte[1] << 8) | (byte[2] << 16) | (byte[3] << 24);
                *reinterpret_cast<uint32_t *>(codes + (b >> 1) * 512 + (4 * n + jb) * 16 + (2 * (b & 1) + st) * 4) =
                    w;
                if constexpr (has_fifth_bit(T)) {
                    const int wi = 2 * (b & 1) + st;
                    uint32_t mask = 0, bits = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        mask |= (1u << (8 * e + 4 + wi)) | (1u << (8 * e + wi));
                        bits |= (uint32_t(c[e] >> 4) << (8 * e + 4 + wi)) | (uint32_t(chi[e] >> 4) << (8 * e + wi));
                    }
                    uint32_t *hw = hb_chunk + (4 * n + jb);
                    atomicAnd(hw, ~mask);  // the bits of other rows of the word are kept
                    atomicOr(hw, bits);
                }
            } else {
                const int vb = vword_byte(pos);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = i0 + e, n2 = r >> 1, qq = r & 1;
                    codes[(b >> 1) * 512 + (4 * n2 + j) * 16 + (2 * (b & 1) + qq) * 4 + vb] =
                        static_cast<uint8_t>(byte[e]);
                    if constexpr (has_fifth_bit(T)) {
                        const int wi = 2 * (b & 1) + qq;
                        const uint32_t mask = (1u << (8 * vb + 4 + wi)) | (1u << (8 * vb + wi));
                        const uint32_t bits =
                            (uint32_t(c[e] >> 4) << (8 * vb + 4 + wi)) | (uint32_t(chi[e] >> 4) << (8 * vb + wi));
                        uint32_t *hw = hb_chunk + (4 * n2 + j);
                        atomicAnd(hw, ~mask);
                        atomicOr(hw, bits);
                    }
                }
            }
        }
        if ((lane & 7) == 0) {
            *reinterpret_cast<__half *>(scales + j * 32 + b * 8 + pos * 2) = __float2half_rn(d);
            if constexpr (has_min(T))
                *reinterpret_cast<__half *>(scales + kScaleTile + j * 32 + b * 8 + pos * 2) = __float2half_rn(lo);
        }
        return;
    }
}

template <int T, bool IS_V>
__device__ __forceinline__ void quantize_store(const float *x, uint8_t *codes, uint8_t *scales, int kt, int lane) {
    quantize_store_vals<T, IS_V>(*reinterpret_cast<const float4 *>(x), codes, scales, kt, lane);
}

// The inverse of quantize_store_vals<KVQ_F16, IS_V>: values 4l..4l+3 of row kt of an f16
// tile slice, widened to fp32 (exact).
template <bool IS_V>
__device__ __forceinline__ float4 load_f16_row(const uint8_t *codes, int kt, int lane) {
    const int dd0 = 4 * lane, b = lane >> 3, i0 = dd0 & 31;
    const int n = kt & 7, st = kt >> 3;
    __half h[4];
    if constexpr (!IS_V) {
        const int jd = (dd0 & 15) >> 2, hd = i0 >> 4;
        const uint2 w = *reinterpret_cast<const uint2 *>(codes + (2 * b + st) * 512 + (4 * n + jd) * 16 + hd * 8);
        const __half2 p0 = u32_as_h2(w.x), p1 = u32_as_h2(w.y);  // (e0, e2), (e1, e3)
        h[0] = __low2half(p0);
        h[2] = __high2half(p0);
        h[1] = __low2half(p1);
        h[3] = __high2half(p1);
    } else {
        int j, pos;
        pair_slot(kt, j, pos);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = i0 + e, r = i & 15, hv = i >> 4, n2 = r >> 1;
            h[e] = *reinterpret_cast<const __half *>(codes + (2 * b + hv) * 512 + (4 * n2 + j) * 16 + (r & 1) * 8 +
                                                     pos * 2);
        }
    }
    return make_float4(__half2float(h[0]), __half2float(h[1]), __half2float(h[2]), __half2float(h[3]));
}

}  // namespace kvq

// launchers implemented in the .cu files
namespace kvq {
cudaError_t launch_append(int type_k, int type_v, const AppendParams &p, cudaStream_t stream);
cudaError_t launch_window_append(int tail_k, int tail_v, const WindowParams &p, cudaStream_t stream);
cudaError_t launch_verify(int type_k, int type_v, const DecodeParams &p, cudaStream_t stream);
// draft verify with all query rows of a (sequence, KV head) in one 128-row tensor-core tile
// (p.QG = 1, at most 128 rows); grid (n_splits, Hkv, B)
cudaError_t launch_verify_tc(int type_k, int type_v, const DecodeParams &p, cudaStream_t stream);
constexpr int kVerifyTileRows = 128;
cudaError_t launch_decode_ext(int type_k, int type_v, const DecodeParams &p, bool fused, cudaStream_t stream);
// one launch over an f16 window (params pw, splits [0, nw)) and a quantised tail (pt, the
// remaining pt.merge_slots - nw splits); cudaErrorNotSupported where it is not built
cudaError_t launch_window_dual(int tail_k, int tail_v, int D, const DecodeParams &pw, const DecodeParams &pt, int nw,
                               cudaStream_t stream);
cudaError_t launch_window_dual_ns1(int tail_k, int tail_v, const DecodeParams &pw, const DecodeParams &pt, int nw,
                                   cudaStream_t stream);
cudaError_t occupancy_ext(int type_k, int type_v, int D, int *ctas_per_sm);
// the (K, V) type pairs a cache may hold: every pair of f16 / q8_0 / q4_0, plus these
__host__ __device__ constexpr bool is_base_type(int t) { return t == KVQ_F16 || t == KVQ_Q8_0 || t == KVQ_Q4_0; }
__host__ __device__ constexpr bool is_ext_pair(int tk, int tv) {
    return (tk == KVQ_Q8_0 && tv == KVQ_Q5_0) || (tk == KVQ_Q5_0 && tv == KVQ_Q5_0) ||
           (tk == KVQ_Q5_1 && tv == KVQ_Q5_1) || (tk == KVQ_Q4_1 && tv == KVQ_Q4_1) ||
           (tk == KVQ_Q5_1 && tv == KVQ_Q4_0);
}
cudaError_t verify_occupancy(int type_k, int type_v, int D, int *ctas_per_sm);
cudaError_t launch_decode(int type_k, int type_v, const DecodeParams &p, bool fused, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
cudaError_t decode_occupancy(int type_k, int type_v, int D, int *ctas_per_sm, int *n_sms);
}  // namespace kvq
