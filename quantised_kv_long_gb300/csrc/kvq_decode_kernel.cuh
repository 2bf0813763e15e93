// kvq_decode_kernel.cuh -- the split-K decode kernel template shared by the decode
// (one query per sequence) and draft-verify (several queries per sequence) entry points.
//
// Method: single-token grouped-query decode attention with the keys of each (sequence,
// KV head) split into contiguous ranges; each range is attended with an online softmax
// in fp32 and the ranges are merged exactly ("HAL #582 -- per-layer KV compression
// study", section 5 P2 read path: the softmax partials of ranges combine without loss).
// The K/V blocks are
// dequantised in registers while they are read, which is the cure the same study
// (section 3b, finding 2) gives for a quantised reader that was kernel-bound: throughput
// has to follow the bytes moved.
//
// GB300 mapping (one CTA per (split, KV head, sequence x row-group), one CTA per SM):
//   * warp 0 (producer): 1-D bulk copies (cp.async.bulk, TMA engine) of a run of whole
//     16-row tiles per stage into a shared-memory ring of two or three stages; completion
//     on mbarriers; every wait is bounded and reports KVQ_DEVERR_TIMEOUT instead of hanging.
//   * consumer warps (11 tile-warps for 128-wide heads with quantised keys, 8 for f16
//     keys, 4 slice-warp pairs for 256-wide heads): each owns two tiles (and one 128-value
//     slice) per stage.  Tiles are
//     stored fragment-native (include/kvq.h), so every lane fetches its mma operands
//     with 16-byte shared loads, converts codes to exact f16 integers with bit tricks
//     (no I2F), and runs mma.sync m16n8k16 (f16 in, fp32 accumulate).
//     S = Q K^T: A = [Q_hi ; Q_lo] (M rows 0-7 / 8-15 = up to 8 query heads split into
//     f16 hi + lo parts, so Q loses nothing; built once per slice in shared memory and
//     read by every tile-warp), B = K codes (exact), one accumulator per 32-value block,
//     multiplied by the f16 scale afterwards in fp32.
//     O += P V: the S accumulator layout is the A layout of the next mma, so P never
//     leaves registers; the V scale of each (row, block) is folded into P, which is
//     again split into f16 hi + lo rows.
//   * the CTA merges its warps in shared memory and writes one split triple; the splits
//     of each (sequence, KV head, row-group) are merged after an arrival counter: by the
//     last CTA, by the last few CTAs column by column when the grid is resident at once,
//     or in two levels (split_merge).  dual_kernel runs an f16 window and a quantised
//     tail of the same sequences in one grid and one merge.
#pragma once
#include <math_constants.h>

#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kTau = 8.0f;  // lazy-rescale threshold (log2 units): p <= 2^8 between rescales

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// f32 pair -> (f16 hi pair, f16 lo pair) with hi + lo == x to ~2^-22 relative
__device__ __forceinline__ void split_hi_lo(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    hi = h2_as_u32(h);
    lo = h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

// ---- codes as f16 subnormals ----
// Code words become mma operands with a permute and a mask.  A q8_0 code is stored as a
// sign-magnitude byte (bit 7 sign, bits 0..6 |q|); placing the magnitude in the low bits
// of an f16 half and the sign in bit 15 gives the subnormal q * 2^-24.  A q4_0 low nibble
// c in the low bits is c * 2^-24 and a high nibble (bits 4..7) is 16c * 2^-24; the offset
// 8 times the sum of the other operand is removed afterwards.  mma.sync multiplies f16
// subnormals exactly, so the accumulators hold exact dot products in units of 2^-24 (or
// 2^-20), and the unit is folded into one final multiply.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt(uint32_t a) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;\n" : "=r"(d) : "r"(a), "n"(SEL));
    return d;
}
// bytes 0, 2 / 1, 3 of a word of q8_0 codes as two f16 halves: byte, then its sign
// replicated (selector nibble with bit 3 set), masked to sign bit and magnitude
__device__ __forceinline__ uint32_t q8_02(uint32_t w) { return prmt<0xA280u>(w) & 0x807f807fu; }
__device__ __forceinline__ uint32_t q8_13(uint32_t w) { return prmt<0xB391u>(w) & 0x807f807fu; }
constexpr uint32_t kNibLo = 0x000f000fu, kNibHi = 0x00f000f0u;
// 5-bit codes of one nibble word w (4 bytes, low and high nibble each) whose fifth bits,
// shifted down by the word's index, sit at bit 8e + 4 (low nibble of byte e) and 8e (high
// nibble): out[0], out[1] = low-nibble codes of bytes (0, 2), (1, 3); out[2], out[3] =
// high-nibble codes of bytes (0, 2), (1, 3); each as two halves holding c in bits 0..4.
__device__ __forceinline__ void fifth_bit_codes(uint32_t w, uint32_t h, uint32_t (&out)[4]) {
    const uint32_t tl = (w & 0x0f0f0f0fu) | (h & 0x10101010u);
    const uint32_t th = ((w >> 4) & 0x0f0f0f0fu) | ((h << 4) & 0x10101010u);
    out[0] = tl & 0x001f001fu;
    out[1] = (tl >> 8) & 0x001f001fu;
    out[2] = th & 0x001f001fu;
    out[3] = (th >> 8) & 0x001f001fu;
}
constexpr float kTwo24 = 16777216.0f, kTwo20 = 1048576.0f;
constexpr float kQ4Offset = 8.0f;  // q4_0 value = scale * (c - 8)

// packed fp32 pair arithmetic (one instruction per pair)
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n add.rn.f32x2 rd, ra, rb;\n"
        " mov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
        " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Split triples of one row group up to this size are merged in one level (one CTA reads
// them all); larger sets use two levels so that no single CTA reads too much.
constexpr int kDirectMergeBytes = 96 * 1024;
constexpr int kMaxMergeWidth = 32;  // ceil(sqrt(kMaxSplits)): widest merge of either level

__device__ __forceinline__ int group_size(int ns) {
    int g = 1;
    while (g * g < ns) ++g;
    return g;
}

// All threads of the CTA call this after writing their results.  Returns true in the
// CTA that is the target-th to arrive on *counter (it then sees every earlier write).
__device__ __forceinline__ bool arrive_last(int32_t *counter, int target, int &s_flag) {
    __threadfence();  // each thread publishes its own writes
    __syncthreads();
    if (threadIdx.x == 0) {
        // the low 16 bits count arrivals (a wide merge of an earlier launch may have left a
        // launch epoch above them)
        const int t = atomicAdd(counter, 1) & 0xffff;
        s_flag = (t == target - 1);
    }
    __syncthreads();
    const bool last = s_flag != 0;
    if (last) __threadfence();
    return last;
}

// Query row (index into q, out, lse) of internal row `pr` (partial-triple row space, where
// the n_q * G rows of one (sequence, KV head) are consecutive).  The identity for n_q = 1.
struct RowMap {
    int n_q, G, Hq, Hkv;
    __device__ __forceinline__ size_t out_row(size_t pr) const {
        if (n_q == 1) return pr;
        const int ur = n_q * G;
        const size_t u = pr / ur;
        const int r = static_cast<int>(pr % ur);
        return (u / Hkv * n_q + r / G) * static_cast<size_t>(Hq) + (u % Hkv) * G + r % G;
    }
};

// Merge NP split triples (o, m, l) of `rows` consecutive query rows starting at row0:
//   M = max_s m_s, w_s = exp(m_s - M), O = sum_s w_s o_s, L = sum_s w_s l_s.
// Triples of row r, split s live at (r * stride + s0 + s).  Writes either the normalised
// output (out = O / L, lse = M + log L; row r goes to query row map.out_row(r)) or one
// unnormalised triple at (r * q_stride + q_s).  The inputs were written by other CTAs and
// sit in L2.  Each thread owns two output columns and merges up to kMergeChunk splits per
// L2 round trip, loading m, l and o together and keeping a running maximum (rescaling
// when it grows), so a merge of up to kMergeChunk splits costs one round trip and needs no
// shared memory or barrier.
constexpr int kMergeChunk = 10;
__device__ void merge_rows(const float *po, const float *pm, const float *pl, int stride, int s0, int NP,
                           size_t row0, int rows, int D, float *out, float *lse, float *qo, float *qm, float *ql,
                           int q_stride, int q_s, const RowMap map = RowMap{1, 1, 1, 1},
                           const float *ext_out = nullptr, const float *ext_lse = nullptr) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int DQ = D / 4;
    const int C = rows * DQ;
    const float4 *po4 = reinterpret_cast<const float4 *>(po);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < C; base += 2 * nthr) {
        int col[2], g[2], dq[2];
        bool v[2];
        float M[2], L[2];
        float4 A[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            col[k] = base + tid + k * nthr;
            v[k] = col[k] < C;
            g[k] = v[k] ? col[k] / DQ : 0;
            dq[k] = v[k] ? col[k] % DQ : 0;
            M[k] = -CUDART_INF_F;
            L[k] = 0.f;
            A[k] = z4;
        }
        for (int sc = 0; sc < NP; sc += kMergeChunk) {
            float mm[2][kMergeChunk], ll[2][kMergeChunk];
            float4 oo[2][kMergeChunk];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const size_t pr = (row0 + g[k]) * stride + s0 + sc;
#pragma unroll
                for (int u = 0; u < kMergeChunk; ++u) {
                    const bool in = v[k] && (sc + u < NP);
                    mm[k][u] = in ? __ldcg(pm + pr + u) : -CUDART_INF_F;
                    ll[k][u] = in ? __ldcg(pl + pr + u) : 0.f;
                    oo[k][u] = in ? __ldcg(po4 + (pr + u) * DQ + dq[k]) : z4;
                }
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float cm = -CUDART_INF_F;
#pragma unroll
                for (int u = 0; u < kMergeChunk; ++u) cm = fmaxf(cm, mm[k][u]);
                const float Mn = fmaxf(M[k], cm);
                if (Mn == -CUDART_INF_F) continue;  // nothing but empty splits so far
                const float a = M[k] == -CUDART_INF_F ? 0.f : expf(M[k] - Mn);
                A[k].x *= a;
                A[k].y *= a;
                A[k].z *= a;
                A[k].w *= a;
                L[k] *= a;
#pragma unroll
                for (int u = 0; u < kMergeChunk; ++u) {
                    const float w = mm[k][u] == -CUDART_INF_F ? 0.f : expf(mm[k][u] - Mn);
                    A[k].x = fmaf(w, oo[k][u].x, A[k].x);
                    A[k].y = fmaf(w, oo[k][u].y, A[k].y);
                    A[k].z = fmaf(w, oo[k][u].z, A[k].z);
                    A[k].w = fmaf(w, oo[k][u].w, A[k].w);
                    L[k] = fmaf(w, ll[k][u], L[k]);
                }
                M[k] = Mn;
            }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (!v[k]) continue;
            if (out) {
                const size_t orow = map.out_row(row0 + g[k]);
                if (ext_out) {  // one more triple: (ext_out, lse, l = 1)
                    const float mx = ext_lse[orow];
                    const float Mn = fmaxf(M[k], mx);
                    if (Mn != -CUDART_INF_F) {
                        const float a = M[k] == -CUDART_INF_F ? 0.f : expf(M[k] - Mn);
                        const float bw = mx == -CUDART_INF_F ? 0.f : expf(mx - Mn);
                        const float4 x = reinterpret_cast<const float4 *>(ext_out + orow * D)[dq[k]];
                        A[k] = make_float4(fmaf(bw, x.x, a * A[k].x), fmaf(bw, x.y, a * A[k].y),
                                           fmaf(bw, x.z, a * A[k].z), fmaf(bw, x.w, a * A[k].w));
                        L[k] = fmaf(a, L[k], bw);
                        M[k] = Mn;
                    }
                }
                const float inv = L[k] > 0.f ? 1.f / L[k] : 0.f;
                reinterpret_cast<float4 *>(out + orow * D)[dq[k]] =
                    make_float4(A[k].x * inv, A[k].y * inv, A[k].z * inv, A[k].w * inv);
                if (dq[k] == 0 && lse) lse[orow] = L[k] > 0.f ? M[k] + logf(L[k]) : -CUDART_INF_F;
            } else {
                const size_t dr = (row0 + g[k]) * static_cast<size_t>(q_stride) + q_s;
                reinterpret_cast<float4 *>(qo + dr * D)[dq[k]] = A[k];
                if (dq[k] == 0) {
                    qm[dr] = M[k];
                    ql[dr] = L[k];
                }
            }
        }
    }
}

// Wide merge: when the grid is resident at once, the last P CTAs to arrive for a row group
// share its merge, each taking a range of output columns (float4 columns c of the rows x
// D/4 grid, row c / (D/4)).  Each column is served by sg threads, thread k taking splits
// k, k + sg, ... with the same running-maximum rule as merge_rows (a handful of splits per
// thread, one L2 round trip); the sg partial triples of a column are then combined in
// shared memory.  Memory for the reduction: 24 bytes per thread at `red`.
constexpr int kWideMinBytes = 16 * 1024;  // smaller row groups merge in one CTA
constexpr int kWideBytes = 12 * 1024;     // triple bytes per merging CTA
constexpr int kWideChunk = 8;
__device__ void merge_cols(const float *po, const float *pm, const float *pl, int stride, int NP, size_t row0,
                           int D, int c0, int c1, float *out, float *lse, const RowMap map, const float *ext_out,
                           const float *ext_lse, uint8_t *red) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int DQ = D / 4;
    const int ncol = c1 - c0;
    const int sg = max(1, min(nthr / max(ncol, 1), (NP + 3) / 4));  // threads per column
    float4 *rA = reinterpret_cast<float4 *>(red);
    float *rM = reinterpret_cast<float *>(red + static_cast<size_t>(nthr) * 16);
    float *rL = rM + nthr;
    const float4 *po4 = reinterpret_cast<const float4 *>(po);
    for (int base = 0; base < ncol * sg; base += nthr) {
        const int item = base + tid;
        const bool v = item < ncol * sg;
        const int ci = v ? item % ncol : 0, k = v ? item / ncol : 0;
        const int col = c0 + ci;
        const size_t pr = (row0 + col / DQ) * stride;
        const int dq = col % DQ;
        float M = -CUDART_INF_F, L = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = k; v && s < NP; s += kWideChunk * sg) {
            float mm[kWideChunk], ll[kWideChunk];
            float4 oo[kWideChunk];
#pragma unroll
            for (int u = 0; u < kWideChunk; ++u) {
                const int su = s + u * sg;
                const bool in = su < NP;
                mm[u] = in ? __ldcg(pm + pr + su) : -CUDART_INF_F;
                ll[u] = in ? __ldcg(pl + pr + su) : 0.f;
                oo[u] = in ? __ldcg(po4 + (pr + su) * DQ + dq) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float cm = -CUDART_INF_F;
#pragma unroll
            for (int u = 0; u < kWideChunk; ++u) cm = fmaxf(cm, mm[u]);
            const float Mn = fmaxf(M, cm);
            if (Mn == -CUDART_INF_F) continue;
            const float a = M == -CUDART_INF_F ? 0.f : expf(M - Mn);
            A = make_float4(A.x * a, A.y * a, A.z * a, A.w * a);
            L *= a;
#pragma unroll
            for (int u = 0; u < kWideChunk; ++u) {
                const float w = mm[u] == -CUDART_INF_F ? 0.f : expf(mm[u] - Mn);
                A = make_float4(fmaf(w, oo[u].x, A.x), fmaf(w, oo[u].y, A.y), fmaf(w, oo[u].z, A.z), fmaf(w, oo[u].w, A.w));
                L = fmaf(w, ll[u], L);
            }
            M = Mn;
        }
        if (sg > 1) {
            if (v) {
                rA[k * ncol + ci] = A;
                rM[k * ncol + ci] = M;
                rL[k * ncol + ci] = L;
            }
            __syncthreads();
            if (v && k == 0) {
                // the maximum over the sg partial triples first, then independent weights
                float Mx = M;
                for (int k2 = 1; k2 < sg; ++k2) Mx = fmaxf(Mx, rM[k2 * ncol + ci]);
                if (Mx != -CUDART_INF_F) {
                    const float a = M == -CUDART_INF_F ? 0.f : expf(M - Mx);
                    A = make_float4(a * A.x, a * A.y, a * A.z, a * A.w);
                    L *= a;
#pragma unroll 4
                    for (int k2 = 1; k2 < sg; ++k2) {
                        const float m2 = rM[k2 * ncol + ci];
                        const float b = m2 == -CUDART_INF_F ? 0.f : expf(m2 - Mx);
                        const float4 x = rA[k2 * ncol + ci];
                        A = make_float4(fmaf(b, x.x, A.x), fmaf(b, x.y, A.y), fmaf(b, x.z, A.z), fmaf(b, x.w, A.w));
                        L = fmaf(b, rL[k2 * ncol + ci], L);
                    }
                    M = Mx;
                }
            }
            __syncthreads();
        }
        if (!v || k != 0) continue;
        const size_t orow = map.out_row(row0 + col / DQ);
        if (ext_out) {  // one more triple: (ext_out, lse, l = 1)
            const float mx = ext_lse[orow];
            const float Mn = fmaxf(M, mx);
            if (Mn != -CUDART_INF_F) {
                const float a = M == -CUDART_INF_F ? 0.f : expf(M - Mn);
                const float bw = mx == -CUDART_INF_F ? 0.f : expf(mx - Mn);
                const float4 x = reinterpret_cast<const float4 *>(ext_out + orow * D)[dq];
                A = make_float4(fmaf(bw, x.x, a * A.x), fmaf(bw, x.y, a * A.y), fmaf(bw, x.z, a * A.z), fmaf(bw, x.w, a * A.w));
                L = fmaf(a, L, bw);
                M = Mn;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<float4 *>(out + orow * D)[dq] = make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
        if (dq == 0 && lse) lse[orow] = L > 0.f ? M + logf(L) : -CUDART_INF_F;
    }
}

// Wait (thread 0) until the arrivals of a wide merge are complete: the arrival count (low
// 16 bits) of *counter reaches target, or its launch epoch (the bits above) is no longer
// `epoch`.  0 within `report` SM cycles, 1 later (reported), 2 not within kWaitCycles (gave
// up).
constexpr int kLaunchEpoch = 1 << 16;
__device__ __forceinline__ int wait_arrivals(const int32_t *counter, unsigned epoch, int target, long long report) {
    const long long t0 = clock64();
    while (true) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(counter) : "memory");
        if (static_cast<int>(v & 0xffffu) >= target || (v >> 16) != epoch) return clock64() - t0 > report ? 1 : 0;
        if (clock64() - t0 > kWaitCycles) return 2;
        __nanosleep(64);
    }
}

// Fused append: every CTA of the grid arrives once, after it has read the lengths; the
// last one advances len[b] by one for each sequence that had room (else it reports
// KVQ_DEVERR_CAPACITY) and resets the ticket.  Called by one thread per CTA.
__device__ __noinline__ void grid_ticket(const DecodeParams &p, int cap_rows) {
    __threadfence();
    const int total = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
    if (atomicAdd(p.ticket, 1) != total - 1) return;
    __threadfence();
    int32_t *len = const_cast<int32_t *>(p.len);
    for (int b = 0; b < p.B; ++b) {
        const int Lb = __ldcg(len + b);
        if (Lb >= 0 && Lb + 1 <= cap_rows)
            len[b] = Lb + 1;
        else
            atomicOr(p.err, KVQ_DEVERR_CAPACITY);
    }
    *p.ticket = 0;
}

// Two-region append (kvq_window_append_decode): the last CTA of the grid advances, per
// sequence, the window's length while it fills, then the tail's (its evicted row), or
// reports KVQ_DEVERR_CAPACITY.  Called by one thread per CTA, once.
__device__ __noinline__ void window_ticket(const DecodeParams &p) {
    __threadfence();
    const int total = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
    if (atomicAdd(p.ticket, 1) != total - 1) return;
    __threadfence();
    for (int b = 0; b < p.B; ++b) {
        const int Lw = __ldcg(p.wl_len + b), Lt = __ldcg(p.tl_len + b);
        if (Lw < 0 || Lw > p.wl_cap || Lt < 0)
            atomicOr(p.wl_err, KVQ_DEVERR_CAPACITY);
        else if (Lw < p.wl_cap)
            p.wl_len[b] = Lw + 1;
        else if (Lt + 1 <= p.tl_cap)
            p.tl_len[b] = Lt + 1;
        else
            atomicOr(p.tl_err, KVQ_DEVERR_CAPACITY);
    }
    *p.ticket = 0;
}
__device__ __forceinline__ void append_ticket(const DecodeParams &p, int cap_rows) {
    if (p.win)
        window_ticket(p);
    else
        grid_ticket(p, cap_rows);
}

// Wait (one thread) until *flag is non-zero, then clear it; reports KVQ_DEVERR_TIMEOUT past
// `report` SM cycles and gives up after kWaitCycles.
__device__ __forceinline__ void wait_flag_clear(int32_t *flag, long long report, int32_t *err) {
    const long long t0 = clock64();
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(flag) : "memory");
        if (v) break;
        if (clock64() - t0 > kWaitCycles) break;
        __nanosleep(64);
    }
    if (clock64() - t0 > report) atomicOr(err, KVQ_DEVERR_TIMEOUT);
    atomicExch(flag, 0);
}

template <int KT, int VT, int NS, int TW_ = 0>
struct Cfg {
    // tile-warps per 128-value slice: 11 for 128-wide heads with quantised keys (the
    // conversion work wants the warps), 8 for f16 keys, 4 pairs for 256-wide heads; TW_
    // overrides (the f16 window body of a two-region launch takes the tail's count)
    static constexpr int TW = TW_ ? TW_ : (NS == 2 ? 4 : (KT == KVQ_F16 ? 8 : 11));
    static constexpr int CW = TW * NS;         // consumer warps
    static constexpr int THREADS = 32 * (CW + 1);
    static constexpr int KC = code_tile_bytes(KT) * NS;
    static constexpr int VC = code_tile_bytes(VT) * NS;
    static constexpr int KS = scale_tile_bytes(KT) * NS;
    static constexpr int VS = scale_tile_bytes(VT) * NS;
    static constexpr int TILE = KC + VC + KS + VS;
    static constexpr int MIN_CTAS = 1;         // one CTA per SM: up to 11 consumer warps + 1 producer
    // ring budget: 204 KB for 256-wide heads, so that three stages of eight q8_0 tiles fit
    // beside the score exchange; 220 KB for 128-wide heads, so that q8_0/q4_0 gets a third
    // stage (more bytes in flight per SM)
    static constexpr int RING_BUDGET = NS == 2 ? 208896 : 225280;
    // tiles each warp takes per stage: two (32 keys share one softmax step) when the ring
    // still holds at least two stages, else one
    static constexpr int TPW = (2 * 2 * TW * TILE <= RING_BUDGET) ? 2 : 1;
    static constexpr int TWT = TW * TPW;       // tiles per stage
    static constexpr int STAGE = TWT * TILE;
    static constexpr int STAGES_RAW = RING_BUDGET / STAGE;
    // 128-wide heads: at most three stages (a fourth, for 4-bit pairs, measured slower)
    static constexpr int STAGES_MAX = NS == 1 ? 3 : 16;
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > STAGES_MAX ? STAGES_MAX : STAGES_RAW);
    static constexpr int RING = STAGES * STAGE;
    // score exchange of the two slice-warps of each tile pair, then one guard flag per warp
    static constexpr int XCHG_SC = NS == 2 ? TW * 2 * 32 * 16 * TPW : 0;
    static constexpr int XCHG = NS == 2 ? XCHG_SC + (TW * 2 * 4 + 15) / 16 * 16 : 0;
    static constexpr int BAR_OFF = RING + XCHG;
    // per slice: the K code-offset corrections of its 8 rows x 4 blocks, and the Q
    // fragments (8 chunks x 32 lanes x 16 B) that every tile-warp of the slice reads
    static constexpr int KCOR_OFF = (BAR_OFF + 2 * STAGES * 8 + 15) / 16 * 16;
    static constexpr int QSM_OFF = KCOR_OFF + NS * 128;
    static constexpr int SMEM = QSM_OFF + NS * 8 * 32 * 16 + 16;
    static constexpr int D = NS * kSlice;
    static constexpr bool F16_PAIR = KT == KVQ_F16 && VT == KVQ_F16;
    // merge / combine scratch reuses the ring
    static_assert(TW * kMaxRowsPerGroup * D * 4 + 2 * TW * kMaxRowsPerGroup * 4 <= RING, "merge buffer");
};

struct QFrag {
    uint32_t a[4];
};

// Scores of one tile over this warp's 128-value slice for keys A=2j, B=2j+1 (S-tile 0) and
// C=8+2j, D=9+2j (S-tile 1), row g = lane/4, in log2 units (Q was prescaled).
template <int KT>
__device__ __forceinline__ void tile_scores(const uint8_t *kc, const uint8_t *ks, const uint8_t *qsm,
                                            const uint8_t *kcor, int lane, int j, float (&s)[4]) {
    // Q fragment of chunk c (16 values), read from shared memory where it is used
    auto qa = [&](int c) {
        const uint4 v = lds128(qsm + (c * 32 + lane) * 16);
        return QFrag{{v.x, v.y, v.z, v.w}};
    };
    if constexpr (KT == KVQ_F16) {
        float acc[2][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint4 w0 = lds128(kc + (2 * b + 0) * 512 + lane * 16);
            const uint4 w1 = lds128(kc + (2 * b + 1) * 512 + lane * 16);
            if (b == 0) {
                mma_16816_z(acc[0], qa(0).a, w0.x, w0.y);
                mma_16816_z(acc[1], qa(0).a, w1.x, w1.y);
            } else {
                mma_16816(acc[0], qa(2 * b).a, w0.x, w0.y);
                mma_16816(acc[1], qa(2 * b).a, w1.x, w1.y);
            }
            mma_16816(acc[0], qa(2 * b + 1).a, w0.z, w0.w);
            mma_16816(acc[1], qa(2 * b + 1).a, w1.z, w1.w);
        }
        s[0] = acc[0][0] + acc[0][2];
        s[1] = acc[0][1] + acc[0][3];
        s[2] = acc[1][0] + acc[1][2];
        s[3] = acc[1][1] + acc[1][3];
    } else {
        // accumulators hold sum q * code in units of 2^-24 (q8_0, q5_0, q5_1) or, with the
        // low-nibble chunk of Q prescaled by 16, sum q * c in units of 2^-20 (q4_0, q4_1).
        // kcorr[b] (per row, same unit): -K * sum_b q for the offset types (c -> c - K), or
        // sum_b q for the types with a minimum (times lo of each key)
        float kcorr[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (is_nibble_type(KT)) {
            const float4 kc4 = *reinterpret_cast<const float4 *>(kcor);
            kcorr[0] = kc4.x;
            kcorr[1] = kc4.y;
            kcorr[2] = kc4.z;
            kcorr[3] = kc4.w;
        }
        const uint4 sc0 = lds128(ks + j * 32), sc1 = lds128(ks + j * 32 + 16);
        const uint32_t kscale[4][2] = {{sc0.x, sc0.y}, {sc0.z, sc0.w}, {sc1.x, sc1.y}, {sc1.z, sc1.w}};
        float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
        uint4 wq4 = make_uint4(0, 0, 0, 0);
        uint32_t hb = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float acc[2][4];
            if constexpr (KT == KVQ_Q8_0) {
                const uint4 w = lds128(kc + b * 512 + lane * 16);
                mma_16816_z(acc[0], qa(2 * b).a, q8_02(w.x), q8_13(w.x));
                mma_16816(acc[0], qa(2 * b + 1).a, q8_02(w.y), q8_13(w.y));
                mma_16816_z(acc[1], qa(2 * b).a, q8_02(w.z), q8_13(w.z));
                mma_16816(acc[1], qa(2 * b + 1).a, q8_02(w.w), q8_13(w.w));
            } else if constexpr (!has_fifth_bit(KT)) {
                if ((b & 1) == 0) wq4 = lds128(kc + (b >> 1) * 512 + lane * 16);
                const uint32_t w0 = (b & 1) ? wq4.z : wq4.x, w0s = w0 >> 8;
                const uint32_t w1 = (b & 1) ? wq4.w : wq4.y, w1s = w1 >> 8;
                mma_16816_z(acc[0], qa(2 * b).a, w0 & kNibLo, w0s & kNibLo);
                mma_16816(acc[0], qa(2 * b + 1).a, w0 & kNibHi, w0s & kNibHi);
                mma_16816_z(acc[1], qa(2 * b).a, w1 & kNibLo, w1s & kNibLo);
                mma_16816(acc[1], qa(2 * b + 1).a, w1 & kNibHi, w1s & kNibHi);
            } else {
                if ((b & 1) == 0) {
                    wq4 = lds128(kc + (b >> 1) * 512 + lane * 16);
                    hb = *reinterpret_cast<const uint32_t *>(kc + kNibbleBytes + (b >> 1) * 128 + lane * 4);
                }
                const int wi0 = 2 * (b & 1), wi1 = wi0 + 1;
                uint32_t c0[4], c1[4];
                fifth_bit_codes((b & 1) ? wq4.z : wq4.x, hb >> wi0, c0);
                fifth_bit_codes((b & 1) ? wq4.w : wq4.y, hb >> wi1, c1);
                mma_16816_z(acc[0], qa(2 * b).a, c0[0], c0[1]);
                mma_16816(acc[0], qa(2 * b + 1).a, c0[2], c0[3]);
                mma_16816_z(acc[1], qa(2 * b).a, c1[0], c1[1]);
                mma_16816(acc[1], qa(2 * b + 1).a, c1[2], c1[3]);
            }
            const float2 dab = __half22float2(u32_as_h2(kscale[b][0]));
            const float2 dcd = __half22float2(u32_as_h2(kscale[b][1]));
            float2 t01 = add2(make_float2(acc[0][0], acc[0][1]), make_float2(acc[0][2], acc[0][3]));
            float2 t23 = add2(make_float2(acc[1][0], acc[1][1]), make_float2(acc[1][2], acc[1][3]));
            if constexpr (KT == KVQ_Q4_0 || KT == KVQ_Q5_0) {
                const float2 cb = make_float2(kcorr[b], kcorr[b]);
                t01 = add2(t01, cb);
                t23 = add2(t23, cb);
            }
            s01 = fma2(dab, t01, s01);
            s23 = fma2(dcd, t23, s23);
            if constexpr (has_min(KT)) {  // + lo * sum_b q
                const uint2 lsc = *reinterpret_cast<const uint2 *>(ks + kScaleTile + j * 32 + b * 8);
                const float2 cb = make_float2(kcorr[b], kcorr[b]);
                s01 = fma2(__half22float2(u32_as_h2(lsc.x)), cb, s01);
                s23 = fma2(__half22float2(u32_as_h2(lsc.y)), cb, s23);
            }
        }
        constexpr float unit = (KT == KVQ_Q4_0 || KT == KVQ_Q4_1) ? kTwo20 : kTwo24;
        s[0] = s01.x * unit;
        s[1] = s01.y * unit;
        s[2] = s23.x * unit;
        s[3] = s23.y * unit;
    }
}

// O += P V for one tile over this warp's slice.  pk: probabilities of keys A,B,C,D of row g;
// vmask: which of A,B,C,D are inside the sequence (rows past the length may hold any bits).
template <int VT, bool PARTIAL>
__device__ __forceinline__ void tile_pv(const uint8_t *vc, const uint8_t *vs, const float (&pk)[4],
                                        const bool (&vmask)[4], int lane, int j, float (&o)[16][4],
                                        uint32_t magic, float (&corr)[4]) {
    if constexpr (VT == KVQ_F16) {
        uint32_t a[4];
        split_hi_lo(pk[0], pk[1], a[0], a[1]);
        split_hi_lo(pk[2], pk[3], a[2], a[3]);
        const uint32_t mab = (vmask[0] ? 0x0000ffffu : 0u) | (vmask[1] ? 0xffff0000u : 0u);
        const uint32_t mcd = (vmask[2] ? 0x0000ffffu : 0u) | (vmask[3] ? 0xffff0000u : 0u);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint4 w0 = lds128(vc + (2 * b + 0) * 512 + lane * 16);
            uint4 w1 = lds128(vc + (2 * b + 1) * 512 + lane * 16);
            if constexpr (PARTIAL) {
                w0.x &= mab;
                w0.y &= mcd;
                w0.z &= mab;
                w0.w &= mcd;
                w1.x &= mab;
                w1.y &= mcd;
                w1.z &= mab;
                w1.w &= mcd;
            }
            mma_16816(o[4 * b + 0], a, w0.x, w0.y);
            mma_16816(o[4 * b + 1], a, w0.z, w0.w);
            mma_16816(o[4 * b + 2], a, w1.x, w1.y);
            mma_16816(o[4 * b + 3], a, w1.z, w1.w);
        }
    } else {
        // P' = p x scale per (key, block) as f16 hi + lo: p is split once per tile
        // (p = ph + pl), then per block  hi = ph*d,  err = fma(ph, d, -hi) (exact: the
        // rounding error of an f16 product), lo = fma(pl, d, err)  -- three packed f16 ops
        // per key pair, about 2^-21 relative.  The scale half2 words already pair keys
        // (A,B) and (C,D), matching the A-fragment pairs.
        uint32_t ph_ab, pl_ab, ph_cd, pl_cd;
        split_hi_lo(pk[0], pk[1], ph_ab, pl_ab);
        split_hi_lo(pk[2], pk[3], ph_cd, pl_cd);
        const uint4 sc0 = lds128(vs + j * 32), sc1 = lds128(vs + j * 32 + 16);
        const uint32_t vscale[4][2] = {{sc0.x, sc0.y}, {sc0.z, sc0.w}, {sc1.x, sc1.y}, {sc1.z, sc1.w}};
        uint32_t mab = 0xffffffffu, mcd = 0xffffffffu;
        if constexpr (PARTIAL) {  // scales past the length may hold any bits
            mab = (vmask[0] ? 0x0000ffffu : 0u) | (vmask[1] ? 0xffff0000u : 0u);
            mcd = (vmask[2] ? 0x0000ffffu : 0u) | (vmask[3] ? 0xffff0000u : 0u);
        }
        uint4 wq4 = make_uint4(0, 0, 0, 0);
        uint32_t hb = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const __half2 dab = u32_as_h2(vscale[b][0] & mab);
            const __half2 dcd = u32_as_h2(vscale[b][1] & mcd);
            const __half2 hab = __hmul2(u32_as_h2(ph_ab), dab);
            const __half2 hcd = __hmul2(u32_as_h2(ph_cd), dcd);
            const __half2 eab = __hfma2(u32_as_h2(ph_ab), dab, __hneg2(hab));
            const __half2 ecd = __hfma2(u32_as_h2(ph_cd), dcd, __hneg2(hcd));
            uint32_t a[4];
            a[0] = h2_as_u32(hab);
            a[1] = h2_as_u32(__hfma2(u32_as_h2(pl_ab), dab, eab));
            a[2] = h2_as_u32(hcd);
            a[3] = h2_as_u32(__hfma2(u32_as_h2(pl_cd), dcd, ecd));
            // q8_0: o accumulates sum P' * q in units of 2^-24; nibble types: exact f16 code
            // values by the magic-number route (nibble | 0x6400 is 1024 + c; a high nibble
            // gives 1024 + 16c, scaled by 1/16), less the offset (8 for q4_0, 16 for q5_0)
            if constexpr (VT == KVQ_Q8_0) {
                const uint4 w = lds128(vc + b * 512 + lane * 16);
                mma_16816(o[4 * b + 0], a, q8_02(w.x), q8_13(w.x));
                mma_16816(o[4 * b + 1], a, q8_02(w.y), q8_13(w.y));
                mma_16816(o[4 * b + 2], a, q8_02(w.z), q8_13(w.z));
                mma_16816(o[4 * b + 3], a, q8_02(w.w), q8_13(w.w));
            } else if constexpr (!has_fifth_bit(VT)) {
                if ((b & 1) == 0) wq4 = lds128(vc + (b >> 1) * 512 + lane * 16);
                const uint32_t wq0 = (b & 1) ? wq4.z : wq4.x, wq0s = wq0 >> 8;  // bytes 2n'   of the block
                const uint32_t wq1 = (b & 1) ? wq4.w : wq4.y, wq1s = wq1 >> 8;  // bytes 2n'+1 of the block
                constexpr float off = VT == KVQ_Q4_0 ? kQ4Offset : 0.0f;
                const __half2 klo = __float2half2_rn(1024.0f + off), k16th = __float2half2_rn(0.0625f),
                              khi = __float2half2_rn(-64.0f - off);
                auto lo = [&](uint32_t x) { return h2_as_u32(__hsub2(u32_as_h2((x & kNibLo) | magic), klo)); };
                auto hi = [&](uint32_t x) { return h2_as_u32(__hfma2(u32_as_h2((x & kNibHi) | magic), k16th, khi)); };
                mma_16816(o[4 * b + 0], a, lo(wq0), lo(wq0s));
                mma_16816(o[4 * b + 2], a, hi(wq0), hi(wq0s));
                mma_16816(o[4 * b + 1], a, lo(wq1), lo(wq1s));
                mma_16816(o[4 * b + 3], a, hi(wq1), hi(wq1s));
            } else {
                if ((b & 1) == 0) {
                    wq4 = lds128(vc + (b >> 1) * 512 + lane * 16);
                    hb = *reinterpret_cast<const uint32_t *>(vc + kNibbleBytes + (b >> 1) * 128 + lane * 4);
                }
                uint32_t c0[4], c1[4];
                fifth_bit_codes((b & 1) ? wq4.z : wq4.x, hb >> (2 * (b & 1)), c0);
                fifth_bit_codes((b & 1) ? wq4.w : wq4.y, hb >> (2 * (b & 1) + 1), c1);
                const __half2 koff = __float2half2_rn(VT == KVQ_Q5_0 ? 1040.0f : 1024.0f);
                auto val = [&](uint32_t x) { return h2_as_u32(__hsub2(u32_as_h2(x | magic), koff)); };
                mma_16816(o[4 * b + 0], a, val(c0[0]), val(c0[1]));
                mma_16816(o[4 * b + 2], a, val(c0[2]), val(c0[3]));
                mma_16816(o[4 * b + 1], a, val(c1[0]), val(c1[1]));
                mma_16816(o[4 * b + 3], a, val(c1[2]), val(c1[3]));
            }
            if constexpr (has_min(VT)) {
                // + p * lo for every value of the block: sum over keys of p * lo (f16 hi + lo
                // like P') lands in column b of corr (B = 1.0 in column b); added at the end
                const uint2 lsc = *reinterpret_cast<const uint2 *>(vs + kScaleTile + j * 32 + b * 8);
                const __half2 lab = u32_as_h2(lsc.x & mab), lcd = u32_as_h2(lsc.y & mcd);
                const __half2 hab2 = __hmul2(u32_as_h2(ph_ab), lab), hcd2 = __hmul2(u32_as_h2(ph_cd), lcd);
                uint32_t a2[4];
                a2[0] = h2_as_u32(hab2);
                a2[1] = h2_as_u32(__hfma2(u32_as_h2(pl_ab), lab, __hfma2(u32_as_h2(ph_ab), lab, __hneg2(hab2))));
                a2[2] = h2_as_u32(hcd2);
                a2[3] = h2_as_u32(__hfma2(u32_as_h2(pl_cd), lcd, __hfma2(u32_as_h2(ph_cd), lcd, __hneg2(hcd2))));
                const uint32_t one = (lane >> 2) == b ? 0x3c003c00u : 0u;
                mma_16816(corr, a2, one, one);
            }
        }
    }
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ void split_range(const DecodeParams &p, int T, int split, int &t0, int &t1) {
    const int ns = max(1, min(p.n_splits, T));
    const int tps = T > 0 ? (T + ns - 1) / ns : 0;
    t0 = min(T, split * tps);
    t1 = min(T, t0 + tps);
}

// Cache tiles this CTA starts with, pulled into L2 while the previous kernel of the stream
// drains (called before the programmatic-launch wait): f16 caches only, which read two
// bytes per value and are bound by HBM; for the quantised ones, whose loop is bound by the
// consumer warps, the extra early traffic slowed the step.  Only a hint: the length read here
// may be one append behind and the tiles may still be written; L2 is the coherence point,
// so later reads see every write either way.  Capped per CTA so that the prefetched set of
// all CTAs stays well inside L2.
constexpr int kPrefetchBytes = 384 * 1024;
template <class C>
__device__ __noinline__ void prefetch_split(const DecodeParams &p, int bseq, int h, int split, int cap_rows,
                                            int skip_tiles) {
    if constexpr (!C::F16_PAIR) return;
    int L = *reinterpret_cast<const volatile int32_t *>(p.len + bseq);
    if (p.k_new != nullptr) ++L;
    L = L < 0 ? 0 : (L > cap_rows ? cap_rows : L);
    const int T = (L + kTileRows - 1) / kTileRows;
    const int ns = max(1, min(p.n_splits, T));
    if (split >= ns || T == 0) return;
    const int tps = (T + ns - 1) / ns;
    const int t0 = min(T, split * tps + skip_tiles), t1 = min(T, split * tps + tps);
    const int nt = min(t1 - t0, kPrefetchBytes / C::TILE - skip_tiles);
    if (nt <= 0) return;
    const size_t bt = (static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles + t0;
    constexpr int kChunk = 32768;
    auto pf = [](const uint8_t *base, size_t bytes) {
        for (size_t o = 0; o < bytes; o += kChunk)
            bulk_prefetch_l2(base + o, static_cast<uint32_t>(min(static_cast<size_t>(kChunk), bytes - o)));
    };
    pf(p.k_codes + bt * C::KC, static_cast<size_t>(nt) * C::KC);
    pf(p.v_codes + bt * C::VC, static_cast<size_t>(nt) * C::VC);
    if constexpr (C::KS > 0) pf(p.k_scales + bt * C::KS, static_cast<size_t>(nt) * C::KS);
    if constexpr (C::VS > 0) pf(p.v_scales + bt * C::VS, static_cast<size_t>(nt) * C::VS);
}

// ---------------- merge of the split triples of one (sequence, KV head, row group) ----------------
// Called by every CTA of the row group once it has written its triple at slot `slot` of
// the NP slots (row r, slot s at r * part_stride + s).  Small sets: the last CTA to arrive
// merges them all.  Larger sets in a grid that is resident at once: the last P arrivals
// share the merge by columns.  Otherwise slots form groups of ceil(sqrt(NP)); the last
// arrival of each group merges its group into a group triple while other CTAs still run,
// and the last group merges the group triples.
__device__ __forceinline__ void split_merge(const DecodeParams &p, int NP, int slot, int rows, int D, size_t row0,
                                            size_t unit, const RowMap &rmap, int &s_flag, uint8_t *smem) {
    const long long tbytes = static_cast<long long>(NP) * rows * (D + 2) * 4;
    if (p.wide && tbytes > kWideMinBytes) {
        // the last P arrivals each merge a range of columns once every split has arrived.
        // The counter holds this launch's arrivals in its low 16 bits and a launch epoch
        // above them: the last arrival adds one epoch and takes the arrivals back to zero
        // in one atomic, so that the counter is ready for the next launch without a second
        // round of arrivals; a merger waits until the arrivals reach NP or the epoch moves.
        // A merger whose wait gave up merges nothing; the counter ends right either way.
        const int C = rows * (D / 4);
        const int P = max(1, min(min(NP, C), static_cast<int>((tbytes + kWideBytes - 1) / kWideBytes)));
        int32_t *cnt = p.counters + unit;
        __threadfence();  // each thread publishes its own writes
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned old = static_cast<unsigned>(atomicAdd(cnt, 1));
            const int t = static_cast<int>(old & 0xffffu);  // earlier arrivals of this launch
            int role = t >= NP - P ? t - (NP - P) : -1;     // merger index, or -1
            if (t == NP - 1) atomicAdd(cnt, kLaunchEpoch - NP);
            const int w = role >= 0 && t != NP - 1 ? wait_arrivals(cnt, old >> 16, NP, p.wait_cycles) : 0;
            if (w) atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
            if (w == 2) role = -1;  // a merger that gave up: no merge
            s_flag = role;
        }
        __syncthreads();
        const int role = s_flag;
        if (role < 0) return;
        __threadfence();
        merge_cols(p.part_o, p.part_m, p.part_l, p.part_stride, NP, row0, D, role * C / P, (role + 1) * C / P, p.out,
                   p.lse, rmap, p.ext_out, p.ext_lse, smem);
        return;
    }
    if (tbytes <= kDirectMergeBytes) {
        if (!arrive_last(p.counters + unit, NP, s_flag)) return;
        merge_rows(p.part_o, p.part_m, p.part_l, p.part_stride, 0, NP, row0, rows, D, p.out, p.lse, nullptr, nullptr,
                   nullptr, 0, 0, rmap, p.ext_out, p.ext_lse);
        if (threadIdx.x == 0) p.counters[unit] = 0;
        return;
    }
    const int gs = group_size(NP);
    const int n_groups = (NP + gs - 1) / gs;
    const int grp = slot / gs;
    const int gsize = min(gs, NP - grp * gs);
    int32_t *cnt1 = p.counters1 + unit * kGroupCounterStride + grp;
    if (!arrive_last(cnt1, gsize, s_flag)) return;
    merge_rows(p.part_o, p.part_m, p.part_l, p.part_stride, grp * gs, gsize, row0, rows, D, nullptr, nullptr, p.grp_o,
               p.grp_m, p.grp_l, p.n_groups_max, grp);
    if (threadIdx.x == 0) *cnt1 = 0;
    if (!arrive_last(p.counters + unit, n_groups, s_flag)) return;
    merge_rows(p.grp_o, p.grp_m, p.grp_l, p.n_groups_max, 0, n_groups, row0, rows, D, p.out, p.lse, nullptr,
               nullptr, nullptr, 0, 0, rmap, p.ext_out, p.ext_lse);
    if (threadIdx.x == 0) p.counters[unit] = 0;
}

// Launch timing (p.stamps): thread 0 of a CTA writes %globaltimer when it starts and when it
// leaves the kernel, to stamps[2c], stamps[2c + 1] for CTA c (every path out of decode_body
// is CTA-uniform).  Stamps inside the body cost registers in the decode loop; two-region
// (window + tail) launches, whose two inlined bodies are tighter still, write none.
constexpr int kStamps = 2;
// Stamp k of this CTA (thread 0), or nothing.  The address is formed at each use, so that no
// register holds it through the decode loop.
__device__ __forceinline__ void stamp(const DecodeParams &sp, int k) {
    if (sp.stamps == nullptr || threadIdx.x != 0) return;
    const unsigned c = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (c >= static_cast<unsigned>(sp.stamp_ctas)) return;
    unsigned long long *st = sp.stamps + kStamps * static_cast<size_t>(c);
    st[k] = global_timer_ns();
}

// The decode of one CTA: split `split` of this launch's cache (blockIdx.y = KV head,
// blockIdx.z = sequence x row group).  MERGE false: the caller runs the split merge (the
// two-region kernel, so that its two bodies share one copy of the merge code).
template <int KT, int VT, int NS, bool MQ, int TW_ = 0, bool MERGE = true>
__device__ __forceinline__ void decode_body(const DecodeParams &p, const int fused, const int split) {
    using C = Cfg<KT, VT, NS, TW_>;
    constexpr int TPW = C::TPW;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_flag;
    __shared__ int s_timeout;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int bseq = blockIdx.z / p.QG, qg = blockIdx.z % p.QG;
    const int cap_rows = p.cap_tiles * kTileRows;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::BAR_OFF);
    uint64_t *empty = full + C::STAGES;
    if (threadIdx.x == 0) {  // shared memory only: may run before the wait below
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, C::CW);
        }
        fence_mbar_init();
        s_timeout = 0;
    }
    __syncthreads();
    // Programmatic dependent launch.  Global memory that the previous kernel of the stream
    // may write (queries, new rows, outputs, workspace, and in general the cache) is read
    // only after griddepcontrol.wait.  With p.early set the host has established that the
    // previous kernel does not write this cache, so its lengths and tiles are final already:
    // the lengths are read at once and the producer fills the ring before the wait.  Every
    // CTA releases its dependents only after its own wait, so while a kernel runs its
    // pre-wait part at most one earlier kernel of the stream can still be running.
    const bool early = p.early != 0;
    if (!early) {
        if (threadIdx.x == 0) prefetch_split<C>(p, bseq, h, split, cap_rows, 0);
        grid_dep_wait();
    }
    int L_old = __ldcg(p.len + bseq);
    L_old = L_old < 0 ? 0 : (L_old > cap_rows ? cap_rows : L_old);
    // fused append: the new row lands at position L_old and is attended to.  Two-region
    // append: the window's new row lands in ring slot (tail + window length) mod capacity
    // (the oldest row once the window is full), and a full window's oldest row is moved, as
    // the tail's new row, to tail position t_len (quantised from its f16 value)
    const bool appending = p.k_new != nullptr || p.win != 0;
    bool do_app, win_full = false;
    int L, app_row = L_old;
    if (p.win == 0) {
        do_app = appending && L_old + 1 <= cap_rows;
        L = do_app ? L_old + 1 : L_old;
    } else {
        int Lw = __ldcg(p.wl_len + bseq), Lt = __ldcg(p.tl_len + bseq);
        Lw = Lw < 0 ? 0 : (Lw > p.wl_cap ? p.wl_cap : Lw);
        Lt = Lt < 0 ? 0 : (Lt > p.tl_cap ? p.tl_cap : Lt);
        win_full = Lw >= p.wl_cap;
        const bool room = !win_full || Lt + 1 <= p.tl_cap;
        if (p.win == 1) {
            do_app = room;
            app_row = static_cast<int>((static_cast<long long>(Lt) + Lw) % p.wl_cap);
            L = do_app && !win_full ? Lw + 1 : Lw;
        } else {
            do_app = win_full && room;
            app_row = Lt;
            L = do_app ? Lt + 1 : Lt;
        }
    }
    const int T = (L + kTileRows - 1) / kTileRows;
    const int ns = max(1, min(p.n_splits, T));
    const int tps = T > 0 ? (T + ns - 1) / ns : 0;
    const int n_q = MQ ? p.n_q : 1;     // queries per sequence (compile-time 1 for decode)
    const int unit_rows = n_q * p.G;    // query rows of this (sequence, KV head)
    const int rows = min(kMaxRowsPerGroup, unit_rows - qg * kMaxRowsPerGroup);
    const int r0 = qg * kMaxRowsPerGroup;  // first of them in this CTA
    const size_t prow0 = (static_cast<size_t>(bseq) * p.Hkv + h) * unit_rows + r0;  // its triple row
    const RowMap rmap{n_q, p.G, p.Hq, p.Hkv};

    // A split beyond ns has no tiles.  Alone it publishes nothing; as a region of a larger
    // merge it runs on with an empty range (t_begin = t_end = T) and publishes an empty triple.
    if (split >= ns && p.merge_slots == 0) {
        if (early) grid_dep_wait();
        grid_dep_launch();
        if (appending && threadIdx.x == 0) append_ticket(p, cap_rows);
        if (!fused) {  // partials mode: splits beyond ns are empty triples
            for (int idx = threadIdx.x; idx < rows * (p.D / 4); idx += blockDim.x) {
                const int g = idx / (p.D / 4), dq = idx % (p.D / 4);
                const size_t pr = (prow0 + g) * p.part_stride + p.part_base + split;
                reinterpret_cast<float4 *>(p.part_o + pr * p.D)[dq] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (dq == 0) {
                    p.part_m[pr] = -CUDART_INF_F;
                    p.part_l[pr] = 0.f;
                }
            }
        }
        return;
    }
    const int t_begin = min(T, split * tps), t_end = min(T, t_begin + tps);
    const int n_stage = (t_end - t_begin + C::TWT - 1) / C::TWT;

    const size_t bh_tile = (static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles;

    // per-consumer results kept until the merge
    float m_run = -CUDART_INF_F, l_acc = 0.f;
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    int tw = 0, sl = 0;

    if (warp == 0) {
        // ---------------- producer ----------------
        // In fused-append mode the CTA whose split holds the appended row's tile first writes
        // the row of its KV head into that tile (all 32 lanes quantise), then copies it in.
        const int app_tile = app_row >> 4;
        const bool owner = do_app && app_tile >= t_begin && app_tile < t_end;
        const int app_stage = owner ? (app_tile - t_begin) / C::TWT : -1;
        int issued_use[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) issued_use[i] = -1;
        // one stage: up to TWT tiles of K codes, V codes, K scales, V scales (lane 0 only)
        auto issue = [&](int k, int slot, int use) {
            const int t0 = t_begin + k * C::TWT;
            const int nt = min(C::TWT, t_end - t0);
            uint8_t *st = smem + slot * C::STAGE;
            mbar_arrive_expect_tx(full + slot, static_cast<uint32_t>(nt * C::TILE));
            bulk_g2s(st, p.k_codes + (bh_tile + t0) * C::KC, nt * C::KC, full + slot);
            bulk_g2s(st + C::TWT * C::KC, p.v_codes + (bh_tile + t0) * C::VC, nt * C::VC, full + slot);
            if constexpr (C::KS > 0)
                bulk_g2s(st + C::TWT * (C::KC + C::VC), p.k_scales + (bh_tile + t0) * C::KS, nt * C::KS, full + slot);
            if constexpr (C::VS > 0)
                bulk_g2s(st + C::TWT * (C::KC + C::VC + C::KS), p.v_scales + (bh_tile + t0) * C::VS, nt * C::VS,
                         full + slot);
            issued_use[slot] = use;
        };
        // early mode: fill the ring before the wait, up to (not including) the stage that
        // holds the row this kernel appends
        int k0 = 0;
        if (early) {
            k0 = min(n_stage, C::STAGES);
            if (app_stage >= 0) k0 = min(k0, app_stage);
            if (lane == 0) {
                for (int k = 0; k < k0; ++k) issue(k, k, 0);
                prefetch_split<C>(p, bseq, h, split, cap_rows, k0 * C::TWT);
            }
            __syncwarp();
            grid_dep_wait();
        }
        grid_dep_launch();
        if (p.win == 2 && owner) {
            // The tail's new row is the window's oldest (slot t_len mod capacity), read as f16
            // and quantised into tail position t_len first of all, so that the window's CTA,
            // which waits for the flag before it overwrites the slot, is not held up; this
            // CTA copies that tile in only at its own stage, after this write.
            const size_t tile = bh_tile + app_tile;
            const int ws_row = app_row % p.wl_cap;
            const size_t wtile = (static_cast<size_t>(bseq) * p.Hkv + h) * (p.wl_cap / kTileRows) + (ws_row >> 4);
#pragma unroll
            for (int s2 = 0; s2 < NS; ++s2) {
                const float4 xk = load_f16_row<false>(p.win_k + (wtile * NS + s2) * code_tile_bytes(KVQ_F16), ws_row & 15, lane);
                const float4 xv = load_f16_row<true>(p.win_v + (wtile * NS + s2) * code_tile_bytes(KVQ_F16), ws_row & 15, lane);
                quantize_store_vals<KT, false>(xk, const_cast<uint8_t *>(p.k_codes) + tile * C::KC + s2 * code_tile_bytes(KT),
                                               const_cast<uint8_t *>(p.k_scales) + tile * C::KS + s2 * scale_tile_bytes(KT),
                                               app_row & 15, lane);
                quantize_store_vals<VT, true>(xv, const_cast<uint8_t *>(p.v_codes) + tile * C::VC + s2 * code_tile_bytes(VT),
                                              const_cast<uint8_t *>(p.v_scales) + tile * C::VS + s2 * scale_tile_bytes(VT),
                                              app_row & 15, lane);
            }
            // before the bulk copy (async proxy) of that tile at its stage
            asm volatile("fence.proxy.async.global;\n" ::: "memory");
            __syncwarp();
            if (lane == 0) {  // the slot may now be overwritten
                __threadfence();
                atomicExch(p.evict + static_cast<size_t>(bseq) * p.Hkv + h, 1);
            }
        }
        bool ok = true;
        int slot = k0 == C::STAGES ? 0 : k0, use = k0 == C::STAGES ? 1 : 0;
        for (int k = k0; k < n_stage; ++k) {
            bool ok_k = true;
            if (lane == 0 && use > 0) {
                const int w = mbar_wait_timed(empty + slot, (use - 1) & 1, p.wait_cycles);
                if (w) atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
                ok_k = w != 2;
            }
            if (!__shfl_sync(0xffffffffu, ok_k ? 1 : 0, 0)) {
                ok = false;
                break;
            }
            if (k == app_stage && p.win != 2) {
                const size_t tile = bh_tile + app_tile;
                const int kt = app_row & 15;
                // a full window's slot is overwritten only once the tail holds its old row
                if (p.win == 1 && win_full && lane == 0)
                    wait_flag_clear(p.evict + static_cast<size_t>(bseq) * p.Hkv + h, p.wait_cycles, p.err);
                __syncwarp();
                const float *kx = p.k_new + (static_cast<size_t>(bseq) * p.Hkv + h) * p.D;
                const float *vx = p.v_new + (static_cast<size_t>(bseq) * p.Hkv + h) * p.D;
#pragma unroll
                for (int s2 = 0; s2 < NS; ++s2) {
                    quantize_store<KT, false>(kx + s2 * kSlice + 4 * lane,
                                              const_cast<uint8_t *>(p.k_codes) + tile * C::KC + s2 * code_tile_bytes(KT),
                                              const_cast<uint8_t *>(p.k_scales) + tile * C::KS + s2 * scale_tile_bytes(KT), kt, lane);
                    quantize_store<VT, true>(vx + s2 * kSlice + 4 * lane,
                                             const_cast<uint8_t *>(p.v_codes) + tile * C::VC + s2 * code_tile_bytes(VT),
                                             const_cast<uint8_t *>(p.v_scales) + tile * C::VS + s2 * scale_tile_bytes(VT), kt, lane);
                }
                // order these generic-proxy stores before the bulk copy (async proxy) that reads them
                asm volatile("fence.proxy.async.global;\n" ::: "memory");
                __syncwarp();
            }
            if (lane == 0) issue(k, slot, use);
            __syncwarp();
            if (++slot == C::STAGES) {
                slot = 0;
                ++use;
            }
        }
        // the length advance of a fused append, off the consumers' critical path
        if (appending && lane == 0) append_ticket(p, cap_rows);
        if (!ok && lane == 0) {
            s_timeout = 1;
            // let the copies already issued land before the CTA can exit
            for (int i = 0; i < C::STAGES; ++i)
                if (issued_use[i] >= 0) (void)mbar_wait(full + i, issued_use[i] & 1);
        }
    } else {
        // ---------------- consumers ----------------
        if (early) grid_dep_wait();
        grid_dep_launch();
        const int cw = warp - 1;
        tw = cw / NS;
        sl = cw % NS;
        const int g = lane >> 2, j = lane & 3;

        // Q fragments (scaled to log2 units, split into f16 hi + lo rows).  For q4_0 keys the
        // low-nibble chunk of each block is prescaled by 16 (exact) to match the high
        // nibbles, which arrive as 16c, and kcorr[b] = -8 times the block's sum of q in the
        // accumulator unit is kept for each row.
        uint8_t *kcor_row = smem + C::KCOR_OFF + sl * 128 + g * 16;
        uint8_t *qsm = smem + C::QSM_OFF + sl * (8 * 32 * 16);
        if (tw == 0) {  // one warp per slice builds what all tile-warps of the slice read
            uint32_t qa[8][4];
            float kcorr[4] = {0.f, 0.f, 0.f, 0.f};
            const bool rv = g < rows;
            const float *qrow = p.q + rmap.out_row(prow0 + (rv ? g : 0)) * p.D + sl * kSlice;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float4 x = rv ? *reinterpret_cast<const float4 *>(qrow + 16 * c + 4 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
                x.x *= p.scale_log2;
                x.y *= p.scale_log2;
                x.z *= p.scale_log2;
                x.w *= p.scale_log2;
                kcorr[c >> 1] += (x.x + x.y) + (x.z + x.w);
                const float f = ((KT == KVQ_Q4_0 || KT == KVQ_Q4_1) && (c & 1) == 0) ? 16.f : 1.f;
                split_hi_lo(x.x * f, x.z * f, qa[c][0], qa[c][1]);  // k = 2j, 2j+1  <->  d + 0, d + 2
                split_hi_lo(x.y * f, x.w * f, qa[c][2], qa[c][3]);  // k = 2j+8, 2j+9 <-> d + 1, d + 3
                *reinterpret_cast<uint4 *>(qsm + (c * 32 + lane) * 16) = make_uint4(qa[c][0], qa[c][1], qa[c][2], qa[c][3]);
            }
            if constexpr (is_nibble_type(KT)) {
                // per row and block: -8 (q4_0) or -16 (q5_0) times sum_b q, or sum_b q for the
                // types with a minimum, in the accumulator unit
                constexpr float unit = (KT == KVQ_Q4_0 || KT == KVQ_Q4_1) ? kTwo20 : kTwo24;
                constexpr float kf = (KT == KVQ_Q4_0 ? -kQ4Offset : (KT == KVQ_Q5_0 ? -16.0f : 1.0f)) / unit;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    kcorr[b] += __shfl_xor_sync(0xffffffffu, kcorr[b], 1);
                    kcorr[b] += __shfl_xor_sync(0xffffffffu, kcorr[b], 2);
                    kcorr[b] *= kf;
                }
                // kept in shared memory (one row of 4 per lane group) instead of registers
                if (j == 0)
                    *reinterpret_cast<float4 *>(kcor_row) = make_float4(kcorr[0], kcorr[1], kcorr[2], kcorr[3]);
            }
        }
        asm volatile("bar.sync 15, %0;\n" ::"r"(C::CW * 32) : "memory");  // consumer warps only
        float corr[4] = {0.f, 0.f, 0.f, 0.f};  // V types with a minimum: sum of p * lo per block (column b)
        uint32_t magic;  // 0x64006400 in a register, so each nibble mask-and-or is one instruction
        asm volatile("mov.b32 %0, 0x64006400;\n" : "=r"(magic));
        float4 *xchg = reinterpret_cast<float4 *>(smem + C::RING);
        int *xflag = reinterpret_cast<int *>(smem + C::RING + C::XCHG_SC);
        bool dead = false;
        // keys of this lane inside a tile: A=2j, B=2j+1, C=8+2j, D=9+2j
        const int kofs[4] = {2 * j, 2 * j + 1, 8 + 2 * j, 9 + 2 * j};


        int slot = 0, use = 0;
        for (int k = 0; k < n_stage; ++k) {
            if (!dead) {
                const int w = mbar_wait_timed(full + slot, use & 1, p.wait_cycles);
                if (w) atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
                if (w == 2) {  // gave up: this CTA publishes an empty triple
                    dead = true;
                    s_timeout = 1;
                }
            }
            const int tA = t_begin + (k * C::TW + tw) * TPW;  // first tile of this warp in the stage
            if (tA < t_end) {
                const uint8_t *st = smem + slot * C::STAGE;
                float sc[TPW][4];
#pragma unroll
                for (int t = 0; t < TPW; ++t) {
                    const int ti = tw * TPW + t;  // tile index inside the stage
                    tile_scores<KT>(st + ti * C::KC + sl * code_tile_bytes(KT),
                                    st + C::TWT * (C::KC + C::VC) + ti * C::KS + sl * scale_tile_bytes(KT), qsm, kcor_row, lane,
                                    j, sc[t]);
                }
                // f16 overflow guard: p = exp2(s - m_run) may reach 2^kTau before the running
                // maximum is moved, so a tile pair holding a V scale with |scale| >= 256 (or
                // inf/nan bits) takes an exact rescale instead.  The exponent test on an OR of
                // the scale words may over-report, which only costs that exact rescale.
                auto guard = [&]() {
                    bool x = false;
                    if constexpr (VT != KVQ_F16) {
                        uint32_t e = 0;
#pragma unroll
                        for (int t = 0; t < TPW; ++t) {
                            const uint8_t *vs = st + C::TWT * (C::KC + C::VC + C::KS) + (tw * TPW + t) * C::VS + sl * scale_tile_bytes(VT);
                            const uint4 sc0 = lds128(vs + j * 32), sc1 = lds128(vs + j * 32 + 16);
                            e |= (sc0.x | sc0.y | sc0.z) | (sc0.w | sc1.x | sc1.y) | (sc1.z | sc1.w);
                        }
                        x = __any_sync(0xffffffffu, __vcmpgeu2(e & 0x7c007c00u, 0x5c005c00u) != 0);
                    }
                    return x;
                };
                bool exact = false;
                if constexpr (NS == 2) exact = guard();
                if constexpr (NS == 2) {
                    // the two slice-warps of this tile pair add their partial scores, and agree
                    // on the guard (each saw the V scales of its own slice only): their running
                    // maxima must move together, as the merge keeps one per tile pair
                    const int xi = tw * 2;
#pragma unroll
                    for (int t = 0; t < TPW; ++t) {
                        float4 *mine = xchg + ((xi + sl) * TPW + t) * 32;
                        mine[lane] = make_float4(sc[t][0], sc[t][1], sc[t][2], sc[t][3]);
                    }
                    if (lane == 0) xflag[xi + sl] = exact ? 1 : 0;
                    asm volatile("bar.sync %0, 64;\n" ::"r"(1 + tw) : "memory");
                    exact = exact || xflag[xi + 1 - sl] != 0;
#pragma unroll
                    for (int t = 0; t < TPW; ++t) {
                        const float4 os = xchg[((xi + 1 - sl) * TPW + t) * 32 + lane];
                        sc[t][0] += os.x;
                        sc[t][1] += os.y;
                        sc[t][2] += os.z;
                        sc[t][3] += os.w;
                    }
                    asm volatile("bar.sync %0, 64;\n" ::"r"(1 + tw) : "memory");  // the buffer is free again
                }
                // rows past the length, and a second tile past this split's range (it belongs
                // to the next split and was not loaded), are masked out
                bool vmask[TPW][4];
                // with several queries per sequence, row g's keys also end at its causal limit
                const int L_split = min(L, t_end * kTileRows);
                const bool any_partial = MQ ? (tA + TPW) * kTileRows > min(L_split, L - n_q + 1)
                                            : (tA + TPW) * kTileRows > L_split;  // warp-uniform
                if (any_partial) {
#pragma unroll
                    for (int t = 0; t < TPW; ++t) {
                        const int nvalid = min(kTileRows, max(0, L_split - (tA + t) * kTileRows));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            vmask[t][i] = kofs[i] < nvalid;
                            if (!vmask[t][i]) sc[t][i] = -CUDART_INF_F;
                        }
                    }
                    if constexpr (MQ) {
                        // draft verify: query i of the draft sees positions < L - n_q + 1 + i
                        const int lim = g < rows ? L - n_q + 1 + (r0 + g) / p.G : L;
#pragma unroll
                        for (int t = 0; t < TPW; ++t)
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                if ((tA + t) * kTileRows + kofs[i] >= lim) sc[t][i] = -CUDART_INF_F;
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < TPW; ++t)
#pragma unroll
                        for (int i = 0; i < 4; ++i) vmask[t][i] = true;
                }

                // ---- online softmax (log2 units) over TPW x 16 keys, lazy rescale ----
                float mt = -CUDART_INF_F;
#pragma unroll
                for (int t = 0; t < TPW; ++t) mt = fmaxf(mt, fmaxf(fmaxf(sc[t][0], sc[t][1]), fmaxf(sc[t][2], sc[t][3])));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                if constexpr (NS == 1) exact = guard();
                const bool need = mt > m_run + (exact ? 0.f : kTau);
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? mt : m_run;
                    const float alpha = (m_run == -CUDART_INF_F) ? 0.f : ex2(m_run - m_new);
                    m_run = m_new;
                    l_acc *= alpha;
                    if constexpr (has_min(VT)) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) corr[i] *= alpha;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        o[i][0] *= alpha;
                        o[i][1] *= alpha;
                        o[i][2] *= alpha;
                        o[i][3] *= alpha;
                    }
                }
                float pk[TPW][4];
                // a draft-verify row may have no position yet (m_run = -inf): its p are 0
                float m_use = m_run;
                if constexpr (MQ) m_use = m_run == -CUDART_INF_F ? 0.f : m_run;
#pragma unroll
                for (int t = 0; t < TPW; ++t) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) pk[t][i] = ex2(sc[t][i] - m_use);
                    l_acc += (pk[t][0] + pk[t][1]) + (pk[t][2] + pk[t][3]);
                }

                // ---- O += P V (masking code only for the rare tile that crosses the end) ----
                if (!any_partial) {
#pragma unroll
                    for (int t = 0; t < TPW; ++t) {
                        const int ti = tw * TPW + t;
                        tile_pv<VT, false>(st + C::TWT * C::KC + ti * C::VC + sl * code_tile_bytes(VT),
                                           st + C::TWT * (C::KC + C::VC + C::KS) + ti * C::VS + sl * scale_tile_bytes(VT), pk[t],
                                           vmask[t], lane, j, o, magic, corr);
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < TPW; ++t) {
                        const int ti = tw * TPW + t;
                        tile_pv<VT, true>(st + C::TWT * C::KC + ti * C::VC + sl * code_tile_bytes(VT),
                                          st + C::TWT * (C::KC + C::VC + C::KS) + ti * C::VS + sl * scale_tile_bytes(VT), pk[t],
                                          vmask[t], lane, j, o, magic, corr);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && !dead) mbar_arrive(empty + slot);
            if (++slot == C::STAGES) {
                slot = 0;
                ++use;
            }
        }
        // V types with a minimum: add sum of p * lo of each block to its values (corr column
        // b, held by lane 4g + b/2 for the hi and lo rows)
        if constexpr (has_min(VT)) {
            const float v0 = corr[0] + corr[2], v1 = corr[1] + corr[3];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const float ct = __shfl_sync(0xffffffffu, (b & 1) ? v1 : v0, (lane & ~3) | (b >> 1));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[4 * b + i][0] += o[4 * b + i][2] + ct;
                    o[4 * b + i][1] += o[4 * b + i][3] + ct;
                    o[4 * b + i][2] = 0.f;
                    o[4 * b + i][3] = 0.f;
                }
            }
        }
        // q8_0 V: o to real units
        if constexpr (VT == KVQ_Q8_0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o[i][0] = (o[i][0] + o[i][2]) * kTwo24;
                o[i][1] = (o[i][1] + o[i][3]) * kTwo24;
                o[i][2] = 0.f;
                o[i][3] = 0.f;
            }
        }
        // row sums over the four lanes of a row
        l_acc += __shfl_xor_sync(0xffffffffu, l_acc, 1);
        l_acc += __shfl_xor_sync(0xffffffffu, l_acc, 2);
    }

    // ---------------- merge the tile-warps of this CTA ----------------
    __syncthreads();  // the ring is free from here on
    constexpr int D = C::D;
    float *Ob = reinterpret_cast<float *>(smem);                    // [TW][8][D]
    float *mb = Ob + C::TW * kMaxRowsPerGroup * D;                 // [TW][8]
    float *lb = mb + C::TW * kMaxRowsPerGroup;                     // [TW][8]
    if (warp > 0) {
        const int g = lane >> 2, j = lane & 3;
        float *orow = Ob + (tw * kMaxRowsPerGroup + g) * D + sl * kSlice;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            // thread holds d = 32b + 4j + {0..3} (ptiles 0,1 of block b) and +16 (ptiles 2,3)
            const float4 lo4 = make_float4(o[4 * b + 0][0] + o[4 * b + 0][2], o[4 * b + 1][0] + o[4 * b + 1][2],
                                           o[4 * b + 0][1] + o[4 * b + 0][3], o[4 * b + 1][1] + o[4 * b + 1][3]);
            const float4 hi4 = make_float4(o[4 * b + 2][0] + o[4 * b + 2][2], o[4 * b + 3][0] + o[4 * b + 3][2],
                                           o[4 * b + 2][1] + o[4 * b + 2][3], o[4 * b + 3][1] + o[4 * b + 3][3]);
            *reinterpret_cast<float4 *>(orow + 32 * b + 4 * j) = lo4;
            *reinterpret_cast<float4 *>(orow + 32 * b + 16 + 4 * j) = hi4;
        }
        if (sl == 0 && j == 0) {
            mb[tw * kMaxRowsPerGroup + g] = m_run;
            lb[tw * kMaxRowsPerGroup + g] = l_acc;
        }
    }
    __syncthreads();
    const bool timed_out = s_timeout != 0;
    const bool single = (ns == 1) && fused && p.merge_slots == 0;
    for (int idx = threadIdx.x; idx < rows * (D / 4); idx += blockDim.x) {
        const int g = idx / (D / 4), dq = idx % (D / 4);
        float M = -CUDART_INF_F;
#pragma unroll
        for (int t = 0; t < C::TW; ++t) M = fmaxf(M, mb[t * kMaxRowsPerGroup + g]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int t = 0; t < C::TW; ++t) {
                const float w = ex2(mb[t * kMaxRowsPerGroup + g] - M);  // exp2(-inf) = 0
                const float4 v = reinterpret_cast<const float4 *>(Ob + (t * kMaxRowsPerGroup + g) * D)[dq];
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
                lsum = fmaf(w, lb[t * kMaxRowsPerGroup + g], lsum);
            }
        }
        if (single) {
            const size_t orow = rmap.out_row(prow0 + g);
            if (p.ext_out) {  // one more triple (ext_out, lse, l = 1), in log2 units here
                const float mx = p.ext_lse[orow] * 1.44269504088896340736f;
                const float Mn = fmaxf(M, mx);
                if (Mn != -CUDART_INF_F) {
                    const float a = M == -CUDART_INF_F ? 0.f : ex2(M - Mn);
                    const float bw = mx == -CUDART_INF_F ? 0.f : ex2(mx - Mn);
                    const float4 x = reinterpret_cast<const float4 *>(p.ext_out + orow * D)[dq];
                    acc = make_float4(fmaf(bw, x.x, a * acc.x), fmaf(bw, x.y, a * acc.y), fmaf(bw, x.z, a * acc.z),
                                      fmaf(bw, x.w, a * acc.w));
                    lsum = fmaf(a, lsum, bw);
                    M = Mn;
                }
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            reinterpret_cast<float4 *>(p.out + orow * D)[dq] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (dq == 0 && p.lse) p.lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -CUDART_INF_F;
        } else {
            // a CTA whose waits gave up publishes an empty triple (its tiles were not all
            // read); the result is then undefined and the error word says so
            const size_t pr = (prow0 + g) * p.part_stride + p.part_base + split;
            reinterpret_cast<float4 *>(p.part_o + pr * D)[dq] = timed_out ? make_float4(0.f, 0.f, 0.f, 0.f) : acc;
            if (dq == 0) {
                p.part_m[pr] = (M == -CUDART_INF_F || timed_out) ? -CUDART_INF_F : M * kLn2;
                p.part_l[pr] = timed_out ? 0.f : lsum;
            }
        }
    }
    // A CTA that timed out still takes its merge arrivals, so the arrival counters of the
    // workspace end at zero once every CTA of the launch has finished.
    if (!fused || single || !MERGE) return;

    const size_t unit = (static_cast<size_t>(bseq) * p.Hkv + h) * p.QG + qg;
    split_merge(p, p.merge_slots ? p.merge_slots : ns, p.part_base + split, rows, D, prow0, unit, rmap, s_flag, smem);
}

template <int KT, int VT, int NS, bool MQ>
__global__ void __launch_bounds__(Cfg<KT, VT, NS>::THREADS, Cfg<KT, VT, NS>::MIN_CTAS) decode_kernel(const DecodeParams p, const int fused) {
    stamp(p, 0);
    decode_body<KT, VT, NS, MQ>(p, fused, blockIdx.x);
    stamp(p, kStamps - 1);
}

// One launch over an f16 window and a quantised tail of the same sequences: splits
// [0, nw) decode the window, the rest the tail; both regions publish their triples into
// one set of merge slots (merge_slots = all splits of the grid), merged exactly as one.
template <int KT, int VT, int NS>
__global__ void __launch_bounds__(Cfg<KT, VT, NS>::THREADS, Cfg<KT, VT, NS>::MIN_CTAS)
    dual_kernel(const DecodeParams pw, const DecodeParams pt, const int nw) {
    constexpr int TWW = Cfg<KT, VT, NS>::TW;  // the window body runs with the tail's warp count
    static_assert(Cfg<KVQ_F16, KVQ_F16, NS, TWW>::THREADS == Cfg<KT, VT, NS>::THREADS, "one block size");
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_flag;
    if (static_cast<int>(blockIdx.x) < nw)
        decode_body<KVQ_F16, KVQ_F16, NS, false, TWW, false>(pw, 1, blockIdx.x);
    else
        decode_body<KT, VT, NS, false, 0, false>(pt, 1, blockIdx.x - nw);
    // One merge for both regions, after either body: every CTA has published its triple at
    // slot blockIdx.x (window splits 0 .. nw - 1, tail splits nw ..); the two parameter
    // sets share the workspace, the outputs and merge_slots.
    const int bseq = blockIdx.z / pt.QG, qg = blockIdx.z % pt.QG, h = blockIdx.y;
    const int rows = min(kMaxRowsPerGroup, pt.G - qg * kMaxRowsPerGroup);
    const size_t prow0 = (static_cast<size_t>(bseq) * pt.Hkv + h) * pt.G + qg * kMaxRowsPerGroup;
    const size_t unit = (static_cast<size_t>(bseq) * pt.Hkv + h) * pt.QG + qg;
    split_merge(pt, pt.merge_slots, static_cast<int>(blockIdx.x), rows, NS * kSlice, prow0, unit, RowMap{1, pt.G, pt.Hq, pt.Hkv},
                s_flag, smem);
}

constexpr int kMaxDevices = 64;

template <int KT, int VT, int NS, bool MQ>
cudaError_t configure_t(int dev) {
    // the dynamic shared-memory opt-in, once per (instance, device)
    static bool configured[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<KT, VT, NS, MQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<KT, VT, NS>::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    return cudaSuccess;
}

template <int KT, int VT, int NS, bool MQ>
cudaError_t occupancy_t(int *ctas) {
    using C = Cfg<KT, VT, NS>;
    // resident CTAs per SM, queried once per (instance, device)
    static int cached[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = configure_t<KT, VT, NS, MQ>(dev);
    if (e != cudaSuccess) return e;
    if (cached[dev] == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<KT, VT, NS, MQ>, C::THREADS, C::SMEM);
        if (e != cudaSuccess) return e;
        cached[dev] = n > 0 ? n : 1;
    }
    *ctas = cached[dev];
    return cudaSuccess;
}

// SM count of a device, queried once
inline cudaError_t sm_count(int dev, int *n) {
    static int cached[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (cached[dev] == 0) {
        int v = 0;
        const cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cached[dev] = v > 0 ? v : 1;
    }
    *n = cached[dev];
    return cudaSuccess;
}

template <int KT, int VT, int NS, bool MQ>
cudaError_t launch_decode_t(const DecodeParams &p, bool fused, cudaStream_t stream) {
    using C = Cfg<KT, VT, NS>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = configure_t<KT, VT, NS, MQ>(dev);
    int occ = 1, sms = 0;
    if (e == cudaSuccess) e = occupancy_t<KT, VT, NS, MQ>(&occ);
    if (e == cudaSuccess) e = sm_count(dev, &sms);
    if (e != cudaSuccess) return e;
    // a grid that is resident at once lets the last CTAs of a row group wait for the rest
    DecodeParams q = p;
    const long long ctas = static_cast<long long>(p.n_splits) * p.Hkv * p.B * p.QG;
    q.wide = (fused && ctas <= static_cast<long long>(occ) * sms) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_splits, p.Hkv, p.B * p.QG);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<KT, VT, NS, MQ>, q, fused ? 1 : 0);
}


template <int KT, int VT, int NS>
cudaError_t launch_dual_t(const DecodeParams &pw, const DecodeParams &pt, int nw, cudaStream_t stream) {
    using C = Cfg<KT, VT, NS>;
    using CW_ = Cfg<KVQ_F16, KVQ_F16, NS, C::TW>;  // the window body's configuration
    constexpr int kSmem = CW_::SMEM > C::SMEM ? CW_::SMEM : C::SMEM;
    static bool configured[kMaxDevices] = {};
    static int occ_cached[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(dual_kernel<KT, VT, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dual_kernel<KT, VT, NS>, C::THREADS, kSmem);
        if (e != cudaSuccess) return e;
        occ_cached[dev] = n > 0 ? n : 1;
        configured[dev] = true;
    }
    int sms = 0;
    e = sm_count(dev, &sms);
    if (e != cudaSuccess) return e;
    DecodeParams a = pw, b = pt;
    const long long ctas = static_cast<long long>(pt.merge_slots) * pt.Hkv * pt.B * pt.QG;
    a.wide = b.wide = ctas <= static_cast<long long>(occ_cached[dev]) * sms ? 1 : 0;
    // the two-region append has CTAs wait on one another: only for a grid resident at once
    if (pw.win && !a.wide) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pt.merge_slots, pt.Hkv, pt.B * pt.QG);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dual_kernel<KT, VT, NS>, a, b, nw);
}

}  // namespace

#define KVQ_DISPATCH(KT_, VT_, NS_, CALL, MQ_)                                   \
    if (type_k == KT_ && type_v == VT_ && ns == NS_) return CALL<KT_, VT_, NS_, MQ_>
#define KVQ_DISPATCH_ALL(CALL, MQ_, ARGS)                 \
    KVQ_DISPATCH(KVQ_F16, KVQ_F16, 1, CALL, MQ_) ARGS;    \
    KVQ_DISPATCH(KVQ_F16, KVQ_Q8_0, 1, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_F16, KVQ_Q4_0, 1, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_F16, 1, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q8_0, 1, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q4_0, 1, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_F16, 1, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_Q8_0, 1, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_Q4_0, 1, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_F16, KVQ_F16, 2, CALL, MQ_) ARGS;    \
    KVQ_DISPATCH(KVQ_F16, KVQ_Q8_0, 2, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_F16, KVQ_Q4_0, 2, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_F16, 2, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q8_0, 2, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q4_0, 2, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_F16, 2, CALL, MQ_) ARGS;   \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_Q8_0, 2, CALL, MQ_) ARGS;  \
    KVQ_DISPATCH(KVQ_Q4_0, KVQ_Q4_0, 2, CALL, MQ_) ARGS;

}  // namespace kvq
