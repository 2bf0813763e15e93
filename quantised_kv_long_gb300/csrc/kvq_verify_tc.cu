// kvq_verify_tc.cu -- draft verify on the fifth-generation tensor cores (tcgen05, tensor
// memory): all n_q * G query rows of a (sequence, KV head) form one M = 128 tile.
//
// Method: the same exact attention as kvq_decode_verify ("HAL #582 -- per-layer KV
// compression study", section 5 P0: the typed reader serves decode batches of up to 16
// query rows; section 5 P2: softmax partials of key ranges combine without loss).  With up to 128
// query rows per KV head the products are real dense tiles, so each key chunk is
// dequantised once into tensor-core operands and shared by every row, instead of once per
// group of 8 rows as in the register-operand kernel.
//
// Per CTA: one (key split, KV head, sequence).  Keys go in chunks of 32 (two 16-row tiles).
//   S = Q K^T   : A = Q (128 rows x D, f16 hi in shared memory, f16 lo in tensor memory),
//                 B = K^ (32 keys x D, f16 hi and lo, shared memory), D = S in tensor memory.
//   O += P V    : A = P (128 rows x 32 keys, f16 hi and lo, tensor memory),
//                 B = V^ (32 keys x D, f16 hi and lo, shared memory), O in tensor memory.
// K^ and V^ are the dequantised values x = scale * code as an exact f16 pair hi + lo (a
// code of at most 8 bits times an f16 scale has at most 19 significant bits), times 2^-e
// for a per-chunk e that keeps |x| below 2^14; S is multiplied by 2^e_k afterwards and P is
// formed as p * 2^e_v, both exact.  Products are hi*hi + hi*lo + lo*hi (the lo*lo term is
// below 2^-21 relative); accumulation is fp32.
//
// Warp roles (512 threads): warp 0 streams the chunks' tiles into a shared-memory ring
// with 1-D bulk copies (as the decode kernel); warp 1 owns the tensor memory and one of its
// threads issues every MMA; warps 2-5 hold one query row per thread (softmax, P, the
// rescale of O, the epilogue); warps 6-15 convert codes into K^ and V^.  Every wait is
// bounded and reports KVQ_DEVERR_TIMEOUT.
#include "kvq_decode_kernel.cuh"

namespace kvq {
namespace {

// ---- tcgen05 / tensor-memory helpers (inline PTX) ----
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor, no swizzle: the operand is stored as 8-row x 16-byte core
// matrices; lbo = byte distance between core matrices adjacent along K, sbo = between
// core matrices adjacent along M (or N).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3fffu) | (static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32) | (static_cast<uint64_t>(1) << 46);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tc_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                 ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t prmt_sel(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;\n" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t prmt2_sel(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Byte offset of element (row, k) in a no-swizzle K-major operand with kext elements per row.
__device__ __forceinline__ int kmaj(int row, int k, int kext) {
    return (row >> 3) * (kext * 16) + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

template <int KT, int VT, int NS>
struct TcCfg {
    static constexpr int D = NS * kSlice;
    static constexpr int M = 128;  // query rows of the tile
    static constexpr int NK = 32;  // keys per chunk: two 16-row tiles
    static constexpr int KC = code_tile_bytes(KT) * NS, VC = code_tile_bytes(VT) * NS;
    static constexpr int KS = scale_tile_bytes(KT) * NS, VS = scale_tile_bytes(VT) * NS;
    static constexpr int TILE = KC + VC + KS + VS;
    static constexpr int STAGE = 2 * TILE;
    static constexpr int QHI = M * D * 2;     // Q hi, K-major (rows x D)
    static constexpr int KHAT = NK * D * 2;   // one of K^ hi / lo, K-major (keys x D)
    static constexpr int VHAT = D * NK * 2;   // one of V^ hi / lo, K-major (values x keys)
    static constexpr bool K_LO = KT != KVQ_F16;  // f16 codes are exact f16 values
    static constexpr bool V_LO = VT != KVQ_F16;
    static constexpr int QT_ROW = 80;             // Q lo transpose rows: 32 halves + 16 bytes of padding
    static constexpr int QT = 4 * 32 * QT_ROW;      // one 32-row block per softmax warp
    static constexpr int OPS = QHI + 2 * (K_LO ? 2 : 1) * KHAT + (V_LO ? 2 : 1) * VHAT + QT;
    static constexpr int O_ROW = D * 4 + 16;       // epilogue staging of O (padded rows)
    static constexpr int BUDGET = 232448 - 512;  // shared memory of one CTA (227 KiB) less the static variables
    static constexpr int STAGES = (BUDGET - OPS - 512) / STAGE >= 3 ? 3 : 2;  // 512: barriers
    static constexpr int RING = STAGES * STAGE;
    static constexpr int OFF_Q = RING;
    static constexpr int OFF_K = OFF_Q + QHI;                      // [buffer 0, 1][hi, lo]
    static constexpr int OFF_V = OFF_K + 2 * (K_LO ? 2 : 1) * KHAT;  // [hi, lo]
    static constexpr int OFF_QT = OFF_V + (V_LO ? 2 : 1) * VHAT;
    static constexpr int OFF_BAR = (OFF_QT + QT + 15) / 16 * 16;
    // barriers: full[STAGES], empty[STAGES], k_ready[2], v_ready, s_done[2] (Q hi stream),
    // s_done_b[2] (Q lo stream), s_free (+1 spare), p_ready (+1 spare), pv_done, e_ready[4],
    // q_ready, drain; then e values [4][2] and the tensor-memory address
    static constexpr int NBAR = 2 * STAGES + 2 + 1 + 2 + 2 + 2 + 2 + 1 + 4 + 2;
    static constexpr int OFF_E = OFF_BAR + NBAR * 8;
    static constexpr int OFF_TADDR = OFF_E + 4 * 2 * 4;
    static constexpr int SMEM = OFF_TADDR + 16;
    // tensor memory columns: O [0, D), S [D, D + 2 NK) as [Q hi K^ hi, Q hi K^ lo], S2 [D + 2 NK,
    // D + 3 NK) (Q lo K^ hi), P [D + 3 NK, D + 4 NK) as [hi NK / 2, lo NK / 2], Q lo [D + 4 NK, D + 4 NK + D / 2)
    static constexpr int T_O = 0, T_S = D, T_S2 = D + 2 * NK, T_P = D + 3 * NK, T_Q = D + 4 * NK;
    static constexpr int TCOLS = 512;
    // converters: warps 6 .. 13; warps 14 and 15 issue the Q lo and P V^ instructions.  16
    // warps leave 128 registers a thread (an SM sub-partition holds 4 warps)
    static constexpr int CONV_THREADS = 256;
    static constexpr int THREADS = 6 * 32 + CONV_THREADS + 64;
    static_assert(T_Q + D / 2 <= TCOLS, "tensor memory");
    static_assert(SMEM <= BUDGET, "shared memory");
    static_assert(M * O_ROW <= OFF_QT, "epilogue staging fits the operand memory");
    static_assert((K_LO ? 2 : 1) * KHAT + (V_LO ? 2 : 1) * VHAT >= 4 * 32 * QT_ROW, "Q transpose blocks of the converters");
    static_assert(NK * M <= TCOLS * 128, "tiles");
};

// Largest |scale| of one chunk's valid keys (0 for none), by one warp: the chunk's scales are
// 2 tiles x NSL slices x 128 bytes; lane l takes the 16 bytes at 16 l, which hold blocks 2h,
// 2h + 1 (h = l & 1) of keys 2j, 2j + 1 (first word of each pair) and 8 + 2j, 9 + 2j (second),
// j = (l % 8) / 2, of tile l / (8 NSL).
// Returns 0 without the reduction when no scale needs an exponent (cmax * |d| <= 2^14 for
// every one: the common case), so that the warp votes once instead of reducing.
template <int NSL>
__device__ __forceinline__ float chunk_scale_max(const uint8_t *sc, int nvalid_keys, float cmax) {
    constexpr int NG = 2 * NSL * kScaleTile / 16;
    const int lane = threadIdx.x & 31;
    uint32_t m = 0u;  // packed |f16| pair
    if (lane < NG) {
        uint4 w = *reinterpret_cast<const uint4 *>(sc + lane * 16);
        if (nvalid_keys < 2 * kTileRows) {
            const int ka = (lane / (8 * NSL)) * kTileRows + 2 * ((lane % 8) >> 1), kb = ka + 8;
            auto mask = [&](uint32_t x, int k) {
                return k >= nvalid_keys ? 0u : (k + 1 >= nvalid_keys ? (x & 0x0000ffffu) : x);
            };
            w = make_uint4(mask(w.x, ka), mask(w.y, kb), mask(w.z, ka), mask(w.w, kb));
        }
        const __half2 a = __hmax2(__habs2(u32_as_h2(w.x)), __habs2(u32_as_h2(w.y)));
        const __half2 b = __hmax2(__habs2(u32_as_h2(w.z)), __habs2(u32_as_h2(w.w)));
        m = h2_as_u32(__hmax2(a, b));
    }
    float2 f = __half22float2(u32_as_h2(m));
    if (!__any_sync(0xffffffffu, cmax * fmaxf(f.x, f.y) > 16384.f)) return 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = h2_as_u32(__hmax2(u32_as_h2(m), u32_as_h2(__shfl_xor_sync(0xffffffffu, m, o))));
    f = __half22float2(u32_as_h2(m));
    return fmaxf(f.x, f.y);
}

// exponent e >= 0 with cmax * dmax * 2^-e < 2^14
__device__ __forceinline__ int chunk_exp(float x) {
    if (!(x > 16384.f)) return 0;
    return ilogbf(x) - 13;
}

// 2^e for an integer e in [-126, 127], exactly
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + e) << 23); }

template <int KT, int VT, int NS>
__global__ void __launch_bounds__(TcCfg<KT, VT, NS>::THREADS, 1) verify_tc_kernel(const DecodeParams p) {
    using C = TcCfg<KT, VT, NS>;
    constexpr int D = C::D, NK = C::NK, M = C::M;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_flag, s_timeout;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, h = blockIdx.y, bseq = blockIdx.z;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars, *empty = full + C::STAGES, *k_ready = empty + C::STAGES, *v_ready = k_ready + 2;
    uint64_t *s_done = v_ready + 1, *s_done_b = s_done + 2, *s_free = s_done_b + 2, *p_ready = s_free + 2;
    uint64_t *pv_done = p_ready + 2;
    uint64_t *e_ready = pv_done + 1, *q_ready = e_ready + 4, *drain = q_ready + 1;
    int *e_val = reinterpret_cast<int *>(smem + C::OFF_E);  // [4][2]: e_k, e_v of chunk c at slot c % 4
    uint32_t *taddr_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TADDR);
    const long long limit = p.wait_cycles;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(k_ready + i, 1);
            mbar_init(s_done + i, 1);
            mbar_init(s_done_b + i, 1);
        }
        mbar_init(s_free, 4);
        mbar_init(p_ready, 4);
        mbar_init(v_ready, 1);
        mbar_init(pv_done, 1);
        mbar_init(q_ready, 8);
        mbar_init(drain, 3);
        for (int i = 0; i < 4; ++i) mbar_init(e_ready + i, 1);
        fence_mbar_init();
        s_timeout = 0;
    }
    if (warp == 1) {  // tensor memory for this CTA (one CTA per SM)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(taddr_slot)),
                     "r"(C::TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *taddr_slot;

    // Queries, lengths and the workspace are read after the previous kernel of the stream.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int cap_rows = p.cap_tiles * kTileRows;
    int L = __ldcg(p.len + bseq);
    L = L < 0 ? 0 : (L > cap_rows ? cap_rows : L);
    const int T = (L + kTileRows - 1) / kTileRows;
    const int ns = max(1, min(p.n_splits, T));
    const int n_q = p.n_q;
    const int R = n_q * p.G;  // query rows of this (sequence, KV head), at most M
    const size_t prow0 = (static_cast<size_t>(bseq) * p.Hkv + h) * R;
    const RowMap rmap{n_q, p.G, p.Hq, p.Hkv};
    if (split >= ns) {  // no keys: nothing to publish (the merge counts ns splits)
        tc_fence_before();
        __syncthreads();
        if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tbase), "r"(C::TCOLS));
        return;
    }
    int t_begin, t_end;
    split_range(p, T, split, t_begin, t_end);
    const int NC = (t_end - t_begin + 1) / 2;  // chunks of two tiles
    const int key_end = min(L, t_end * kTileRows);  // keys past this are not loaded or not valid
    const size_t bh_tile = (static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles;

    uint8_t *qhi = smem + C::OFF_Q;
    auto khat = [&](int buf, int lo) { return smem + C::OFF_K + (buf * (C::K_LO ? 2 : 1) + lo) * C::KHAT; };
    auto vhat = [&](int lo) { return smem + C::OFF_V + lo * C::VHAT; };
    constexpr uint32_t IDESC_S = tc_idesc(M, NK), IDESC_S2 = tc_idesc(M, C::K_LO ? 2 * NK : NK), IDESC_O = tc_idesc(M, D);

    // Q: scaled to log2 units, hi into shared memory (A of S), lo into tensor memory.  Two
    // warps share the 32 rows of each tensor-memory lane quarter (a softmax warp takes the
    // first half of the values, a converter warp the second).  A warp loads its rows with
    // coalesced 16-byte requests (one covers 4 rows x 32 values), writes hi straight to the
    // operand and lo through a padded row-major block `qt`, from which every lane takes its
    // own row for the tensor-memory store.
    auto stage_q = [&](int quarter, int d_begin, int d_end, uint8_t *qt) {
        const int R0 = 32 * quarter;
        const uint32_t trow = tbase + (static_cast<uint32_t>(R0) << 16);
        const float sl = p.scale_log2;
        // the rows of this lane's requests, R0 + 4i + lane / 8: row = G qi + g of the KV head is
        // query head h G + g of draft position qi
        const float4 *qsrc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = R0 + 4 * i + (lane >> 3);
            const size_t qrow = (static_cast<size_t>(bseq) * n_q + row / p.G) * p.Hq + static_cast<size_t>(h) * p.G + row % p.G;
            qsrc[i] = row < R ? reinterpret_cast<const float4 *>(p.q + qrow * D) + (lane & 7) : nullptr;
        }
        // loads of the next 32 values are in flight while this block is converted
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = qsrc[i] ? __ldg(qsrc[i] + d_begin / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int kb0 = d_begin; kb0 < d_end; kb0 += 32) {
            float4 nv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                nv[i] = (qsrc[i] && kb0 + 32 < d_end) ? __ldg(qsrc[i] + (kb0 + 32) / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 x = v[i];
                const int row = R0 + 4 * i + (lane >> 3), dim = kb0 + 4 * (lane & 7);
                uint32_t h0, h1, l0, l1;
                split_hi_lo(x.x * sl, x.y * sl, h0, l0);
                split_hi_lo(x.z * sl, x.w * sl, h1, l1);
                *reinterpret_cast<uint2 *>(qhi + kmaj(row, dim, D)) = make_uint2(h0, h1);
                *reinterpret_cast<uint2 *>(qt + (4 * i + (lane >> 3)) * C::QT_ROW + 8 * (lane & 7)) = make_uint2(l0, l1);
            }
            __syncwarp();
            uint32_t lo32[16];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 w = *reinterpret_cast<const uint4 *>(qt + lane * C::QT_ROW + 16 * j);
                lo32[4 * j] = w.x;
                lo32[4 * j + 1] = w.y;
                lo32[4 * j + 2] = w.z;
                lo32[4 * j + 3] = w.w;
            }
            __syncwarp();
            tc_st16(trow + C::T_Q + kb0 / 2, lo32);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = nv[i];
        }
        tc_wait_st();
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
    };

    if (warp == 0) {
        // ---------------- producer: one ring stage = one chunk (two tiles) ----------------
        int issued_use[4] = {-1, -1, -1, -1};
        bool ok = true;
        for (int c = 0; c < NC && ok; ++c) {
            const int slot = c % C::STAGES, use = c / C::STAGES;
            if (lane == 0) {
                if (use > 0 && !mbar_wait(empty + slot, (use - 1) & 1, limit)) ok = false;
                if (ok) {
                    const int t0 = t_begin + 2 * c, nt = min(2, t_end - t0);
                    uint8_t *st = smem + slot * C::STAGE;
                    mbar_arrive_expect_tx(full + slot, static_cast<uint32_t>(nt * C::TILE));
                    bulk_g2s(st, p.k_codes + (bh_tile + t0) * C::KC, nt * C::KC, full + slot);
                    bulk_g2s(st + 2 * C::KC, p.v_codes + (bh_tile + t0) * C::VC, nt * C::VC, full + slot);
                    if constexpr (C::KS > 0)
                        bulk_g2s(st + 2 * (C::KC + C::VC), p.k_scales + (bh_tile + t0) * C::KS, nt * C::KS, full + slot);
                    if constexpr (C::VS > 0)
                        bulk_g2s(st + 2 * (C::KC + C::VC) + 2 * C::KS, p.v_scales + (bh_tile + t0) * C::VS, nt * C::VS,
                                 full + slot);
                    issued_use[slot] = use;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0) {
            if (!ok) {
                atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
                s_timeout = 1;
            }
            for (int i = 0; i < C::STAGES; ++i)  // every copy lands before the CTA reuses or frees its memory
                if (issued_use[i] >= 0) (void)mbar_wait(full + i, issued_use[i] & 1);
        }
    } else if (warp == 1 || warp >= 14) {
        // ---------------- MMA issue: three threads, one instruction stream each ----------------
        // An issuing thread waits about 120 cycles per small-N instruction, so the streams run
        // in parallel: warp 1 issues S = Q hi [K^ hi; K^ lo]^T (N = 2 NK: Q hi read once for
        // both halves), warp 14 S2 = Q lo K^ hi^T, warp 15 O += P V^.  S and S2 of chunk c + 1
        // are issued as soon as K^(c + 1) is converted and the softmax warps have read S(c)
        // and S2(c); O += P(c) V^(c) once P(c) and V^(c) are written.
        if (lane == 0) {
            bool ok = mbar_wait(q_ready, 0, limit);  // Q hi (shared) and Q lo (tensor memory) written
            if (warp == 1 || warp == 14) {
                const bool hi = warp == 1;
                const uint32_t d = tbase + (hi ? C::T_S : C::T_S2), tq = tbase + C::T_Q;
                const uint64_t a0 = tc_desc(smem_u32(qhi), 128, D * 16);
                for (int c = 0; c < NC && ok; ++c) {
                    const int kb = c & 1;
                    if (!mbar_wait(k_ready + kb, (c >> 1) & 1, limit) || (c >= 1 && !mbar_wait(s_free, (c - 1) & 1, limit))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors built once; a 16-dim step moves the start address by 256
                    // bytes, i.e. 16 in the descriptor's address field
                    const uint64_t b0 = tc_desc(smem_u32(khat(kb, 0)), 128, D * 16);
                    if (hi) {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) tc_mma_ss(d, a0 + 16 * ks, b0 + 16 * ks, IDESC_S2, ks > 0 ? 1 : 0);
                        tc_commit(s_done + kb);
                    } else {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) tc_mma_ts(d, tq + ks * 8, b0 + 16 * ks, IDESC_S, ks > 0 ? 1 : 0);
                        tc_commit(s_done_b + kb);
                    }
                }
            } else {
                const uint64_t vh0 = tc_desc(smem_u32(vhat(0)), 128, NK * 16);
                const uint64_t vl0 = tc_desc(smem_u32(vhat(C::V_LO ? 1 : 0)), 128, NK * 16);
                for (int c = 0; c < NC && ok; ++c) {
                    if (!mbar_wait(p_ready, c & 1, limit) || !mbar_wait(v_ready, c & 1, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < NK / 16; ++kk) {
                        const uint32_t ph = tbase + C::T_P + kk * 8, pl = ph + NK / 2;
                        tc_mma_ts(tbase + C::T_O, ph, vh0 + 16 * kk, IDESC_O, (c > 0 || kk > 0) ? 1 : 0);
                        if constexpr (C::V_LO) tc_mma_ts(tbase + C::T_O, ph, vl0 + 16 * kk, IDESC_O, 1);
                        tc_mma_ts(tbase + C::T_O, pl, vh0 + 16 * kk, IDESC_O, 1);
                    }
                    tc_commit(pv_done);
                }
            }
            if (!ok) {
                atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
                s_timeout = 1;
            }
            // every MMA issued has completed before the tensor memory is read or released
            tc_commit(drain);
            (void)mbar_wait(drain, 0);
        }
        __syncwarp();
    } else if (warp >= 6) {  // warps 6 .. 13
        // ---------------- converters: codes -> K^, V^ ----------------
        // Order K^(0), K^(1), V^(0), K^(2), V^(1), ...: K^(c + 1) is ready while the softmax
        // of chunk c runs, and V^(c) (one buffer) waits only for O += P(c - 1) V^(c - 1).
        // Each lane takes one 16-byte group of a tile slice (4 code words), so the loads are
        // contiguous and the K^ stores of a warp fill whole core matrices.  Packed f16
        // arithmetic: a code becomes an exact f16 integer by the magic-number route (bits |
        // 0x6400 is 1024 + bits), then hi = c * d rounded (one f16 product) and lo = fma(c,
        // d, -hi), the exact residual rounded once, with d the block's f16 scale times 2^-e.
        const int ct = threadIdx.x - 6 * 32;  // 0 .. NTH - 1
        const int cw = ct >> 5;               // converter warp
        constexpr int NTH = C::CONV_THREADS, NCW = NTH / 32;
        const uint32_t magic = 0x64006400u;
        const __half2 k1024 = __float2half2_rn(1024.0f), k1032 = __float2half2_rn(1032.0f);
        const __half2 k16th = __float2half2_rn(0.0625f), km72 = __float2half2_rn(-72.0f);
        auto q8pair = [&](uint32_t word, uint32_t sel_mag, uint32_t sel_sign) {  // two sign-magnitude bytes
            const uint32_t m = (prmt_sel(word, sel_mag) & 0x007f007fu) | magic;
            const uint32_t sg = prmt_sel(word, sel_sign) & 0x80008000u;
            return u32_as_h2(h2_as_u32(__hsub2(u32_as_h2(m), k1024)) | sg);
        };
        auto q4lo = [&](uint32_t x) { return __hsub2(u32_as_h2((x & 0x000f000fu) | magic), k1032); };
        auto q4hi = [&](uint32_t x) { return __hfma2(u32_as_h2((x & 0x00f000f0u) | magic), k16th, km72); };
        auto stage_of = [&](int c) { return smem + (c % C::STAGES) * C::STAGE; };
        auto nvalid_of = [&](int c) { return max(0, min(NK, key_end - (t_begin + 2 * c) * kTileRows)); };
        auto half_of = [](uint32_t w, int upper) { return upper ? (w >> 16) : (w & 0xffffu); };

        auto convert_k = [&](int c) {
            const int slot = c % C::STAGES, use = c / C::STAGES, kb = c & 1;
            const uint8_t *st = stage_of(c);
            const uint8_t *kcs = st, *kss = st + 2 * (C::KC + C::VC), *vss = kss + 2 * C::KS;
            const int nvalid = nvalid_of(c);
            bool okc = mbar_wait(full + slot, use & 1, limit);
            if (c >= 2) {  // both S streams of chunk c - 2 have read this K^ buffer
                okc = mbar_wait(s_done + kb, ((c >> 1) - 1) & 1, limit) && okc;
                okc = mbar_wait(s_done_b + kb, ((c >> 1) - 1) & 1, limit) && okc;
            }
            // the chunk's exponents (largest scale of its valid keys), found by every converter
            // warp on its own
            constexpr float cmaxk = KT == KVQ_Q8_0 ? 127.f : 8.f, cmaxv = VT == KVQ_Q8_0 ? 127.f : 8.f;
            float mk = 0.f, mv = 0.f;
            if constexpr (KT != KVQ_F16) mk = chunk_scale_max<NS>(kss, nvalid, cmaxk);
            if constexpr (VT != KVQ_F16) mv = chunk_scale_max<NS>(vss, nvalid, cmaxv);
            const int ek = chunk_exp(cmaxk * mk), ev = chunk_exp(cmaxv * mv);
            const __half2 fk = __float2half2_rn(pow2i(-ek));
            if (ct == 0) {
                e_val[(c & 3) * 2] = ek;
                e_val[(c & 3) * 2 + 1] = ev;
            }
            uint8_t *kh = khat(kb, 0), *kl = khat(kb, C::K_LO ? 1 : 0);
            auto put_k = [&](int kc, int dim, __half2 c01, __half2 c23, __half2 d2) {
                // values (dim, dim+1) and (dim+2, dim+3) of key kc: hi and lo parts
                const __half2 h01 = __hmul2(c01, d2), h23 = __hmul2(c23, d2);
                const __half2 l01 = __hfma2(c01, d2, __hneg2(h01)), l23 = __hfma2(c23, d2, __hneg2(h23));
                const int off = kmaj(kc, dim, D);
                *reinterpret_cast<uint2 *>(kh + off) = make_uint2(h2_as_u32(h01), h2_as_u32(h23));
                *reinterpret_cast<uint2 *>(kl + off) = make_uint2(h2_as_u32(l01), h2_as_u32(l23));
            };
            const int n = lane >> 2, jd = lane & 3;  // key n (and n + 8) of the tile, 4-dim group jd
            if constexpr (KT == KVQ_Q8_0) {
                // 16-byte group (b, lane) of a slice: words q = 2 stt + hd, values 32b + 16hd + 4jd
                // .. + 3 of key n + 8 stt; the block's scales of keys (n, n + 8) in one 8-byte load
                constexpr int NWU = 2 * NS * 4;
                auto load = [&](int wu, uint4 &w, uint2 &sc) {
                    const int ts = wu >> 2, b = wu & 3;
                    w = *reinterpret_cast<const uint4 *>(kcs + ts * 2048 + (b * 32 + lane) * 16);
                    sc = *reinterpret_cast<const uint2 *>(kss + ts * kScaleTile + (n >> 1) * 32 + b * 8);
                };
                auto conv = [&](int wu, const uint4 &w, const uint2 &sc) {
                    const int ts = wu >> 2, b = wu & 3, t = ts / NS, s = ts % NS;
                    const int k0 = t * kTileRows + n, k1 = k0 + 8, dim0 = s * kSlice + 32 * b + 4 * jd;
                    const uint32_t da = k0 < nvalid ? half_of(sc.x, n & 1) : 0u;
                    const uint32_t db = k1 < nvalid ? half_of(sc.y, n & 1) : 0u;
                    const __half2 d2a = __hmul2(u32_as_h2(da | (da << 16)), fk);
                    const __half2 d2b = __hmul2(u32_as_h2(db | (db << 16)), fk);
                    put_k(k0, dim0, q8pair(w.x, 0x4140u, 0x1404u), q8pair(w.x, 0x4342u, 0x3424u), d2a);
                    put_k(k0, dim0 + 16, q8pair(w.y, 0x4140u, 0x1404u), q8pair(w.y, 0x4342u, 0x3424u), d2a);
                    put_k(k1, dim0, q8pair(w.z, 0x4140u, 0x1404u), q8pair(w.z, 0x4342u, 0x3424u), d2b);
                    put_k(k1, dim0 + 16, q8pair(w.w, 0x4140u, 0x1404u), q8pair(w.w, 0x4342u, 0x3424u), d2b);
                };
                for (int wu = cw; wu < NWU; wu += 2 * NCW) {
                    uint4 w0, w1;
                    uint2 s0, s1;
                    load(wu, w0, s0);
                    if (wu + NCW < NWU) load(wu + NCW, w1, s1);
                    conv(wu, w0, s0);
                    if (wu + NCW < NWU) conv(wu + NCW, w1, s1);
                }
            } else if constexpr (KT == KVQ_Q4_0) {
                // 16-byte group (b2, lane): words q = 2 (b - 2 b2) + stt, low nibbles values
                // 32b + 4jd .. + 3, high nibbles + 16, of key n + 8 stt; scales of blocks 2 b2, 2 b2 + 1
                constexpr int NWU = 2 * NS * 2;
                auto load = [&](int wu, uint4 &w, uint4 &sc) {
                    const int ts = wu >> 1, b2 = wu & 1;
                    w = *reinterpret_cast<const uint4 *>(kcs + ts * 1024 + (b2 * 32 + lane) * 16);
                    sc = *reinterpret_cast<const uint4 *>(kss + ts * kScaleTile + (n >> 1) * 32 + b2 * 16);
                };
                auto conv = [&](int wu, const uint4 &w, const uint4 &sc) {
                    const int ts = wu >> 1, b2 = wu & 1, t = ts / NS, s = ts % NS;
                    const int k0 = t * kTileRows + n, k1 = k0 + 8, dim0 = s * kSlice + 64 * b2 + 4 * jd;
                    const uint32_t dbits[4] = {k0 < nvalid ? half_of(sc.x, n & 1) : 0u, k1 < nvalid ? half_of(sc.y, n & 1) : 0u,
                                               k0 < nvalid ? half_of(sc.z, n & 1) : 0u, k1 < nvalid ? half_of(sc.w, n & 1) : 0u};
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int kc = (q & 1) ? k1 : k0, dim = dim0 + 32 * (q >> 1);
                        const __half2 d2 = __hmul2(u32_as_h2(dbits[q] | (dbits[q] << 16)), fk);
                        const uint32_t w01 = prmt_sel(words[q], 0x4140u), w23 = prmt_sel(words[q], 0x4342u);
                        put_k(kc, dim, q4lo(w01), q4lo(w23), d2);
                        put_k(kc, dim + 16, q4hi(w01), q4hi(w23), d2);
                    }
                };
                for (int wu = cw; wu < NWU; wu += 2 * NCW) {
                    uint4 w0, w1, s0, s1;
                    load(wu, w0, s0);
                    if (wu + NCW < NWU) load(wu + NCW, w1, s1);
                    conv(wu, w0, s0);
                    if (wu + NCW < NWU) conv(wu + NCW, w1, s1);
                }
            } else {
                // f16: 16-byte group (ch, lane), ch = 2b + stt: words (hd, odd) hold the halves
                // (v0, v2), (v1, v3) of values 32b + 16hd + 4jd .. + 3 of key n + 8 stt
                constexpr int NWU = 2 * NS * 8;
                for (int wu = cw; wu < NWU; wu += NCW) {
                    const int ts = wu >> 3, ch = wu & 7, t = ts / NS, s = ts % NS;
                    uint4 w = *reinterpret_cast<const uint4 *>(kcs + ts * 4096 + (ch * 32 + lane) * 16);
                    const int kc = t * kTileRows + n + 8 * (ch & 1), dim0 = s * kSlice + 32 * (ch >> 1) + 4 * jd;
                    if (kc >= nvalid) w = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint2 *>(kh + kmaj(kc, dim0, D)) =
                        make_uint2(prmt2_sel(w.x, w.y, 0x5410u), prmt2_sel(w.x, w.y, 0x7632u));
                    *reinterpret_cast<uint2 *>(kh + kmaj(kc, dim0 + 16, D)) =
                        make_uint2(prmt2_sel(w.z, w.w, 0x5410u), prmt2_sel(w.z, w.w, 0x7632u));
                }
            }
            fence_async_smem();
            asm volatile("bar.sync 2, %0;\n" ::"r"(NTH) : "memory");
            if (ct == 0) {
                mbar_arrive(e_ready + (c & 3));
                mbar_arrive(k_ready + kb);
            }
            return okc;
        };

        auto convert_v = [&](int c) {
            const int slot = c % C::STAGES;
            const uint8_t *st = stage_of(c);
            const uint8_t *vcs = st + 2 * C::KC, *vss = st + 2 * (C::KC + C::VC) + 2 * C::KS;
            const int nvalid = nvalid_of(c);
            // the single V^ buffer is free once O += P(c - 1) V^(c - 1) has completed
            const bool okc = c >= 1 ? mbar_wait(pv_done, (c - 1) & 1, limit) : true;
            const __half2 fv = __float2half2_rn(pow2i(-e_val[(c & 3) * 2 + 1]));
            uint8_t *vh = vhat(0), *vl = vhat(C::V_LO ? 1 : 0);
            // a V word holds one value of keys [byte 0] 2j, [1] 8 + 2j, [2] 2j + 1, [3] 9 + 2j;
            // the scales of keys (2j, 2j+1) and (8+2j, 9+2j) of block b are the two words of
            // the 8 bytes at j*32 + b*8
            auto put_v = [&](int dim, int k0, int k1, __half2 ca, __half2 cb, __half2 da, __half2 db) {
                const __half2 ha = __hmul2(ca, da), hb = __hmul2(cb, db);
                *reinterpret_cast<uint32_t *>(vh + kmaj(dim, k0, NK)) = h2_as_u32(ha);
                *reinterpret_cast<uint32_t *>(vh + kmaj(dim, k1, NK)) = h2_as_u32(hb);
                *reinterpret_cast<uint32_t *>(vl + kmaj(dim, k0, NK)) = h2_as_u32(__hfma2(ca, da, __hneg2(ha)));
                *reinterpret_cast<uint32_t *>(vl + kmaj(dim, k1, NK)) = h2_as_u32(__hfma2(cb, db, __hneg2(hb)));
            };
            // scale pair (keys k, k + 1) with keys past the valid range set to 0 (their codes may be any bits)
            auto mask_pair = [&](uint32_t sc, int k) {
                return k >= nvalid ? 0u : (k + 1 >= nvalid ? (sc & 0x0000ffffu) : sc);
            };
            const int np = lane >> 2, j = lane & 3;
            if constexpr (VT == KVQ_Q8_0) {
                // 16-byte group (b, lane): word w4 holds value 32b + 16 (w4 >> 1) + 2np + (w4 & 1)
                constexpr int NWU = 2 * NS * 4;
                auto load = [&](int wu, uint4 &w, uint2 &sc) {
                    const int ts = wu >> 2, b = wu & 3;
                    w = *reinterpret_cast<const uint4 *>(vcs + ts * 2048 + (b * 32 + lane) * 16);
                    sc = *reinterpret_cast<const uint2 *>(vss + ts * kScaleTile + j * 32 + b * 8);
                };
                auto conv = [&](int wu, const uint4 &w, const uint2 &sc) {
                    const int ts = wu >> 2, b = wu & 3, t = ts / NS, s = ts % NS;
                    const int k0 = t * kTileRows + 2 * j, k1 = k0 + 8, dim0 = s * kSlice + 32 * b + 2 * np;
                    const __half2 da = __hmul2(u32_as_h2(mask_pair(sc.x, k0)), fv);
                    const __half2 db = __hmul2(u32_as_h2(mask_pair(sc.y, k1)), fv);
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4)  // bytes (0, 2) are keys (2j, 2j+1); bytes (1, 3) keys (8+2j, 9+2j)
                        put_v(dim0 + 16 * (w4 >> 1) + (w4 & 1), k0, k1, q8pair(words[w4], 0x4240u, 0x2404u),
                              q8pair(words[w4], 0x4341u, 0x3414u), da, db);
                };
                for (int wu = cw; wu < NWU; wu += 2 * NCW) {
                    uint4 w0, w1;
                    uint2 s0, s1;
                    load(wu, w0, s0);
                    if (wu + NCW < NWU) load(wu + NCW, w1, s1);
                    conv(wu, w0, s0);
                    if (wu + NCW < NWU) conv(wu + NCW, w1, s1);
                }
            } else if constexpr (VT == KVQ_Q4_0) {
                // 16-byte group (b2, lane): word w4 holds value 2np + (w4 & 1) of block
                // 2 b2 + (w4 >> 1) in its low nibbles, and that value + 16 in its high nibbles
                constexpr int NWU = 2 * NS * 2;
                auto load = [&](int wu, uint4 &w, uint4 &sc) {
                    const int ts = wu >> 1, b2 = wu & 1;
                    w = *reinterpret_cast<const uint4 *>(vcs + ts * 1024 + (b2 * 32 + lane) * 16);
                    sc = *reinterpret_cast<const uint4 *>(vss + ts * kScaleTile + j * 32 + b2 * 16);
                };
                auto conv = [&](int wu, const uint4 &w, const uint4 &sc) {
                    const int ts = wu >> 1, b2 = wu & 1, t = ts / NS, s = ts % NS;
                    const int k0 = t * kTileRows + 2 * j, k1 = k0 + 8, dim0 = s * kSlice + 64 * b2 + 2 * np;
                    const __half2 da0 = __hmul2(u32_as_h2(mask_pair(sc.x, k0)), fv);
                    const __half2 db0 = __hmul2(u32_as_h2(mask_pair(sc.y, k1)), fv);
                    const __half2 da1 = __hmul2(u32_as_h2(mask_pair(sc.z, k0)), fv);
                    const __half2 db1 = __hmul2(u32_as_h2(mask_pair(sc.w, k1)), fv);
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const int dim = dim0 + 32 * (w4 >> 1) + (w4 & 1);
                        const __half2 da = (w4 >> 1) ? da1 : da0, db = (w4 >> 1) ? db1 : db0;
                        const uint32_t wa = prmt_sel(words[w4], 0x4240u), wb = prmt_sel(words[w4], 0x4341u);
                        put_v(dim, k0, k1, q4lo(wa), q4lo(wb), da, db);
                        put_v(dim + 16, k0, k1, q4hi(wa), q4hi(wb), da, db);
                    }
                };
                for (int wu = cw; wu < NWU; wu += 2 * NCW) {
                    uint4 w0, w1, s0, s1;
                    load(wu, w0, s0);
                    if (wu + NCW < NWU) load(wu + NCW, w1, s1);
                    conv(wu, w0, s0);
                    if (wu + NCW < NWU) conv(wu + NCW, w1, s1);
                }
            } else {
                // f16: 16-byte group (ch, lane), ch = 2b + hv: word q = 2 rodd + cd holds value
                // 32b + 16hv + 2np + rodd of keys (2j, 2j+1) (cd = 0) or (8+2j, 9+2j) (cd = 1)
                constexpr int NWU = 2 * NS * 8;
                for (int wu = cw; wu < NWU; wu += NCW) {
                    const int ts = wu >> 3, ch = wu & 7, t = ts / NS, s = ts % NS;
                    const uint4 w = *reinterpret_cast<const uint4 *>(vcs + ts * 4096 + (ch * 32 + lane) * 16);
                    const int dim = s * kSlice + 32 * (ch >> 1) + 16 * (ch & 1) + 2 * np;
                    const int k0 = t * kTileRows + 2 * j, k1 = k0 + 8;
                    *reinterpret_cast<uint32_t *>(vh + kmaj(dim, k0, NK)) = mask_pair(w.x, k0);
                    *reinterpret_cast<uint32_t *>(vh + kmaj(dim, k1, NK)) = mask_pair(w.y, k1);
                    *reinterpret_cast<uint32_t *>(vh + kmaj(dim + 1, k0, NK)) = mask_pair(w.z, k0);
                    *reinterpret_cast<uint32_t *>(vh + kmaj(dim + 1, k1, NK)) = mask_pair(w.w, k1);
                }
            }
            fence_async_smem();
            asm volatile("bar.sync 2, %0;\n" ::"r"(NTH) : "memory");
            if (ct == 0) {
                mbar_arrive(v_ready);
                mbar_arrive(empty + slot);  // the stage's codes are consumed
            }
            return okc;
        };

        // warps 6 .. 9 (lane quarters 2, 3, 0, 1) stage the second half of Q first; their
        // transpose blocks sit in K^ buffer 1 and V^, which no conversion writes before the
        // first chunk's K^ is complete (every converter passes its closing barrier)
        if (cw < 4) stage_q(warp & 3, D / 2, D, smem + C::OFF_K + (C::K_LO ? 2 : 1) * C::KHAT + cw * 32 * C::QT_ROW);
        bool ok = true;
        if (NC > 0) ok = convert_k(0);
        for (int c = 0; c < NC; ++c) {
            if (c + 1 < NC) ok = convert_k(c + 1) && ok;
            ok = convert_v(c) && ok;
        }
        if (ct == 0 && !ok) {
            atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
            s_timeout = 1;
        }
    } else {
        // ---------------- softmax warps: one query row per thread ----------------
        const int quarter = warp & 3;          // the lanes this warp may access
        const int r = 32 * quarter + lane;     // query row = tensor-memory lane
        const uint32_t trow = tbase + (static_cast<uint32_t>(32 * quarter) << 16);
        const bool rv = r < R;
        const int qi = rv ? r / p.G : 0;       // draft query of the row
        const int lim = L - n_q + qi;          // last position the row attends to
        stage_q(quarter, 0, D / 2, smem + C::OFF_QT + quarter * 32 * C::QT_ROW);
        float m_run = -CUDART_INF_F, l_acc = 0.f;
        bool ok = true;
        for (int c = 0; c < NC; ++c) {
            const int kb = c & 1;
            bool okc = mbar_wait(s_done + kb, (c >> 1) & 1, limit);
            okc = mbar_wait(s_done_b + kb, (c >> 1) & 1, limit) && okc;
            okc = mbar_wait(e_ready + (c & 3), (c >> 2) & 1, limit) && okc;
            okc = __all_sync(0xffffffffu, okc);
            tc_fence_after();
            const int ek = e_val[(c & 3) * 2], ev = e_val[(c & 3) * 2 + 1];
            const float fk = pow2i(ek), fv = pow2i(ev);
            const int key0 = (t_begin + 2 * c) * kTileRows;
            float s[32], mx = -CUDART_INF_F;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {  // 16 keys at a time
                uint32_t a[16];  // S = Q hi K^ hi + Q lo K^ hi (S2) + Q hi K^ lo
                {
                    uint32_t a2[16];
                    tc_ld16(trow + C::T_S + 16 * h2, a);
                    tc_ld16(trow + C::T_S2 + 16 * h2, a2);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(a2[j]));
                }
                if constexpr (C::K_LO) {
                    uint32_t b[16];
                    tc_ld16(trow + C::T_S + NK + 16 * h2, b);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(b[j]));
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int key = key0 + 16 * h2 + j;
                    const bool valid = rv && key < key_end && key <= lim;
                    s[16 * h2 + j] = valid ? __uint_as_float(a[j]) * fk : -CUDART_INF_F;
                    mx = fmaxf(mx, s[16 * h2 + j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);  // the S columns may take the next chunk
            // lazy rescale: only when the row maximum grows by more than 2^6 (p * 2^e_v stays
            // below 2^15 in f16); O is rescaled in tensor memory once the previous PV is done
            const bool need = mx > m_run + 6.f;
            float alpha = 1.f;
            if (need) {
                alpha = m_run == -CUDART_INF_F ? 0.f : ex2(m_run - mx);
                m_run = mx;
                l_acc *= alpha;
            }
            const float m_use = m_run == -CUDART_INF_F ? 0.f : m_run;
            uint32_t phw[16], plw[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float p0 = ex2(s[2 * u] - m_use), p1 = ex2(s[2 * u + 1] - m_use);
                l_acc += p0 + p1;
                split_hi_lo(p0 * fv, p1 * fv, phw[u], plw[u]);
            }
            // O and the P buffer are free once O += P(c - 1) V^(c - 1) is done
            if (c >= 1) okc = mbar_wait(pv_done, (c - 1) & 1, limit) && okc;
            okc = __all_sync(0xffffffffu, okc);
            tc_fence_after();
            if (c >= 1 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
                for (int k0 = 0; k0 < D; k0 += 16) {
                    uint32_t o[16];
                    tc_ld16(trow + C::T_O + k0, o);
                    tc_wait_ld();
#pragma unroll
                    for (int u = 0; u < 16; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                    tc_st16(trow + C::T_O + k0, o);
                }
            }
            tc_st16(trow + C::T_P, phw);  // one P buffer: P(c - 1) V^ has completed
            tc_st16(trow + C::T_P + NK / 2, plw);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready);
            if (!okc) ok = false;
        }
        // epilogue: the row's split triple (o unnormalised, m natural log, l)
        if (NC > 0) ok = mbar_wait(pv_done, (NC - 1) & 1, limit) && ok;
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (!ok && lane == 0) {
            atomicOr(p.err, KVQ_DEVERR_TIMEOUT);
            s_timeout = 1;
        }
        // O leaves through shared memory: each thread writes its row (the operands are no
        // longer read: every MMA has completed), then the warp stores its 32 rows with
        // coalesced 16-byte writes, half a row per request.
        {
            uint8_t *ost = smem + static_cast<size_t>(r) * C::O_ROW;
#pragma unroll 1
            for (int k0 = 0; k0 < D; k0 += 16) {
                uint32_t o[16];
                tc_ld16(trow + C::T_O + k0, o);
                tc_wait_ld();
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4 *>(ost + (k0 + 4 * u) * 4) =
                        NC > 0 ? make_uint4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]) : make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
            const int R0 = 32 * quarter;
#pragma unroll 1
            for (int i = 0; i < 32; ++i) {
                const int row = R0 + i;
                if (row >= R) break;
                const size_t pr = (prow0 + row) * p.part_stride + p.part_base + split;
                float4 *dst = reinterpret_cast<float4 *>(p.part_o + pr * D);
                const uint8_t *srow = smem + static_cast<size_t>(row) * C::O_ROW;
#pragma unroll
                for (int c4 = lane; c4 < D / 4; c4 += 32) dst[c4] = *reinterpret_cast<const float4 *>(srow + 16 * c4);
            }
        }
        if (rv) {
            const size_t pr = (prow0 + r) * p.part_stride + p.part_base + split;
            p.part_m[pr] = m_run == -CUDART_INF_F ? -CUDART_INF_F : m_run * kLn2;
            p.part_l[pr] = l_acc;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tbase), "r"(C::TCOLS));
    // a CTA whose waits gave up published a triple that may be incomplete; the error word says so
    const size_t unit = static_cast<size_t>(bseq) * p.Hkv + h;
    split_merge(p, ns, split, R, D, prow0, unit, rmap, s_flag, smem);
}

}  // namespace
}  // namespace kvq

namespace kvq {
namespace {

template <int KT, int VT, int NS>
cudaError_t launch_verify_tc_t(const DecodeParams &p, cudaStream_t stream) {
    using C = TcCfg<KT, VT, NS>;
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(verify_tc_kernel<KT, VT, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    DecodeParams q = p;
    int sms = 0;
    e = sm_count(dev, &sms);
    if (e != cudaSuccess) return e;
    // one CTA per SM (shared memory): the grid is resident at once when it fits the SMs
    q.wide = static_cast<long long>(p.n_splits) * p.Hkv * p.B <= sms ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_splits, p.Hkv, p.B);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_tc_kernel<KT, VT, NS>, q);
}

}  // namespace

cudaError_t launch_verify_tc(int type_k, int type_v, const DecodeParams &p, cudaStream_t stream) {
    const int ns = p.D / kSlice;
#define KVQ_TC_CASE(KT_, VT_)                                                     \
    if (type_k == KT_ && type_v == VT_) {                                         \
        if (ns == 1) return launch_verify_tc_t<KT_, VT_, 1>(p, stream);           \
        if (ns == 2) return launch_verify_tc_t<KT_, VT_, 2>(p, stream);           \
    }
    KVQ_TC_CASE(KVQ_F16, KVQ_F16)
    KVQ_TC_CASE(KVQ_F16, KVQ_Q8_0)
    KVQ_TC_CASE(KVQ_F16, KVQ_Q4_0)
    KVQ_TC_CASE(KVQ_Q8_0, KVQ_F16)
    KVQ_TC_CASE(KVQ_Q8_0, KVQ_Q8_0)
    KVQ_TC_CASE(KVQ_Q8_0, KVQ_Q4_0)
    KVQ_TC_CASE(KVQ_Q4_0, KVQ_F16)
    KVQ_TC_CASE(KVQ_Q4_0, KVQ_Q8_0)
    KVQ_TC_CASE(KVQ_Q4_0, KVQ_Q4_0)
#undef KVQ_TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvq
