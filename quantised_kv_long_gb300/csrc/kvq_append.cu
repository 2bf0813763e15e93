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

// round half away from zero, written from the definition (|y - trunc(y)| is exact in fp32)
__device__ __forceinline__ float round_half_away(float y) {
    float t = truncf(y);
    float r = y - t;
    if (fabsf(r) >= 0.5f) t += copysignf(1.0f, y);
    return t;
}

template <int T, bool IS_V>
__device__ __forceinline__ void quantize_store(const float *x, uint8_t *codes, uint8_t *scales, int kt, int lane) {
    const float4 v4 = *reinterpret_cast<const float4 *>(x);
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
        for (int e = 0; e < 4; ++e) c[e] = static_cast<int>(round_half_away(__fmul_rn(xs[e], id)));
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

    if constexpr (T == KVQ_Q4_0) {
        // value of largest magnitude; the lowest index wins a tie
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
        const float d = __fdiv_rn(best, -8.0f);
        const float id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
        int c[4], chi[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = static_cast<int>(__fadd_rn(__fmul_rn(xs[e], id), 8.5f));  // truncation
            c[e] = t < 15 ? t : 15;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) chi[e] = __shfl_down_sync(0xffffffffu, c[e], 4);
        if ((lane & 7) < 4) {
            // this lane holds values i0..i0+3 (< 16) and, from lane+4, values i0+16..i0+19
            uint32_t byte[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) byte[e] = uint32_t(c[e]) | (uint32_t(chi[e]) << 4);
            if constexpr (!IS_V) {
                const int jb = lane & 7;  // bytes 4jb..4jb+3 of the block
                const uint32_t w = byte[0] | (byte[1] << 8) | (byte[2] << 16) | (byte[3] << 24);
                *reinterpret_cast<uint32_t *>(codes + (b >> 1) * 512 + (4 * n + jb) * 16 + (2 * (b & 1) + st) * 4) =
                    w;
            } else {
                const int vb = vword_byte(pos);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = i0 + e, n2 = r >> 1, qq = r & 1;
                    codes[(b >> 1) * 512 + (4 * n2 + j) * 16 + (2 * (b & 1) + qq) * 4 + vb] =
                        static_cast<uint8_t>(byte[e]);
                }
            }
        }
        if ((lane & 7) == 0)
            *reinterpret_cast<__half *>(scales + j * 32 + b * 8 + pos * 2) = __float2half_rn(d);
        return;
    }
}

template <int KT, int VT>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
    __shared__ int s_last;
    const int lane = threadIdx.x & 31;
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int NS = p.D / kSlice;
    if (warp_global < p.total_warps) {
        const int sl = warp_global % NS;
        int rest = warp_global / NS;
        const int row = rest % p.n_new;
        rest /= p.n_new;
        const int h = rest % p.Hkv;
        const int bl = rest / p.Hkv;
        const int bseq = p.b0 + bl;
        const int L = __ldcg(p.len + bseq);
        if (L >= 0 && L + p.n_new <= p.cap) {
            const int pos = L + row;
            const size_t tile = (static_cast<size_t>(bseq) * p.Hkv + h) * p.cap_tiles + (pos >> 4);
            const int kt = pos & 15;
            const size_t src = ((static_cast<size_t>(bl) * p.Hkv + h) * p.n_new + row) * p.D + sl * kSlice + 4 * lane;
            quantize_store<KT, false>(p.k + src, p.k_codes + (tile * NS + sl) * code_tile_bytes(KT),
                                      p.k_scales + (tile * NS + sl) * kScaleTile, kt, lane);
            quantize_store<VT, true>(p.v + src, p.v_codes + (tile * NS + sl) * code_tile_bytes(VT),
                                     p.v_scales + (tile * NS + sl) * kScaleTile, kt, lane);
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
    const int warps_per_block = 8;
    const int blocks = (p.total_warps + warps_per_block - 1) / warps_per_block;
    append_kernel<KT, VT><<<blocks, 32 * warps_per_block, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

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
#undef KVQ_APPEND_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kvq
