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
