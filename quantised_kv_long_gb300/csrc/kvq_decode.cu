// kvq_decode.cu -- single-token decode launches (kvq_decode_kernel.cuh, one query per
// sequence), the occupancy query behind the automatic split count, and the public merge
// of split triples.
#include "kvq_decode_kernel.cuh"

namespace kvq {
namespace {

// ---------------- public merge of split triples ----------------
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
    extern __shared__ float wsm[];  // [S]
    __shared__ float s_M, s_L;
    const int r = blockIdx.x;
    const float *pm = p.part_m + static_cast<size_t>(r) * p.S;
    const float *pl = p.part_l + static_cast<size_t>(r) * p.S;
    if (threadIdx.x < 32) {
        float M = -CUDART_INF_F;
        for (int s = threadIdx.x; s < p.S; s += 32) M = fmaxf(M, pm[s]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float Ls = 0.f;
        for (int s = threadIdx.x; s < p.S; s += 32) {
            const float w = (M == -CUDART_INF_F || pm[s] == -CUDART_INF_F) ? 0.f : expf(pm[s] - M);
            wsm[s] = w;
            Ls = fmaf(w, pl[s], Ls);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
        if (threadIdx.x == 0) {
            s_M = M;
            s_L = Ls;
        }
    }
    __syncthreads();
    const float inv = s_L > 0.f ? 1.f / s_L : 0.f;
    for (int dq = threadIdx.x; dq < p.D / 4; dq += blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < p.S; ++s) {
            const float w = wsm[s];
            if (w == 0.f) continue;
            const float4 v = reinterpret_cast<const float4 *>(p.part_o + (static_cast<size_t>(r) * p.S + s) * p.D)[dq];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        reinterpret_cast<float4 *>(p.out + static_cast<size_t>(r) * p.D)[dq] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (threadIdx.x == 0 && p.lse) p.lse[r] = s_L > 0.f ? s_M + logf(s_L) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_decode(int type_k, int type_v, const DecodeParams &p, bool fused, cudaStream_t stream) {
    const int ns = p.D / kSlice;
    KVQ_DISPATCH_ALL(launch_decode_t, false, (p, fused, stream))
    return launch_decode_ext(type_k, type_v, p, fused, stream);
}

cudaError_t decode_occupancy(int type_k, int type_v, int D, int *ctas_per_sm, int *n_sms) {
    static int sm_cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (sm_cache[dev] == 0) {
        e = cudaDeviceGetAttribute(&sm_cache[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *n_sms = sm_cache[dev];
    const int ns = D / kSlice;
    KVQ_DISPATCH_ALL(occupancy_t, false, (ctas_per_sm))
    return occupancy_ext(type_k, type_v, D, ctas_per_sm);
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(p.S) * sizeof(float);
    combine_kernel<<<p.rows, 128, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kvq
