// kvq_window_dual1.cu -- the one-launch window + tail decode (dual_kernel in
// kvq_decode_kernel.cuh) for 128-wide heads: the f16 window's splits run with the tail's
// tile-warp count, so that both regions share one block size; all split triples of both
// regions are merged as one set ("HAL #582 -- per-layer KV compression study", section 5
// P2 read path).
#include "kvq_decode_kernel.cuh"

namespace kvq {

cudaError_t launch_window_dual_ns1(int tail_k, int tail_v, const DecodeParams &pw, const DecodeParams &pt, int nw,
                                   cudaStream_t stream) {
#define KVQ_DUAL_CASE(KT, VT) \
    if (tail_k == KT && tail_v == VT) return launch_dual_t<KT, VT, 1>(pw, pt, nw, stream);
    KVQ_DUAL_CASE(KVQ_F16, KVQ_F16)
    KVQ_DUAL_CASE(KVQ_F16, KVQ_Q8_0)
    KVQ_DUAL_CASE(KVQ_F16, KVQ_Q4_0)
    KVQ_DUAL_CASE(KVQ_Q8_0, KVQ_F16)
    KVQ_DUAL_CASE(KVQ_Q8_0, KVQ_Q8_0)
    KVQ_DUAL_CASE(KVQ_Q8_0, KVQ_Q4_0)
    KVQ_DUAL_CASE(KVQ_Q4_0, KVQ_F16)
    KVQ_DUAL_CASE(KVQ_Q4_0, KVQ_Q8_0)
    KVQ_DUAL_CASE(KVQ_Q4_0, KVQ_Q4_0)
#undef KVQ_DUAL_CASE
    return cudaErrorNotSupported;
}

}  // namespace kvq
