// kvq_window_dual.cu -- one decode launch over an f16 window and a quantised tail of the
// same sequences (dual_kernel in kvq_decode_kernel.cuh): the window's splits and the
// tail's splits publish their split triples into one set and are merged exactly as one
// ("HAL #582 -- per-layer KV compression study", section 5 P2 read path: the softmax
// partials of the two regions combine without loss).  256-wide heads here; 128-wide heads in
// kvq_window_dual1.cu (the window body there runs with the tail's tile-warp count, so
// that both regions share one block size).
#include "kvq_decode_kernel.cuh"

namespace kvq {

cudaError_t launch_window_dual(int tail_k, int tail_v, int D, const DecodeParams &pw, const DecodeParams &pt, int nw,
                               cudaStream_t stream) {
    if (D == kSlice) return launch_window_dual_ns1(tail_k, tail_v, pw, pt, nw, stream);
    if (D != 2 * kSlice) return cudaErrorNotSupported;
#define KVQ_DUAL_CASE(KT, VT) \
    if (tail_k == KT && tail_v == VT) return launch_dual_t<KT, VT, 2>(pw, pt, nw, stream);
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
