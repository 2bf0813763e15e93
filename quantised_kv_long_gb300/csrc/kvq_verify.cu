// kvq_verify.cu -- draft-verify launches of the decode kernel (kvq_decode_kernel.cuh):
// up to 16 queries per sequence, query i attending causally to positions
// [0, len - n_q + i] ("HAL #582 -- per-layer KV compression study", section 5 P0: the
// scalar-quant MMA reader is gated to Q->ne[1] <= 16, i.e. decode and draft verify).
#include "kvq_decode_kernel.cuh"

namespace kvq {

cudaError_t launch_verify(int type_k, int type_v, const DecodeParams &p, cudaStream_t stream) {
    const int ns = p.D / kSlice;
    KVQ_DISPATCH_ALL(launch_decode_t, true, (p, true, stream))
    return cudaErrorInvalidValue;
}

cudaError_t verify_occupancy(int type_k, int type_v, int D, int *ctas_per_sm) {
    const int ns = D / kSlice;
    KVQ_DISPATCH_ALL(occupancy_t, true, (ctas_per_sm))
    return cudaErrorInvalidValue;
}

}  // namespace kvq
