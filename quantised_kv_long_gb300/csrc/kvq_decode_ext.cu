// kvq_decode_ext.cu -- decode launches of the further scalar types (q4_1, q5_0, q5_1) in
// the pairs of "HAL #582 -- per-layer KV compression study", section 5 P0 note (q8K/q5V,
// q5/q5, q5_1/q5_1, q4_1/q4_1) and the P1 ladder floor (q5_1 K / q4_0 V).  Kept in their
// own translation unit so that the library builds in parallel.
#include "kvq_decode_kernel.cuh"

namespace kvq {

#define KVQ_DISPATCH_EXT(CALL, ARGS)                      \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q5_0, 1, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_0, KVQ_Q5_0, 1, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_1, KVQ_Q5_1, 1, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q4_1, KVQ_Q4_1, 1, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_1, KVQ_Q4_0, 1, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q8_0, KVQ_Q5_0, 2, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_0, KVQ_Q5_0, 2, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_1, KVQ_Q5_1, 2, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q4_1, KVQ_Q4_1, 2, CALL, false) ARGS; \
    KVQ_DISPATCH(KVQ_Q5_1, KVQ_Q4_0, 2, CALL, false) ARGS;

cudaError_t launch_decode_ext(int type_k, int type_v, const DecodeParams &p, bool fused, cudaStream_t stream) {
    const int ns = p.D / kSlice;
    KVQ_DISPATCH_EXT(launch_decode_t, (p, fused, stream))
    return cudaErrorInvalidValue;
}

cudaError_t occupancy_ext(int type_k, int type_v, int D, int *ctas_per_sm) {
    const int ns = D / kSlice;
    KVQ_DISPATCH_EXT(occupancy_t, (ctas_per_sm))
    return cudaErrorInvalidValue;
}

}  // namespace kvq
