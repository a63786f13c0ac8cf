// tcgen05 attention kernel for 9..32 query rows per kv head, q8_0 V.
#include "kvq_verify.cuh"

namespace kvq {
cudaError_t launch_verify_q8(const AttnParams &p, int n_ctas, cudaStream_t s, bool pdl)
{
    return launch_verify_t<KVQ_V_Q8_0>(p, n_ctas, s, pdl);
}
cudaError_t prepare_verify_q8() { return prepare_verify_t<KVQ_V_Q8_0>(); }
}  // namespace kvq
