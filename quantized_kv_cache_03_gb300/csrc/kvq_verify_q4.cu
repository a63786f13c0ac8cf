// tcgen05 attention kernel for 9..32 query rows per kv head, q4_0 V.
#include "kvq_verify.cuh"

namespace kvq {
cudaError_t launch_verify_q4(const AttnParams &p, int n_ctas, cudaStream_t s, bool pdl)
{
    return launch_verify_t<KVQ_V_Q4_0>(p, n_ctas, s, pdl);
}
cudaError_t prepare_verify_q4() { return prepare_verify_t<KVQ_V_Q4_0>(); }
}  // namespace kvq
