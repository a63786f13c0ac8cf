// tcgen05 attention kernel for long query chunks, q8_0 V.
#include "kvq_prefill.cuh"

namespace kvq {
cudaError_t launch_prefill_q8(const AttnParams &p, int n_ctas, bool dump, cudaStream_t s, bool pdl)
{
    return launch_prefill_t<KVQ_V_Q8_0>(p, n_ctas, dump, s, pdl);
}
cudaError_t prepare_prefill_q8() { return prepare_prefill_t<KVQ_V_Q8_0>(); }
}  // namespace kvq
