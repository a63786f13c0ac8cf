// Split-KV attention kernels for q8_0 V.
#include "kvq_attn.cuh"

namespace kvq {
KVQ_DEFINE_SPLIT_ENTRY(q8, KVQ_V_Q8_0)
}  // namespace kvq
