// Split-KV attention kernels for q4_0 V.
#include "kvq_attn.cuh"

namespace kvq {
KVQ_DEFINE_SPLIT_ENTRY(q4, KVQ_V_Q4_0)
}  // namespace kvq
