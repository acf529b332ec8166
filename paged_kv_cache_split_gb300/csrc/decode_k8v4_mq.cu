// decode_k8v4_mq.cu — chunked-prefill attention for K8V4: several queries of one sequence
// per tensor-core tile (8 rows of (query, head) pairs).
#include "decode_packed_mma.cuh"

namespace pkv {
cudaError_t launch_decode_k8v4_mq(const DecodeArgs& a) { return launch_decode_packed_mma_mq<PKV_FMT_K8V4, kGroup, false>(a); }
}  // namespace pkv
