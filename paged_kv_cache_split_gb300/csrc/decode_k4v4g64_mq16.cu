// decode_k4v4g64_mq16.cu — chunked-prefill attention for K4V4 with groups of 64: several queries of one sequence
// per tensor-core tile (16 rows of (query, head) pairs).
#include "decode_packed_mma.cuh"

namespace pkv {
cudaError_t launch_decode_k4v4_g64_mq16(const DecodeArgs& a) { return launch_decode_packed_mma_mq<PKV_FMT_K4V4, kGroupWide, true>(a); }
}  // namespace pkv
