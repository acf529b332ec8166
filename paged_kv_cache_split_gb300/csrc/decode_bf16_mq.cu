// decode_bf16_mq.cu — bf16 attention with several queries of one sequence per tile
// (chunked prefill): the S tile's rows are (query, head) pairs, nq x heads per kv
// head <= 16 (8 at head_dim 256).
#include "decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_bf16_mq(const DecodeArgs& a) {
  const int G = a.G / a.nq;  // query heads per kv head
#define PKV_CASE(DD, GG, NN) \
  if (a.D == DD && G == GG && a.nq == NN) return launch_decode_bf16_mma_t<DD, GG, NN>(a);
  PKV_CASE(64, 1, 2) PKV_CASE(64, 1, 4) PKV_CASE(64, 1, 8) PKV_CASE(64, 2, 2) PKV_CASE(64, 2, 4) PKV_CASE(64, 4, 2)
  PKV_CASE(128, 1, 2) PKV_CASE(128, 1, 4) PKV_CASE(128, 1, 8) PKV_CASE(128, 2, 2) PKV_CASE(128, 2, 4)
  PKV_CASE(128, 4, 2)
  PKV_CASE(256, 1, 2) PKV_CASE(256, 1, 4) PKV_CASE(256, 1, 8) PKV_CASE(256, 2, 2) PKV_CASE(256, 2, 4)
  PKV_CASE(256, 4, 2)
  // 16 rows (head_dim <= 128)
  PKV_CASE(64, 1, 16) PKV_CASE(64, 2, 8) PKV_CASE(64, 4, 4) PKV_CASE(64, 8, 2)
  PKV_CASE(128, 1, 16) PKV_CASE(128, 2, 8) PKV_CASE(128, 4, 4) PKV_CASE(128, 8, 2)
#undef PKV_CASE
  return cudaErrorInvalidValue;
}
}  // namespace pkv
