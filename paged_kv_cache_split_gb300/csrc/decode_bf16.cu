// decode_bf16.cu — decode attention for the native bf16 format (tensor-core tiles).
#include "decode_mma.cuh"

namespace pkv {
static cudaError_t launch_decode_bf16_mma(const DecodeArgs& a) {
#define PKV_CASE(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_decode_bf16_mma_t<DD, GG>(a);
  PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
  PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_bf16(const DecodeArgs& a) {
  if (a.nq > 1) return launch_decode_bf16_mq(a);
  return launch_decode_bf16_mma(a);
}
}  // namespace pkv
