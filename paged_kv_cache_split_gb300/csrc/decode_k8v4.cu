// decode_k8v4.cu — decode attention for the K8V4 packed format (tensor-core tiles).
#include "decode_packed_mma.cuh"

namespace pkv {
cudaError_t launch_decode_k8v4(const DecodeArgs& a) {
  if (a.nq > 1) return a.G > 8 ? launch_decode_k8v4_mq16(a) : launch_decode_k8v4_mq(a);
  return launch_decode_packed_mma<PKV_FMT_K8V4>(a);
}
}  // namespace pkv
