// decode_k4v4.cu — decode attention for the K4V4 packed format (tensor-core tiles).
#include "decode_packed_mma.cuh"

namespace pkv {
cudaError_t launch_decode_k4v4(const DecodeArgs& a) {
  if (a.nq > 1 && a.G > 8)
    return a.group == kGroupWide ? launch_decode_k4v4_g64_mq16(a) : launch_decode_k4v4_mq16(a);
  if (a.nq > 1) return a.group == kGroupWide ? launch_decode_k4v4_g64_mq(a) : launch_decode_k4v4_mq(a);
  if (a.group == kGroupWide) return launch_decode_k4v4_g64(a);
  return launch_decode_packed_mma<PKV_FMT_K4V4>(a);
}
}  // namespace pkv
