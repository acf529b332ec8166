// decode_k4v4g64.cu — decode attention for K4V4 with groups of 64 values (one FP32
// scale/offset pair per 64 dims: five bits per value), head_dim 128 or 256.
#include "decode_packed_mma.cuh"

namespace pkv {
cudaError_t launch_decode_k4v4_g64(const DecodeArgs& a) { return launch_decode_packed_mma<PKV_FMT_K4V4, kGroupWide>(a); }
}  // namespace pkv
