// decode_bf16.cu — decode attention for the native bf16 format (tensor-core tiles).
#include "decode_mma.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeArgs& a) { return launch_decode_bf16_mma(a); }
}  // namespace pkv
