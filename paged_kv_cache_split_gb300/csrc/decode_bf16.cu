// decode_bf16.cu — decode-attention instantiations for the BF16 stored format.
#include "decode.cuh"

namespace pkv {
cudaError_t launch_decode_bf16(const DecodeArgs& a) { return launch_decode_fmt<PKV_FMT_BF16>(a); }
}  // namespace pkv
