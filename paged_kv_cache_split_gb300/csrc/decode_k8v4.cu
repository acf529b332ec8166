// decode_k8v4.cu — decode-attention instantiations for the K8V4 stored format.
#include "decode.cuh"

namespace pkv {
cudaError_t launch_decode_k8v4(const DecodeArgs& a) { return launch_decode_fmt<PKV_FMT_K8V4>(a); }
}  // namespace pkv
