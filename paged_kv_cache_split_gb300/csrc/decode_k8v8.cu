// decode_k8v8.cu — decode-attention instantiations for the K8V8 stored format.
#include "decode.cuh"

namespace pkv {
cudaError_t launch_decode_k8v8(const DecodeArgs& a) { return launch_decode_fmt<PKV_FMT_K8V8>(a); }
}  // namespace pkv
