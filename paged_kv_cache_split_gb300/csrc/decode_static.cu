// decode_static.cu — decode attention for callers that cannot allocate device
// memory.
//
// pkv_paged_decode_attention needs a caller-provided workspace (split-K partials
// and per-sequence arrival counters).  Some callers have no way to obtain one: a
// serving loop that reserved all of its device memory when it started and may not
// allocate (or risk running out of memory) in the middle of a decode step, or a
// plugin hosted by a framework that owns the device allocator and does not lend it
// out.  For them this file keeps the workspace in a fixed array in device memory
// that is part of the library image: every GPU that loads the library holds
// PKV_STATIC_SCRATCH_BYTES of it until the process exits, and no call here
// allocates or frees anything.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "pkv_internal.cuh"

// The scratch array.  Host code must not use this name as a device address (on the
// host it names a stand-in object); the device address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (the first call on a device does this).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attention_noalloc(pkv_pool* pool, int layer, int B, int Hq,
                                                         const void* q_bf16_dev, const int32_t* block_table_dev,
                                                         int max_blocks, const int32_t* ctx_lens_dev, int max_ctx,
                                                         float scale, void* out_bf16_dev, void* stream) {
  if (!pool) return PKV_ERR_INVALID;
  size_t need = 0;
  pkv_status st = pkv_decode_workspace_bytes(pool, B, Hq, max_ctx, &need);
  if (st != PKV_OK) return st;
  if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "pkv_paged_decode_attention_noalloc: B=%d, Hq=%d needs %zu bytes of scratch; the fixed array holds %zu",
             B, Hq, need, (size_t)PKV_STATIC_SCRATCH_BYTES);
    pkv::set_last_error(msg);
    return PKV_ERR_RANGE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    pkv::set_last_error(cudaGetErrorString(e));
    return PKV_ERR_CUDA;
  }
  // The array keeps whatever the previous call left; the arrival counters at its
  // front must start at zero, so clear them on the caller's stream.
  if (B > 0) {
    e = cudaMemsetAsync(scratch, 0, (size_t)B * sizeof(int32_t), (cudaStream_t)stream);
    if (e != cudaSuccess) {
      pkv::set_last_error(cudaGetErrorString(e));
      return PKV_ERR_CUDA;
    }
  }
  return pkv_paged_decode_attention(pool, layer, B, Hq, q_bf16_dev, block_table_dev, max_blocks, ctx_lens_dev,
                                    max_ctx, scale, out_bf16_dev, scratch, (size_t)PKV_STATIC_SCRATCH_BYTES, stream);
}
