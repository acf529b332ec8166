// pkv_internal.cuh — definitions shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "pkv.h"

namespace pkv {

// Device error word bits (documented in pkv.h, pkv_pool_check_errors).
enum : int32_t {
  ERR_ROW = 1,       // block-table or write row outside the pool
  ERR_CTX = 2,       // context length negative or beyond max_blocks * block_size
  ERR_SLOT = 4,      // write slot outside [0, block_size)
  ERR_TIMEOUT = 8,   // a bounded wait gave up
};

constexpr int kBlockTokens = 32;  // tokens per block (block_size)
constexpr int kGroup = 32;        // values per affine group (default)
constexpr int kGroupWide = 64;    // K4/V4 only, D >= 128: one (scale, offset) pair per 64 values

struct FormatBits {
  int k, v;  // bits per stored K / V value (16 = bf16)
};

inline FormatBits format_bits(int fmt) {
  switch (fmt) {
    case PKV_FMT_BF16: return {16, 16};
    case PKV_FMT_K4V4: return {4, 4};
    case PKV_FMT_K8V4: return {8, 4};
    case PKV_FMT_K8V8: return {8, 8};
    default: return {0, 0};
  }
}

// Slab pointer table view for one layer: entry (slab, kind) lives at
// base[slab * stride + kind], with base = table + layer * n_kinds and
// stride = n_layers * n_kinds.
struct SlabTable {
  uint8_t* const* base;
  int stride;
};

// Everything a kernel needs to address one layer of a pool.
struct LayerView {
  SlabTable tab;
  int n_kinds;
  int hkv;
  int slab_blocks;
  int64_t rows_capacity;  // rows valid at enqueue time (n_slabs * slab_blocks)
  int row_bytes[4];       // per (token, head) row, per kind
  int32_t* err;           // device error word
  // Packed formats: TMA tensor maps.  The map of (slab, this layer, kind) lives at
  // (slab's kind-0 pointer of this layer) + map_delta + kind * 128.
  int64_t map_delta;
  int box_bytes[4];       // inner box width (bytes) per kind: 128, 64, 32 or 16
};

// Bytes of one stage of the packed decode kernel: four 1024-byte-aligned regions
// of T rows (K codes, V codes, K meta, V meta; all kv heads) and q of one sequence.
inline int packed_stage_bytes(int T, int krow, int vrow, int mrow, int qbytes) {
  auto a = [](int x) { return (x + 1023) & ~1023; };
  return a(T * krow) + a(T * vrow) + 2 * a(T * mrow) + a(qbytes);
}

// Inner box width for a row of `row_bytes` (all kv heads of one token): the
// largest of 128/64/32/16 bytes that divides it (its swizzle span).
inline int tma_box_bytes(int64_t row_bytes) {
  for (int w = 128; w >= 16; w >>= 1)
    if (row_bytes % w == 0) return w;
  return 0;
}

// ---------------------------------------------------------------------------
// Inline PTX helpers (sm_90+ mbarrier and bulk-copy forms, used on sm_103a).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete, giving up after ~1 s of wall
// time: then the error word gets ERR_TIMEOUT and false is returned.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) {
      atomicOr(err, ERR_TIMEOUT);
      return false;
    }
  }
}

// One-dimensional bulk copy global -> shared, completing on `bar` (tx bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same copy with an L2 cache policy (e.g. evict-first for data read once).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D tensor (TMA) copy of one box into shared memory, completing on `bar`, with an
// L2 cache policy.  `tmap` is the global address of a CUtensorMap; x (innermost,
// bytes for a uint8 map) must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Make a tensor map written outside this kernel visible to the tensor-map proxy.
// 3-D tiled copy: box origin (x, y, z) of the tensor map, complete_tx on bar.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tensormap_acquire(const void* tmap) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(tmap) : "memory");
}

// L2 policy: lines fetched under it are the first candidates for eviction.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy: lines fetched under it are kept like ordinary loads.
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// bf16 pair (one 32-bit word) -> two floats, exactly.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

}  // namespace pkv

// Launchers implemented in the kernel translation units (host side).
namespace pkv {

struct DecodeArgs {
  LayerView lv;
  int fmt, D, G, B, Hq, max_blocks;
  const uint16_t* q;
  const int32_t* bt;
  const int32_t* ctx;
  float scale_log2;     // scale * log2(e)
  float inv_sqrt_d;     // 1/sqrt(D) as float (packed q rotation)
  const float* signs;   // [D] +-1 (packed)
  uint16_t* out;
  int32_t* counters;    // [B]
  float* partials;      // [(grid + B) * Hq * (D + 2)]
  int grid;
  int tokens_per_stage;
  int n_stages;
  size_t smem_bytes;
  cudaStream_t stream;
  int dim_split;        // see DecodePlan
  int group;            // values per affine group of the packed formats: 32 or 64 (K4/V4)
  int kv_reuse;         // 1: K/V blocks are read again soon (chunked prefill): keep them in L2
  int seg_cost;         // cost of a sequence start for the CTA split, in quarter units (Split)
  int nq;               // queries per (virtual) sequence: 1 for decode; > 1 for chunked prefill,
                        // where Hq and G count the nq queries' heads (G = nq x heads per kv head)
};

// Returns cudaSuccess or the launch error.  Defined per format in decode_*.cu.
cudaError_t launch_decode_bf16(const DecodeArgs& a);
cudaError_t launch_decode_bf16_mq(const DecodeArgs& a);  // nq > 1 (decode_bf16_mq.cu)
cudaError_t launch_decode_k4v4(const DecodeArgs& a);
cudaError_t launch_decode_k4v4_g64(const DecodeArgs& a);  // groups of 64 (decode_k4v4g64.cu)
// nq > 1 (chunked prefill), per format: 8 tile rows in decode_*_mq.cu, 16 in
// decode_*_mq16.cu
cudaError_t launch_decode_k4v4_mq(const DecodeArgs& a);
cudaError_t launch_decode_k4v4_g64_mq(const DecodeArgs& a);
cudaError_t launch_decode_k8v4_mq(const DecodeArgs& a);
cudaError_t launch_decode_k8v8_mq(const DecodeArgs& a);
cudaError_t launch_decode_k4v4_mq16(const DecodeArgs& a);
cudaError_t launch_decode_k4v4_g64_mq16(const DecodeArgs& a);
cudaError_t launch_decode_k8v4_mq16(const DecodeArgs& a);
cudaError_t launch_decode_k8v8_mq16(const DecodeArgs& a);
cudaError_t launch_decode_k8v4(const DecodeArgs& a);
cudaError_t launch_decode_k8v8(const DecodeArgs& a);

// Stage-size planning shared by the launcher and the workspace query.
struct DecodePlan {
  int tokens_per_stage;
  int n_stages;
  size_t stage_bytes;
  size_t smem_bytes;
  int threads;
  int dim_split;  // packed D = 256, at most 4 kv heads, 128-byte rows: two warps per kv head
};
bool plan_decode(int fmt, int D, int G, int hkv, int B, int group, DecodePlan* plan);

cudaError_t launch_write(const LayerView& lv, int fmt, int D, int group, int n, const int32_t* rows,
                         const int32_t* slots, const uint16_t* k, const uint16_t* v,
                         const float* signs, double inv_sqrt_d, cudaStream_t s);
cudaError_t launch_copy_blocks(const uint8_t* const* table, int n_layers, int n_kinds,
                               const int64_t* block_bytes, int slab_blocks, int64_t rows_capacity,
                               int n, const int32_t* src, const int32_t* dst, int32_t* err,
                               cudaStream_t s);
cudaError_t launch_gather(const LayerView& lv, const int32_t* bt_row, int ctx, uint8_t* const* outs,
                          cudaStream_t s);

// Message returned by pkv_last_error() on this thread.
void set_last_error(const char* msg);

}  // namespace pkv
