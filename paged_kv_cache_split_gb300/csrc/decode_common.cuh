// decode_common.cuh — pieces shared by the decode-attention kernels: launch
// parameters, the per-CTA unit prefix over sequences, and the split-K epilogue
// (arrival ticket and in-order merge of partials by the last CTA of a sequence).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pkv_internal.cuh"

namespace pkv {

struct DecodeParams {
  LayerView lv;
  int B, Hq, max_blocks;
  const uint16_t* q;
  const int32_t* bt;
  const int32_t* ctx;
  float scale_log2;
  float inv_sqrt_d;
  const float* signs;
  uint16_t* out;
  int32_t* counters;
  float* partials;
  int T;            // tokens per unit / stage
  int NS;           // stages in the ring
  int stage_bytes;  // bytes of one stage
};

constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;

__device__ __forceinline__ uint16_t f2bf(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Unit u -> sequence: the largest b with UP[b] <= u (then UP[b+1] > u).
__device__ __forceinline__ int find_seq(const int32_t* UP, int B, int32_t u) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (UP[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Prologue of every decode kernel: thread 0 initialises the stage barriers (full:
// one producer arrival plus the copied bytes; empty: one arrival per consumer
// warp) and warp 0 builds the unit prefix UP[0..B] over sequences (unit = T tokens
// of one sequence) and LS[b], the context length clamped to the block table.  The
// caller runs __syncthreads() afterwards.
__device__ __forceinline__ void decode_prologue(const DecodeParams& P, uint64_t* full, uint64_t* empty, int NC,
                                                int32_t* UP, int32_t* LS) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    const int lim = P.max_blocks * kBlockTokens;
    int32_t carry = 0;
    for (int base = 0; base < P.B; base += 32) {
      const int b = base + lane;
      int32_t n = 0;
      if (b < P.B) {
        int32_t L = P.ctx[b];
        if (L < 0 || L > lim) {
          atomicOr(P.lv.err, ERR_CTX);
          L = L < 0 ? 0 : lim;
        }
        LS[b] = L;
        n = (L + P.T - 1) / P.T;
      }
      int32_t inc = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
      }
      if (b < P.B) UP[b] = carry + inc - n;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) UP[P.B] = carry;
  }
}

// Zero output rows of empty sequences (handled by CTA b % grid).
template <int D>
__device__ __forceinline__ void zero_empty_sequences(const DecodeParams& P, const int32_t* LS) {
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    if (LS[b] != 0) continue;
    for (int i = threadIdx.x; i < P.Hq * D; i += blockDim.x) P.out[(size_t)b * P.Hq * D + i] = 0;
  }
}

// Split-K epilogue, run by every consumer warp of the CTA (warp h owns query heads
// h*G .. h*G+G-1) after it has written its partial (m, l, acc[D]) of sequence b to
// slot blockIdx.x + b.  The CTA takes an arrival ticket on the sequence's counter;
// the CTA whose ticket completes the count merges the partials of CTAs c_lo..c_hi
// in CTA order (so the result does not depend on arrival order), writes the bf16
// output and resets the counter for the next launch.
template <int D, int G>
__device__ __forceinline__ void finish_split_sequence(const DecodeParams& P, int b, int32_t c_lo, int32_t c_hi,
                                                      int NC, int h, int32_t* flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __threadfence();
  named_barrier_sync(1, NC * 32);
  if (warp == 0 && lane == 0) {
    const int32_t ticket = atomicAdd(&P.counters[b], 1);
    const bool last = ticket == (c_hi - c_lo);
    if (last) P.counters[b] = 0;
    flag[0] = last ? 1 : 0;
  }
  named_barrier_sync(1, NC * 32);
  if (!flag[0]) return;
  __threadfence();
  // Lanes own parts for the max and the denominator, and dims for the numerator,
  // so that the L2 round trips overlap instead of chaining.
  const int nparts = c_hi - c_lo + 1;
  const size_t pstride = (size_t)P.Hq * (D + 2);  // CTAs c, c+1 use slots c+b, c+1+b
#pragma unroll 1
  for (int g = 0; g < G; ++g) {
    const size_t head = (size_t)h * G + g;
    const float* base = P.partials + (((size_t)c_lo + b) * P.Hq + head) * (D + 2);
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, __ldcg(base + (size_t)i * pstride));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float den = 0.f;
    for (int i = lane; i < nparts; i += 32) {
      const float* pp = base + (size_t)i * pstride;
      den += exp2f(__ldcg(pp) - M) * __ldcg(pp + 1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float inv = 1.0f / den;
    float num[D / 32];
#pragma unroll
    for (int j = 0; j < D / 32; ++j) num[j] = 0.f;
    for (int i0 = 0; i0 < nparts; i0 += 32) {
      const int i = i0 + lane;
      const float wgt = i < nparts ? exp2f(__ldcg(base + (size_t)i * pstride) - M) : 0.f;
      const int cnt = min(32, nparts - i0);
#pragma unroll 4
      for (int k = 0; k < cnt; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wgt, k);
        const float* pp = base + (size_t)(i0 + k) * pstride + 2;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) num[j] = fmaf(wk, __ldcg(pp + lane + 32 * j), num[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < D / 32; ++j) P.out[((size_t)b * P.Hq + head) * D + lane + 32 * j] = f2bf(num[j] * inv);
  }
}

}  // namespace pkv
