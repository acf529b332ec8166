// decode_packed_mma.cuh — paged decode attention over packed K4/V4, K8/V4, K8/V8
// pages on tensor-core tiles (fp16 in, fp32 accumulate).
//
// Work partition and split-K epilogue are those of the bf16 kernel
// (decode_mma.cuh): units of T tokens x all kv heads split evenly over one CTA per
// SM, a producer warp and one consumer warp per kv head.  Staging uses TMA tensor
// copies: each stored tensor of a slab (K codes, V codes, K meta, V meta) has a 2-D
// tensor map [tokens][all-heads row bytes]; a stage holds T tokens of each tensor as
// boxes of 16 tokens x W bytes (W = 128, 64, 32 or 16, the largest dividing the
// row), written with the W-byte shared-memory swizzle (16-byte chunk c of box row r
// lands at chunk c ^ f(r)), so reads of one column across 8 tokens are
// conflict-free.  A 32-token stage of K4/V4 with 8 heads of 128 dims is 24 box
// copies.  q comes with the first unit of a sequence (one bulk copy).  The packed
// pages are consumed directly, never expanded in memory (mlx-swift-lm PR #142,
// Summary: direct attention on packed pages):
//
//  * q is rotated into K's signed Hadamard basis (q~ = H diag(s) q / sqrt(D), FWHT
//    in per-warp shared scratch) when a sequence starts and kept as fp16 A
//    fragments (rows = query heads, rows >= G zero).
//  * QK, one affine group of 32 dims at a time: a code c becomes the fp16 value
//    1024 + c by OR-ing it into the mantissa of 1024 (exact; for 4-bit codes in odd
//    nibble positions the value is 1024 + 16c and the matching q entries are
//    stored divided by 16).  The group's product C = sum_k A_k (1024 + c_k') gives
//    q~.c = C - 1024 * sum_k A_k, and the stored (scale s, offset o) of the token
//    and group fold in on the accumulator fragment:
//        logit += s (C - bias) + o * sum(q~ over the group).
//    A consistent permutation of the 32 dims of a group is used on both operands
//    (the dot product does not depend on the order), chosen so that each lane's
//    B fragment comes from one 32-bit word of codes.
//  * PV as O^T = V^T P^T: the A operand holds V codes of two tokens per register,
//    dequantised in fp16 (v = s (c) + o with the tokens' own s and o), the B
//    operand is P (fp16) straight from the S accumulator fragments.  Each 16-row
//    M tile covers 16 dims of one group; the order of dims inside a group is
//    permuted so that a lane's two dims come from one half-word (4-bit) or one byte
//    pair (8-bit) of a code word, and the output store undoes the permutation.
#pragma once

#include <cuda_fp16.h>

#include "decode_common.cuh"

namespace pkv {

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t r) {
  return __half22float2(*reinterpret_cast<const __half2*>(&r));
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}

constexpr uint32_t kF16Magic2 = 0x64006400u;  // (1024.0h, 1024.0h)

template <int FMT, int D>
struct PackedTraits {
  static constexpr int KBITS = FMT == PKV_FMT_K4V4 ? 4 : 8;
  static constexpr int VBITS = FMT == PKV_FMT_K8V8 ? 8 : 4;
  static constexpr int KB = D * KBITS / 8;   // K code bytes per (token, head)
  static constexpr int VB = D * VBITS / 8;
  static constexpr int NG = D / kGroup;      // affine groups per row
  static constexpr int MB = NG * 8;          // (scale, offset) bytes per (token, head)
};

// B fragments of K for one group and one token (this lane's token of the n-tile):
// k-step ks in {0,1} of the group gets (b[ks][0], b[ks][1]).
// 4-bit: word t of the group holds elements 8t..8t+7 (element n in bits 4n..4n+3).
__device__ __forceinline__ void k_group_frags4(uint32_t w, uint32_t (&b)[2][2]) {
  const uint32_t w8 = w >> 8;
  b[0][0] = (w & 0x000F000Fu) | kF16Magic2;   // elements 0, 4      : 1024 + c
  b[0][1] = (w & 0x00F000F0u) | kF16Magic2;   // elements 1, 5      : 1024 + 16 c
  b[1][0] = (w8 & 0x000F000Fu) | kF16Magic2;  // elements 2, 6
  b[1][1] = (w8 & 0x00F000F0u) | kF16Magic2;  // elements 3, 7      : 1024 + 16 c
}

// 8-bit: k-step ks uses word 4 ks + t of the group: elements 16 ks + 4t + j.
__device__ __forceinline__ void k_group_frags8(uint32_t w0, uint32_t w1, uint32_t (&b)[2][2]) {
  b[0][0] = __byte_perm(w0, 0x64646464u, 0x4140);  // (1024 + c0, 1024 + c1)
  b[0][1] = __byte_perm(w0, 0x64646464u, 0x4342);  // (1024 + c2, 1024 + c3)
  b[1][0] = __byte_perm(w1, 0x64646464u, 0x4140);
  b[1][1] = __byte_perm(w1, 0x64646464u, 0x4342);
}

// Group-relative dims of the A (q) entries matching k_group_frags4/8, and whether the
// entry is stored divided by 16: k-step ks, register r (0: k = 2t, 2t+1; 1: k = 2t+8,
// 2t+9), half hh.
template <int KBITS>
__device__ __forceinline__ int k_dim(int t, int ks, int r, int hh, bool& div16) {
  if constexpr (KBITS == 4) {
    // ks 0: r0 -> elements (0, 4), r1 -> (1, 5)/16; ks 1: r0 -> (2, 6), r1 -> (3, 7)/16
    const int e = (ks ? 2 : 0) + r + 4 * hh;
    div16 = (r == 1);
    return 8 * t + e;
  } else {
    div16 = false;
    return 16 * ks + 4 * t + 2 * r + hh;
  }
}

// A fragments of V^T for one group, one 16-token chunk: the four code words of
// tokens (2t, 2t+1, 2t+8, 2t+9) at this lane's word; returns raw (1024 + c) fp16
// pairs a[mi][r] for M tile mi in {0,1}, register r in 0..3 (tokens pair 0: r 0,1;
// pair 1: r 2,3; rows g: r 0,2; rows g+8: r 1,3).
template <int VBITS>
__device__ __forceinline__ void v_group_frags(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, int g,
                                              uint32_t (&a)[2][4]) {
  if constexpr (VBITS == 4) {
    const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;  // half-word g&1 of each token's word
    const uint32_t x01 = __byte_perm(w0, w1, sel);
    const uint32_t x23 = __byte_perm(w2, w3, sel);
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      a[mi][0] = ((x01 >> (8 * mi)) & 0x000F000Fu) | kF16Magic2;      // nibble 2mi   (row g)
      a[mi][1] = ((x01 >> (8 * mi + 4)) & 0x000F000Fu) | kF16Magic2;  // nibble 2mi+1 (row g+8)
      a[mi][2] = ((x23 >> (8 * mi)) & 0x000F000Fu) | kF16Magic2;
      a[mi][3] = ((x23 >> (8 * mi + 4)) & 0x000F000Fu) | kF16Magic2;
    }
  } else {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      const int j0 = 2 * mi, j1 = 2 * mi + 1;  // bytes of the word: rows g and g+8
      a[mi][0] = (__byte_perm(w0, w1, (uint32_t)(j0 | (j0 << 4) | ((4 + j0) << 8) | ((4 + j0) << 12))) & 0x00FF00FFu) | kF16Magic2;
      a[mi][1] = (__byte_perm(w0, w1, (uint32_t)(j1 | (j1 << 4) | ((4 + j1) << 8) | ((4 + j1) << 12))) & 0x00FF00FFu) | kF16Magic2;
      a[mi][2] = (__byte_perm(w2, w3, (uint32_t)(j0 | (j0 << 4) | ((4 + j0) << 8) | ((4 + j0) << 12))) & 0x00FF00FFu) | kF16Magic2;
      a[mi][3] = (__byte_perm(w2, w3, (uint32_t)(j1 | (j1 << 4) | ((4 + j1) << 8) | ((4 + j1) << 12))) & 0x00FF00FFu) | kF16Magic2;
    }
  }
}

// Byte offset, inside one (token, head) V code row, of this lane's word for group grp.
template <int VBITS>
__device__ __forceinline__ int v_word_offset(int grp, int g) {
  return VBITS == 4 ? 16 * grp + 4 * (g >> 1) : 32 * grp + 4 * g;
}

// Output dim of M tile mi of group grp, row half hh (0: row g, 1: row g+8).
template <int VBITS>
__device__ __forceinline__ int v_out_dim(int grp, int mi, int hh, int g) {
  return VBITS == 4 ? 32 * grp + 8 * (g >> 1) + 4 * (g & 1) + 2 * mi + hh : 32 * grp + 4 * g + 2 * mi + hh;
}

// One stored tensor's region of a stage: byte offset, log2 of the box width, boxes
// per token row.
struct SwzRegion {
  int off, lg, nx;
};

// Byte offset in the stage of byte b of token tok's row (all kv heads) in region z:
// box (tok / 16, b / W), box row tok % 16, 16-byte chunk XOR-swizzled by the row as
// the W-byte swizzle mode stores it (W=128: r & 7; 64: (r >> 1) & 3; 32: (r >> 2) & 1).
__device__ __forceinline__ int swz(const SwzRegion& z, int tok, int b) {
  const int r = tok & 15;
  const int sw = z.lg == 7 ? (r & 7) : (z.lg == 6 ? ((r >> 1) & 3) : (z.lg == 5 ? ((r >> 2) & 1) : 0));
  const int mask = (1 << z.lg) - 1;
  return z.off + ((((tok >> 4) * z.nx + (b >> z.lg)) * 16 + r) << z.lg) + (((((b & mask) >> 4) ^ sw) << 4) | (b & 15));
}

__device__ __forceinline__ int ilog2i(int v) { return 31 - __clz(v); }

// W128: every stored tensor's all-heads row is a multiple of 128 bytes, so every box
// is 128 bytes wide; then all addressing below reduces to per-lane constants.
template <int FMT, int D, int G, bool W128>
__global__ void __launch_bounds__(kMaxThreads, 1) decode_packed_mma_kernel(const DecodeParams P) {
  using Tr = PackedTraits<FMT, D>;
  static_assert(G >= 1 && G <= 8 && D % 32 == 0, "geometry");
  constexpr int NG = Tr::NG;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = P.lv.hkv;
  const int NC = hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = P.T, NS = P.NS, B = P.B;
  int32_t* err = P.lv.err;
  // Per-token rows of all kv heads in the slab; stage regions of T such rows.
  const int KR = hkv * Tr::KB, VR = hkv * Tr::VB, MR = hkv * Tr::MB;
  const int rows_b[4] = {KR, VR, MR, MR};
  int off[5];
  off[0] = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) off[k + 1] = off[k] + ((T * rows_b[k] + 1023) & ~1023);
  const int offQ = off[4];
  const int QB = P.Hq * D * 2;
  SwzRegion zr[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    zr[k].off = off[k];
    zr[k].lg = ilog2i(P.lv.box_bytes[k]);
    zr[k].nx = rows_b[k] >> zr[k].lg;
  }

  // Stages start on a 1024-byte boundary (the 128-byte swizzle repeats every 1 KB).
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)NS * P.stage_bytes);
  uint64_t* empty = full + NS;
  const uint8_t** tab = reinterpret_cast<const uint8_t**>(empty + NS);
  int32_t* UP = reinterpret_cast<int32_t*>(tab + kSmemTableEntries);
  int32_t* LS = UP + (B + 1);
  float* qscr = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(LS + B) + 15) & ~uintptr_t(15));

  decode_prologue(P, full, empty, NC, UP, LS, tab);
  __syncthreads();
  const int32_t U = UP[B];
  const int32_t C = (U + (int32_t)gridDim.x - 1) / (int32_t)gridDim.x;
  zero_empty_sequences<D>(P, LS);
  if (C == 0) return;
  const int32_t u0 = (int32_t)blockIdx.x * C;
  const int32_t u1 = min(U, u0 + C);
  if (u0 >= u1) return;

  if (warp == NC) {
    // ----------------------------- producer ---------------------------------
    const bool use_stab = smem_table_entries(P) > 0;
    const uint64_t kv_policy = l2_policy_evict_first();
    const int nboxes = (T / 16) * (zr[0].nx + zr[1].nx + zr[2].nx + zr[3].nx);
    int issued = 0;
    bool dead = false;
    for (int32_t ub = u0; ub < u1 && !dead; ub += 32) {
      const int32_t u = ub + lane;
      const uint8_t* mapbase = nullptr;
      const uint8_t* qsrc = nullptr;
      int y0 = 0, ok = 0;
      if (u < u1) {
        const int b = find_seq(UP, B, u);
        if (u == u0 || u == UP[b]) qsrc = reinterpret_cast<const uint8_t*>(P.q + (size_t)b * P.Hq * D);
        const int32_t tok0 = (u - UP[b]) * T;
        const int j = tok0 / kBlockTokens, slot0 = tok0 % kBlockTokens;
        const int32_t row = P.bt[(size_t)b * P.max_blocks + j];
        if (row >= 0 && (int64_t)row < P.lv.rows_capacity) {
          const int32_t slab = row / P.lv.slab_blocks;
          const int32_t r = row - slab * P.lv.slab_blocks;
          const uint8_t* ent0 = use_stab ? tab[(size_t)slab * P.lv.n_kinds]
                                         : P.lv.tab.base[(size_t)slab * P.lv.tab.stride];
          mapbase = ent0 + P.lv.map_delta;
          y0 = r * kBlockTokens + slot0;
          ok = 1;
        } else {
          atomicOr(err, ERR_ROW);
        }
      }
      const int cnt = min(32, u1 - ub);
      for (int i = 0; i < cnt; ++i) {
        const uint8_t* mb = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)mapbase, i);
        const uint8_t* qs = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)qsrc, i);
        const int yi = __shfl_sync(0xffffffffu, y0, i);
        const int oki = __shfl_sync(0xffffffffu, ok, i);
        const int s = issued % NS;
        if (lane == 0) {
          if (issued >= NS && !mbar_wait_bounded(&empty[s], ((issued / NS) & 1) ^ 1, err)) dead = true;
          if (!dead)
            mbar_arrive_expect_tx(&full[s], (oki ? (uint32_t)(T * (KR + VR + 2 * MR)) : 0u) + (qs ? (uint32_t)QB : 0u));
        }
        dead = __shfl_sync(0xffffffffu, dead, 0);
        if (dead) break;
        __syncwarp();
        uint8_t* st = stages + (size_t)s * P.stage_bytes;
        if (qs && lane == 31) bulk_g2s(st + offQ, qs, (uint32_t)QB, &full[s]);
        if (oki) {
          for (int c = lane; c < nboxes; c += 32) {
            // box c -> (kind, row of boxes cy, column cx)
            int kind = 0, rem = c;
            while (rem >= (T / 16) * zr[kind].nx) {
              rem -= (T / 16) * zr[kind].nx;
              ++kind;
            }
            const int cy = rem / zr[kind].nx, cx = rem - cy * zr[kind].nx;
            const uint8_t* map = mb + kind * 128;
            tensormap_acquire(map);
            tma_load_2d(st + zr[kind].off + ((cy * zr[kind].nx + cx) << (zr[kind].lg + 4)), map,
                        cx << zr[kind].lg, yi + 16 * cy, &full[s], kv_policy);
          }
        }
        ++issued;
      }
    }
    if (lane == 0) {
      const int first = issued > NS ? issued - NS : 0;
      for (int n = first; n < issued; ++n) mbar_wait_bounded(&full[n % NS], (n / NS) & 1, err);
    }
    return;
  }

  // ------------------------------ consumers ---------------------------------
  const int h = warp;
  const int g = lane >> 2, t = lane & 3;
  float* qs = qscr + (size_t)warp * G * D;
  uint32_t qa[NG][2][2];  // A fragments per group, k-step, register (rows g; rows g+8 zero)
  float qbias[NG], qsum[NG];
  float o[NG][2][4];      // O^T accumulators: group, M tile, fragment
  float m_run = -INFINITY, l_run = 0.f;
  bool dead = false;

  int b = find_seq(UP, B, u0);
  int n = 0;
  for (int32_t u = u0; u < u1; ++u, ++n) {
    while (u >= UP[b + 1]) ++b;
    const bool seg_start = (u == u0) || (u == UP[b]);
    const bool seg_end = (u == u1 - 1) || (u == UP[b + 1] - 1);
    if (seg_start) {
#pragma unroll
      for (int grp = 0; grp < NG; ++grp)
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[grp][mi][i] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }
    const int32_t tok0 = (u - UP[b]) * T;
    const int nv = min(T, LS[b] - tok0);
    const int s = n % NS;
    if (!dead && !mbar_wait_bounded(&full[s], (n / NS) & 1, err)) dead = true;
    dead = __shfl_sync(0xffffffffu, dead, 0);
    const uint8_t* st = stages + (size_t)s * P.stage_bytes;
    if (!dead && seg_start) {
      // q~ = H diag(s) q / sqrt(D) for this kv head's G query heads (FWHT in scratch).
      const uint16_t* qsm = reinterpret_cast<const uint16_t*>(st + offQ) + (size_t)h * G * D;
      for (int i = lane; i < G * D; i += 32) qs[i] = __uint_as_float((uint32_t)qsm[i] << 16) * P.signs[i % D];
      __syncwarp();
      for (int hs = 1; hs < D; hs <<= 1) {
        for (int i = lane; i < G * D / 2; i += 32) {
          const int gg = i / (D / 2), pi = i % (D / 2);
          const int a = gg * D + (pi / hs) * 2 * hs + (pi % hs);
          const float x = qs[a], y = qs[a + hs];
          qs[a] = x + y;
          qs[a + hs] = x - y;
        }
        __syncwarp();
      }
#pragma unroll
      for (int grp = 0; grp < NG; ++grp) {
        float bsum = 0.f, tsum = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float v[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              bool d16;
              const int dd = 32 * grp + k_dim<Tr::KBITS>(t, ks, r, hh, d16);
              const float qv = g < G ? qs[g * D + dd] * P.inv_sqrt_d : 0.f;
              v[hh] = d16 ? qv * 0.0625f : qv;
            }
            qa[grp][ks][r] = pack_f16x2(v[0], v[1]);
            const float2 back = unpack_f16x2(qa[grp][ks][r]);  // the values the MMA sees
            bsum += back.x + back.y;
            bool d16;
            (void)k_dim<Tr::KBITS>(t, ks, r, 0, d16);
            tsum += d16 ? 16.f * (back.x + back.y) : (back.x + back.y);
          }
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
        tsum += __shfl_xor_sync(0xffffffffu, tsum, 1);
        tsum += __shfl_xor_sync(0xffffffffu, tsum, 2);
        qbias[grp] = 1024.f * bsum;
        qsum[grp] = tsum;
      }
      __syncwarp();
    }
    if (!dead) {
      // Fast-path addressing (W128).  A lane touches token rows whose 128-byte
      // swizzle key is fixed: K code rows 8j+g (key g), meta and V rows 8p+2t+e
      // (key 2t^e).  base = region + head's box column + first row (+ lane bytes);
      // key = (head's chunk ^ row key) << 4.  Chunk offsets inside the row are
      // compile-time and enter through one XOR with the key.
      const int KBASE = zr[0].off + ((h * Tr::KB) >> 7) * 2048 + g * 128 + 4 * t;
      const int KKEY = ((((h * Tr::KB) >> 4) & 7) ^ g) << 4;
      const int MKEY = ((((h * Tr::MB) >> 4) & 7) ^ (2 * t)) << 4;
      const int KMBASE = zr[2].off + ((h * Tr::MB) >> 7) * 2048 + 2 * t * 128;
      const int VMBASE = zr[3].off + ((h * Tr::MB) >> 7) * 2048 + 2 * t * 128;
      const int VBASE = zr[1].off + ((h * Tr::VB) >> 7) * 2048 + 2 * t * 128 +
                        (Tr::VBITS == 4 ? 4 * (g >> 1) : 4 * (g & 3));
      const int VKEY = (((((h * Tr::VB) >> 4) & 7) ^ (2 * t)) << 4) ^ (Tr::VBITS == 8 ? 16 * (g >> 2) : 0);
      for (int kc = 0; kc * 16 < nv; ++kc) {
        // ---- logits for 16 tokens: n-tiles 2kc, 2kc+1 ----
        float x[2][2];
        if constexpr (W128) {
          const uint8_t* kq = st + KBASE + kc * zr[0].nx * 2048;
          const uint8_t* km = st + KMBASE + kc * zr[2].nx * 2048;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float sa0 = 0.f, sa1 = 0.f;
#pragma unroll
            for (int gp = 0; gp < NG / 2; ++gp) {
              // (scale, offset) of groups 2gp, 2gp+1 for tokens 8j+2t (e=0) and 8j+2t+1 (e=1)
              const int moc = 16 * gp;
              const float4 me0 = *reinterpret_cast<const float4*>(km + 1024 * j + (moc >> 7) * 2048 + (MKEY ^ (moc & 112)));
              const float4 me1 =
                  *reinterpret_cast<const float4*>(km + 1024 * j + 128 + (moc >> 7) * 2048 + (MKEY ^ ((moc & 112) ^ 16)));
#pragma unroll
              for (int q2 = 0; q2 < 2; ++q2) {
                const int grp = 2 * gp + q2;
                const int oc = grp * (kGroup * Tr::KBITS / 8);
                uint32_t bfr[2][2];
                if constexpr (Tr::KBITS == 4) {
                  k_group_frags4(*reinterpret_cast<const uint32_t*>(kq + 1024 * j + (oc >> 7) * 2048 + (KKEY ^ (oc & 112))),
                                 bfr);
                } else {
                  k_group_frags8(
                      *reinterpret_cast<const uint32_t*>(kq + 1024 * j + (oc >> 7) * 2048 + (KKEY ^ (oc & 112))),
                      *reinterpret_cast<const uint32_t*>(kq + 1024 * j + ((oc + 16) >> 7) * 2048 +
                                                         (KKEY ^ ((oc + 16) & 112))),
                      bfr);
                }
                float cacc[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(cacc, qa[grp][0][0], 0u, qa[grp][0][1], 0u, bfr[0][0], bfr[0][1]);
                mma_f16_16816(cacc, qa[grp][1][0], 0u, qa[grp][1][1], 0u, bfr[1][0], bfr[1][1]);
                const float s0 = q2 ? me0.z : me0.x, o0 = q2 ? me0.w : me0.y;
                const float s1 = q2 ? me1.z : me1.x, o1 = q2 ? me1.w : me1.y;
                sa0 = fmaf(s0, cacc[0] - qbias[grp], fmaf(o0, qsum[grp], sa0));
                sa1 = fmaf(s1, cacc[1] - qbias[grp], fmaf(o1, qsum[grp], sa1));
              }
            }
            const int tk = kc * 16 + 8 * j + 2 * t;
            x[j][0] = tk < nv ? sa0 * P.scale_log2 : -INFINITY;
            x[j][1] = tk + 1 < nv ? sa1 * P.scale_log2 : -INFINITY;
          }
        } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tb = kc * 16 + 8 * j;  // first token of the n-tile
          float sa0 = 0.f, sa1 = 0.f;
#pragma unroll
          for (int grp = 0; grp < NG; ++grp) {
            uint32_t bfr[2][2];
            const int kb = h * Tr::KB + grp * (kGroup * Tr::KBITS / 8) + 4 * t;
            if constexpr (Tr::KBITS == 4) {
              k_group_frags4(*reinterpret_cast<const uint32_t*>(st + swz(zr[0], tb + g, kb)), bfr);
            } else {
              k_group_frags8(*reinterpret_cast<const uint32_t*>(st + swz(zr[0], tb + g, kb)),
                             *reinterpret_cast<const uint32_t*>(st + swz(zr[0], tb + g, kb + 16)), bfr);
            }
            float cacc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16_16816(cacc, qa[grp][0][0], 0u, qa[grp][0][1], 0u, bfr[0][0], bfr[0][1]);
            mma_f16_16816(cacc, qa[grp][1][0], 0u, qa[grp][1][1], 0u, bfr[1][0], bfr[1][1]);
            const int mbo = h * Tr::MB + 8 * grp;
            const float2 m0 = *reinterpret_cast<const float2*>(st + swz(zr[2], tb + 2 * t, mbo));
            const float2 m1 = *reinterpret_cast<const float2*>(st + swz(zr[2], tb + 2 * t + 1, mbo));
            sa0 = fmaf(m0.x, cacc[0] - qbias[grp], fmaf(m0.y, qsum[grp], sa0));
            sa1 = fmaf(m1.x, cacc[1] - qbias[grp], fmaf(m1.y, qsum[grp], sa1));
          }
          const int tk = tb + 2 * t;
          x[j][0] = tk < nv ? sa0 * P.scale_log2 : -INFINITY;
          x[j][1] = tk + 1 < nv ? sa1 * P.scale_log2 : -INFINITY;
        }
        }
        // ---- online softmax for head g ----
        float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool grow = mx > m_run;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? exp2f(m_run - mx) : 1.0f;
          if (grow) m_run = mx;
          l_run *= alpha;
          const float ae = __shfl_sync(0xffffffffu, alpha, 8 * t);
          const float ao = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
          for (int grp = 0; grp < NG; ++grp)
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
              o[grp][mi][0] *= ae;
              o[grp][mi][2] *= ae;
              o[grp][mi][1] *= ao;
              o[grp][mi][3] *= ao;
            }
        }
        const float p00 = exp2f(x[0][0] - m_run), p01 = exp2f(x[0][1] - m_run);
        const float p10 = exp2f(x[1][0] - m_run), p11 = exp2f(x[1][1] - m_run);
        l_run += (p00 + p01) + (p10 + p11);
        const uint32_t pb0 = pack_f16x2(p00, p01), pb1 = pack_f16x2(p10, p11);
        // ---- O^T += V^T P^T over these 16 tokens ----
        const int t0 = kc * 16 + 2 * t;
        if constexpr (W128) {
          const uint8_t* vq = st + VBASE + kc * zr[1].nx * 2048;
          const uint8_t* vm = st + VMBASE + kc * zr[3].nx * 2048;
#pragma unroll
          for (int gp = 0; gp < NG / 2; ++gp) {
            // (scale, offset) of groups 2gp, 2gp+1 for tokens 2t+e+8p
            const int moc = 16 * gp;
            float4 mv[2][2];
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
              for (int e = 0; e < 2; ++e)
                mv[pp][e] = *reinterpret_cast<const float4*>(vm + 1024 * pp + 128 * e + (moc >> 7) * 2048 +
                                                             (MKEY ^ ((moc & 112) ^ (16 * e))));
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              const int grp = 2 * gp + q2;
              const int oc = Tr::VBITS == 4 ? 16 * grp : 32 * grp;
              uint32_t w[2][2];
#pragma unroll
              for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                  w[pp][e] = *reinterpret_cast<const uint32_t*>(vq + 1024 * pp + 128 * e + (oc >> 7) * 2048 +
                                                                (VKEY ^ ((oc & 112) ^ (16 * e))));
              const float2 s0 = q2 ? make_float2(mv[0][0].z, mv[0][0].w) : make_float2(mv[0][0].x, mv[0][0].y);
              const float2 s1 = q2 ? make_float2(mv[0][1].z, mv[0][1].w) : make_float2(mv[0][1].x, mv[0][1].y);
              const float2 s2 = q2 ? make_float2(mv[1][0].z, mv[1][0].w) : make_float2(mv[1][0].x, mv[1][0].y);
              const float2 s3 = q2 ? make_float2(mv[1][1].z, mv[1][1].w) : make_float2(mv[1][1].x, mv[1][1].y);
              const uint32_t sc01 = pack_f16x2(s0.x, s1.x), of01 = pack_f16x2(s0.y, s1.y);
              const uint32_t sc23 = pack_f16x2(s2.x, s3.x), of23 = pack_f16x2(s2.y, s3.y);
              uint32_t a[2][4];
              v_group_frags<Tr::VBITS>(w[0][0], w[0][1], w[1][0], w[1][1], g, a);
#pragma unroll
              for (int mi = 0; mi < 2; ++mi) {
                const uint32_t d0 = hfma2_u32(hsub2_u32(a[mi][0], kF16Magic2), sc01, of01);
                const uint32_t d1 = hfma2_u32(hsub2_u32(a[mi][1], kF16Magic2), sc01, of01);
                const uint32_t d2 = hfma2_u32(hsub2_u32(a[mi][2], kF16Magic2), sc23, of23);
                const uint32_t d3 = hfma2_u32(hsub2_u32(a[mi][3], kF16Magic2), sc23, of23);
                mma_f16_16816(o[grp][mi], d0, d1, d2, d3, pb0, pb1);
              }
            }
          }
        } else {
#pragma unroll
        for (int grp = 0; grp < NG; ++grp) {
          const int vb = h * Tr::VB + v_word_offset<Tr::VBITS>(grp, g);
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(st + swz(zr[1], t0, vb));
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(st + swz(zr[1], t0 + 1, vb));
          const uint32_t w2 = *reinterpret_cast<const uint32_t*>(st + swz(zr[1], t0 + 8, vb));
          const uint32_t w3 = *reinterpret_cast<const uint32_t*>(st + swz(zr[1], t0 + 9, vb));
          const int mbo = h * Tr::MB + 8 * grp;
          const float2 s0 = *reinterpret_cast<const float2*>(st + swz(zr[3], t0, mbo));
          const float2 s1 = *reinterpret_cast<const float2*>(st + swz(zr[3], t0 + 1, mbo));
          const float2 s2 = *reinterpret_cast<const float2*>(st + swz(zr[3], t0 + 8, mbo));
          const float2 s3 = *reinterpret_cast<const float2*>(st + swz(zr[3], t0 + 9, mbo));
          const uint32_t sc01 = pack_f16x2(s0.x, s1.x), of01 = pack_f16x2(s0.y, s1.y);
          const uint32_t sc23 = pack_f16x2(s2.x, s3.x), of23 = pack_f16x2(s2.y, s3.y);
          uint32_t a[2][4];
          v_group_frags<Tr::VBITS>(w0, w1, w2, w3, g, a);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            // v = s * c + o in fp16, with c = (1024 + c) - 1024 exact
            const uint32_t d0 = hfma2_u32(hsub2_u32(a[mi][0], kF16Magic2), sc01, of01);
            const uint32_t d1 = hfma2_u32(hsub2_u32(a[mi][1], kF16Magic2), sc01, of01);
            const uint32_t d2 = hfma2_u32(hsub2_u32(a[mi][2], kF16Magic2), sc23, of23);
            const uint32_t d3 = hfma2_u32(hsub2_u32(a[mi][3], kF16Magic2), sc23, of23);
            mma_f16_16816(o[grp][mi], d0, d1, d2, d3, pb0, pb1);
          }
        }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    if (seg_end) {
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
      const float me = __shfl_sync(0xffffffffu, m_run, 8 * t), mo = __shfl_sync(0xffffffffu, m_run, 8 * t + 4);
      const float le = __shfl_sync(0xffffffffu, l_run, 8 * t), lo = __shfl_sync(0xffffffffu, l_run, 8 * t + 4);
      const int he = 2 * t, ho = 2 * t + 1;
      const int32_t c_lo = UP[b] / C, c_hi = (UP[b + 1] - 1) / C;
      if (c_lo == c_hi) {
        const float ie = 1.0f / le, io = 1.0f / lo;
        uint16_t* oe = P.out + ((size_t)b * P.Hq + (size_t)h * G + he) * D;
        uint16_t* oo = P.out + ((size_t)b * P.Hq + (size_t)h * G + ho) * D;
#pragma unroll
        for (int grp = 0; grp < NG; ++grp)
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            const int d0 = v_out_dim<Tr::VBITS>(grp, mi, 0, g), d1 = v_out_dim<Tr::VBITS>(grp, mi, 1, g);
            if (he < G) {
              oe[d0] = f2bf(o[grp][mi][0] * ie);
              oe[d1] = f2bf(o[grp][mi][2] * ie);
            }
            if (ho < G) {
              oo[d0] = f2bf(o[grp][mi][1] * io);
              oo[d1] = f2bf(o[grp][mi][3] * io);
            }
          }
      } else {
        float* pe = partial_ptr(P, D, (size_t)blockIdx.x, b, (size_t)h * G + he);
        float* po = partial_ptr(P, D, (size_t)blockIdx.x, b, (size_t)h * G + ho);
        if (he < G && g == 0) {
          pe[0] = me;
          pe[1] = le;
        }
        if (ho < G && g == 0) {
          po[0] = mo;
          po[1] = lo;
        }
#pragma unroll
        for (int grp = 0; grp < NG; ++grp)
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            const int d0 = v_out_dim<Tr::VBITS>(grp, mi, 0, g), d1 = v_out_dim<Tr::VBITS>(grp, mi, 1, g);
            if (he < G) {
              pe[kPartialHeader + d0] = o[grp][mi][0];
              pe[kPartialHeader + d1] = o[grp][mi][2];
            }
            if (ho < G) {
              po[kPartialHeader + d0] = o[grp][mi][1];
              po[kPartialHeader + d1] = o[grp][mi][3];
            }
          }
      }
    }
  }
}

template <int FMT, int D, int G, bool W128>
cudaError_t launch_decode_packed_mma_t(const DecodeArgs& a) {
  using Tr = PackedTraits<FMT, D>;
  DecodeParams P;
  P.lv = a.lv;
  P.B = a.B;
  P.Hq = a.Hq;
  P.max_blocks = a.max_blocks;
  P.q = a.q;
  P.bt = a.bt;
  P.ctx = a.ctx;
  P.scale_log2 = a.scale_log2;
  P.inv_sqrt_d = a.inv_sqrt_d;
  P.signs = a.signs;
  P.out = a.out;
  P.counters = a.counters;
  P.partials = a.partials;
  P.T = a.tokens_per_stage;
  P.NS = a.n_stages;
  const int hkv = a.lv.hkv;
  P.stage_bytes = packed_stage_bytes(P.T, hkv * Tr::KB, hkv * Tr::VB, hkv * Tr::MB, a.Hq * D * 2);
  auto kern = decode_packed_mma_kernel<FMT, D, G, W128>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_with_pdl(kern, a.grid, (hkv + 1) * 32, a.smem_bytes, a.stream, P);
  if (e != cudaSuccess) return e;
  return launch_combine<D>(P, a.grid, a.stream);
}

template <int FMT>
cudaError_t launch_decode_packed_mma(const DecodeArgs& a) {
  const bool w128 = a.lv.box_bytes[0] == 128 && a.lv.box_bytes[1] == 128 && a.lv.box_bytes[2] == 128 &&
                    a.lv.box_bytes[3] == 128;
#define PKV_CASE(DD, GG)                                                      \
  if (a.D == DD && a.G == GG)                                                 \
    return w128 ? launch_decode_packed_mma_t<FMT, DD, GG, true>(a)            \
                : launch_decode_packed_mma_t<FMT, DD, GG, false>(a);
  PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
  PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
