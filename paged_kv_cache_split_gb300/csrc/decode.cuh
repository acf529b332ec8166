// decode.cuh — batched single-token paged decode attention (split-K flash
// decoding) over the chunked-slab pool, for one stored format.
//
// What it computes: for every sequence b and query head h (GQA: KV head h / G),
//   out[b,h] = softmax(scale * q[b,h] . K_b^T) V_b   over tokens [0, ctx[b]),
// single query token, no mask (mlxcel #2171, "one KV storage abstraction",
// Proposed Solution and Edge cases).  Packed formats consume the stored codes
// directly, dequantising in registers (mlx-swift-lm #142, Summary: "direct
// attention consumes packed pages without expanding the history"); q is rotated
// into K's signed Hadamard basis in the prologue of each sequence.
//
// GB300 design.
//  * Work unit = T tokens of one sequence for ALL kv heads.  In a slab
//    [slab_blocks, 32, Hkv, row] those bytes are contiguous per stored tensor, so
//    one 1-D bulk copy (cp.async.bulk, completing on an mbarrier) moves a whole
//    unit of K (and one each for V and the two metadata tensors).
//  * Units of all sequences are laid end to end and split evenly over the CTAs
//    (one per SM); the split is computed on the device from ctx, with no host sync.
//  * Warp specialisation: one producer warp walks the CTA's units, reads the block
//    table and the per-slab base-pointer table (mlxcel #235, touch point 4) and
//    issues the bulk copies into an NS-deep ring; consumer warp w owns kv head w.
//  * Consumer lane layout: NCG lanes share one token (each owns D/NCG dims); the
//    warp covers 32/NCG tokens per sub-step.  q and the output accumulator live in
//    registers for the whole sequence; logits are reduced with NCG-wide xor
//    shuffles; the online softmax works in base 2 (q is pre-scaled by scale*log2 e).
//  * A sequence split over several CTAs leaves (m, l, acc) partials; the last CTA
//    to finish it (atomic ticket, no spin) merges them in CTA order, so results are
//    deterministic; a sequence inside one CTA is written directly.
//  * Every wait is bounded (about 1 s) and reports ERR_TIMEOUT instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_common.cuh"

namespace pkv {

template <int FMT, int D, int G>
struct DecodeTraits {
  static constexpr int KBITS = FMT == PKV_FMT_BF16 ? 16 : (FMT == PKV_FMT_K4V4 ? 4 : 8);
  static constexpr int VBITS = FMT == PKV_FMT_BF16 ? 16 : (FMT == PKV_FMT_K8V8 ? 8 : 4);
  static constexpr bool PACKED = FMT != PKV_FMT_BF16;
  static constexpr int KB = D * KBITS / 8;  // bytes of one (token, head) K row
  static constexpr int VB = D * VBITS / 8;
  static constexpr int MB = PACKED ? (D / kGroup) * 8 : 0;  // (scale, offset) pairs
  // Lanes per token: at least 8 when a row has 128+ bytes (then 8 consecutive lanes
  // read 128 contiguous bytes: conflict-free 16-byte shared loads), and enough that
  // q and the accumulator take at most 64 registers each.
  static constexpr int NCG_A = (KB / 16 < 8) ? KB / 16 : 8;
  static constexpr int NCG_B = D * G / 64;
  static constexpr int NCG = (NCG_A > NCG_B ? NCG_A : NCG_B) < 1 ? 1 : (NCG_A > NCG_B ? NCG_A : NCG_B);
  static constexpr int TSUB = 32 / NCG;  // tokens per warp sub-step
  static constexpr int KSEG = KB / NCG, VSEG = VB / NCG;  // bytes per lane per token
  static constexpr int KLU = KSEG < 16 ? KSEG : 16, VLU = VSEG < 16 ? VSEG : 16;  // load unit
  static constexpr int KP = KSEG / KLU, VP = VSEG / VLU;  // pieces per lane
  static constexpr int KEPP = KLU * 8 / KBITS, VEPP = VLU * 8 / VBITS;  // values per piece
  static constexpr int DPL = D / NCG;  // dims per lane
  static_assert(NCG <= 32 && (NCG & (NCG - 1)) == 0, "lanes per token");
  static_assert(KSEG >= 4 && VSEG >= 4, "at least one word per lane");
  static_assert(KP * KEPP == DPL && VP * VEPP == DPL, "piece geometry");
  static_assert(!PACKED || (KEPP <= kGroup && VEPP <= kGroup), "a piece stays inside one group");
};

// ---- conversions of one loaded piece (w[] = LU/4 words) to floats ------------
template <int BITS, int LU>
__device__ __forceinline__ void piece_to_float(const uint32_t (&w)[LU / 4], float (&f)[LU * 8 / BITS]) {
  if constexpr (BITS == 16) {
#pragma unroll
    for (int i = 0; i < LU / 4; ++i) bf16x2_to_f32(w[i], f[2 * i], f[2 * i + 1]);
  } else if constexpr (BITS == 8) {
    // Exponent-bias conversion: the byte becomes the low mantissa bits of 2^23,
    // so (bits as float) - 2^23 is the byte's value exactly.
#pragma unroll
    for (int i = 0; i < LU / 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) f[4 * i + j] = __uint_as_float(__byte_perm(w[i], 0x4B000000u, 0x7650 + j)) - 8388608.0f;
  } else {
#pragma unroll
    for (int i = 0; i < LU / 4; ++i) {
      const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[8 * i + 2 * j] = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650 + j)) - 8388608.0f;
        f[8 * i + 2 * j + 1] = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650 + j)) - 8388608.0f;
      }
    }
  }
}

template <int LU>
__device__ __forceinline__ void load_piece(const uint8_t* p, uint32_t (&w)[LU / 4]) {
  if constexpr (LU == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (LU == 8) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

template <int FMT, int D, int G>
__global__ void __launch_bounds__(kMaxThreads, 1) decode_kernel(const DecodeParams P) {
  using Tr = DecodeTraits<FMT, D, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = P.lv.hkv;
  const int NC = hkv;  // consumer warps
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = P.T, NS = P.NS, B = P.B;
  int32_t* err = P.lv.err;

  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * P.stage_bytes);
  uint64_t* empty = full + NS;
  const uint8_t** tab = reinterpret_cast<const uint8_t**>(empty + NS);  // [kSmemTableEntries]
  int32_t* UP = reinterpret_cast<int32_t*>(tab + kSmemTableEntries);  // [B + 1] unit prefix
  int32_t* LS = UP + (B + 1);                             // [B] clamped lengths
  int32_t* flag = LS + B;                                 // [4]
  float* qscr = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(flag + 4) + 15) & ~uintptr_t(15));

  decode_prologue(P, full, empty, NC, UP, LS, tab);
  __syncthreads();

  const int32_t U = UP[B];
  const int32_t C = (U + (int32_t)gridDim.x - 1) / (int32_t)gridDim.x;
  zero_empty_sequences<D>(P, LS);
  if (C == 0) return;
  const int32_t u0 = (int32_t)blockIdx.x * C;
  const int32_t u1 = min(U, u0 + C);
  if (u0 >= u1) return;

  const int KBt = Tr::KB, VBt = Tr::VB, MBt = Tr::MB;
  const int off_v = T * hkv * KBt;
  const int off_km = off_v + T * hkv * VBt;
  const int off_vm = off_km + T * hkv * MBt;

  if (warp == NC) {
    // ----------------------------- producer ---------------------------------
    const bool use_stab = smem_table_entries(P) > 0;
    const uint64_t kv_policy = l2_policy_evict_first();  // K/V are read once
    int issued = 0;
    bool dead = false;
    for (int32_t ub = u0; ub < u1 && !dead; ub += 32) {
      const int32_t u = ub + lane;
      const uint8_t* src[4] = {nullptr, nullptr, nullptr, nullptr};
      int nvc = 0;
      if (u < u1) {
        const int b = find_seq(UP, B, u);
        const int32_t tok0 = (u - UP[b]) * T;
        const int j = tok0 / kBlockTokens, slot0 = tok0 % kBlockTokens;
        const int nv = min(T, LS[b] - tok0);
        const int32_t row = P.bt[(size_t)b * P.max_blocks + j];
        if (row >= 0 && (int64_t)row < P.lv.rows_capacity) {
          const int32_t slab = row / P.lv.slab_blocks;
          const int32_t r = row - slab * P.lv.slab_blocks;
          const uint8_t* const* ent = use_stab ? tab + (size_t)slab * P.lv.n_kinds
                                                : P.lv.tab.base + (size_t)slab * P.lv.tab.stride;
          const size_t first = (size_t)(r * kBlockTokens + slot0) * hkv;
          src[0] = ent[0] + first * KBt;
          src[1] = ent[1] + first * VBt;
          if (Tr::PACKED) {
            src[2] = ent[2] + first * MBt;
            src[3] = ent[3] + first * MBt;
          }
          nvc = nv;
        } else {
          atomicOr(err, ERR_ROW);
        }
      }
      const int cnt = min(32, u1 - ub);
      for (int i = 0; i < cnt; ++i) {
        const uint8_t* s0 = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src[0], i);
        const uint8_t* s1 = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src[1], i);
        const uint8_t* s2 = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src[2], i);
        const uint8_t* s3 = (const uint8_t*)__shfl_sync(0xffffffffu, (unsigned long long)src[3], i);
        const int nv = __shfl_sync(0xffffffffu, nvc, i);
        if (lane == 0 && !dead) {
          const int s = issued % NS;
          if (issued >= NS && !mbar_wait_bounded(&empty[s], ((issued / NS) & 1) ^ 1, err)) dead = true;
          if (!dead) {
            const uint32_t kbytes = (uint32_t)(nv * hkv * KBt), vbytes = (uint32_t)(nv * hkv * VBt);
            const uint32_t mbytes = (uint32_t)(nv * hkv * MBt);
            mbar_arrive_expect_tx(&full[s], kbytes + vbytes + 2 * mbytes);
            uint8_t* st = stages + (size_t)s * P.stage_bytes;
            if (nv > 0) {
              bulk_g2s_hint(st, s0, kbytes, &full[s], kv_policy);
              bulk_g2s_hint(st + off_v, s1, vbytes, &full[s], kv_policy);
              if (Tr::PACKED) {
                bulk_g2s_hint(st + off_km, s2, mbytes, &full[s], kv_policy);
                bulk_g2s_hint(st + off_vm, s3, mbytes, &full[s], kv_policy);
              }
            }
          }
        }
        dead = __shfl_sync(0xffffffffu, dead, 0);
        if (!dead) ++issued;  // count only stages whose barrier was armed
      }
    }
    // Drain: make sure none of this CTA's copies is still in flight at exit.
    if (lane == 0) {
      const int first = issued > NS ? issued - NS : 0;
      for (int n = first; n < issued; ++n) mbar_wait_bounded(&full[n % NS], (n / NS) & 1, err);
    }
    return;
  }

  // ------------------------------ consumers ---------------------------------
  const int h = warp;  // kv head
  const int tsub = lane / Tr::NCG, cg = lane % Tr::NCG;
  float q[G][Tr::DPL];
  float qsum[G][Tr::KP];
  float acc[G][Tr::DPL];
  float accO[G][Tr::VP];
  float m[G], lsum[G];
  float* qs = qscr + (size_t)warp * G * D;
  bool dead = false;

  int b = find_seq(UP, B, u0);
  int n = 0;
  for (int32_t u = u0; u < u1; ++u, ++n) {
    while (u >= UP[b + 1]) ++b;
    const bool seg_start = (u == u0) || (u == UP[b]);
    const bool seg_end = (u == u1 - 1) || (u == UP[b + 1] - 1);
    if (seg_start) {
      // Load q for (b, kv head h): G query heads, this lane's K dims.
      const uint16_t* qb = P.q + ((size_t)b * P.Hq + (size_t)h * G) * D;
      if constexpr (Tr::PACKED) {
        // q~ = H diag(s) q / sqrt(D), then scale * log2(e); FWHT in shared memory.
        for (int i = lane; i < G * D; i += 32) {
          const int d = i % D;
          qs[i] = __uint_as_float((uint32_t)qb[i] << 16) * P.signs[d];
        }
        __syncwarp();
        for (int hs = 1; hs < D; hs <<= 1) {
          for (int i = lane; i < G * D / 2; i += 32) {
            const int g = i / (D / 2), pi = i % (D / 2);
            const int a = g * D + (pi / hs) * 2 * hs + (pi % hs);
            const float x = qs[a], y = qs[a + hs];
            qs[a] = x + y;
            qs[a + hs] = x - y;
          }
          __syncwarp();
        }
        const float f = P.inv_sqrt_d * P.scale_log2;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int p = 0; p < Tr::KP; ++p) {
            const int d0 = (p * Tr::NCG + cg) * Tr::KEPP;
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < Tr::KEPP; ++e) {
              const float v = qs[g * D + d0 + e] * f;
              q[g][p * Tr::KEPP + e] = v;
              sum += v;
            }
            qsum[g][p] = sum;
          }
        __syncwarp();
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int p = 0; p < Tr::KP; ++p) {
            const int d0 = (p * Tr::NCG + cg) * Tr::KEPP;
            uint32_t w[Tr::KLU / 4];
            load_piece<Tr::KLU>(reinterpret_cast<const uint8_t*>(qb + (size_t)g * D + d0), w);
            float f[Tr::KEPP];
            piece_to_float<16, Tr::KLU>(w, f);
#pragma unroll
            for (int e = 0; e < Tr::KEPP; ++e) q[g][p * Tr::KEPP + e] = f[e] * P.scale_log2;
            qsum[g][p] = 0.f;
          }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        lsum[g] = 0.f;
#pragma unroll
        for (int i = 0; i < Tr::DPL; ++i) acc[g][i] = 0.f;
#pragma unroll
        for (int p = 0; p < Tr::VP; ++p) accO[g][p] = 0.f;
      }
    }

    const int32_t tok0 = (u - UP[b]) * T;
    const int nv = min(T, LS[b] - tok0);
    const int s = n % NS;
    if (!dead && !mbar_wait_bounded(&full[s], (n / NS) & 1, err)) dead = true;
    dead = __shfl_sync(0xffffffffu, dead, 0);
    if (!dead) {
      const uint8_t* st = stages + (size_t)s * P.stage_bytes;
      for (int i0 = 0; i0 < nv; i0 += Tr::TSUB) {
        const int t = i0 + tsub;
        const bool valid = t < nv;
        const int rowi = t * hkv + h;
        float sdot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sdot[g] = 0.f;
        if (valid) {
#pragma unroll
          for (int p = 0; p < Tr::KP; ++p) {
            const int c = p * Tr::NCG + cg;
            uint32_t w[Tr::KLU / 4];
            load_piece<Tr::KLU>(st + (size_t)rowi * KBt + c * Tr::KLU, w);
            float kf[Tr::KEPP];
            piece_to_float<Tr::KBITS, Tr::KLU>(w, kf);
            if constexpr (Tr::PACKED) {
              const float2 sm = *reinterpret_cast<const float2*>(st + off_km + (size_t)rowi * MBt +
                                                                  ((c * Tr::KEPP) / kGroup) * 8);
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float dsum = 0.f;
#pragma unroll
                for (int e = 0; e < Tr::KEPP; ++e) dsum = fmaf(q[g][p * Tr::KEPP + e], kf[e], dsum);
                sdot[g] = fmaf(sm.x, dsum, fmaf(sm.y, qsum[g][p], sdot[g]));
              }
            } else {
#pragma unroll
              for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < Tr::KEPP; ++e) sdot[g] = fmaf(q[g][p * Tr::KEPP + e], kf[e], sdot[g]);
            }
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int off = 1; off < Tr::NCG; off <<= 1) sdot[g] += __shfl_xor_sync(0xffffffffu, sdot[g], off);
          if (!valid) sdot[g] = -INFINITY;
        }
        // Online softmax over this sub-step's tokens (warp-uniform running max).
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mx = sdot[g];
#pragma unroll
          for (int off = Tr::NCG; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          if (mx > m[g]) {
            const float alpha = exp2f(m[g] - mx);
            lsum[g] *= alpha;
#pragma unroll
            for (int i = 0; i < Tr::DPL; ++i) acc[g][i] *= alpha;
#pragma unroll
            for (int p = 0; p < Tr::VP; ++p) accO[g][p] *= alpha;
            m[g] = mx;
          }
          sdot[g] = exp2f(sdot[g] - m[g]);  // probability weight (0 for invalid)
          lsum[g] += sdot[g];
        }
        if (valid) {
#pragma unroll
          for (int p = 0; p < Tr::VP; ++p) {
            const int c = p * Tr::NCG + cg;
            uint32_t w[Tr::VLU / 4];
            load_piece<Tr::VLU>(st + off_v + (size_t)rowi * VBt + c * Tr::VLU, w);
            float vf[Tr::VEPP];
            piece_to_float<Tr::VBITS, Tr::VLU>(w, vf);
            if constexpr (Tr::PACKED) {
              const float2 sm = *reinterpret_cast<const float2*>(st + off_vm + (size_t)rowi * MBt +
                                                                  ((c * Tr::VEPP) / kGroup) * 8);
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const float ps = sdot[g] * sm.x;
#pragma unroll
                for (int e = 0; e < Tr::VEPP; ++e) acc[g][p * Tr::VEPP + e] = fmaf(ps, vf[e], acc[g][p * Tr::VEPP + e]);
                accO[g][p] = fmaf(sdot[g], sm.y, accO[g][p]);
              }
            } else {
#pragma unroll
              for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < Tr::VEPP; ++e) acc[g][p * Tr::VEPP + e] = fmaf(sdot[g], vf[e], acc[g][p * Tr::VEPP + e]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    if (seg_end) {
      // Merge the token sub-groups of the warp (lanes with equal cg).
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int off = Tr::NCG; off < 32; off <<= 1) {
          lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], off);
#pragma unroll
          for (int i = 0; i < Tr::DPL; ++i) acc[g][i] += __shfl_xor_sync(0xffffffffu, acc[g][i], off);
#pragma unroll
          for (int p = 0; p < Tr::VP; ++p) accO[g][p] += __shfl_xor_sync(0xffffffffu, accO[g][p], off);
        }
        if constexpr (Tr::PACKED) {
#pragma unroll
          for (int p = 0; p < Tr::VP; ++p)
#pragma unroll
            for (int e = 0; e < Tr::VEPP; ++e) acc[g][p * Tr::VEPP + e] += accO[g][p];
        }
      }
      const int32_t c_lo = UP[b] / C, c_hi = (UP[b + 1] - 1) / C;
      if (c_lo == c_hi) {
        // The whole sequence is in this CTA: normalise and store.
        if (tsub == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float inv = 1.0f / lsum[g];
            uint16_t* o = P.out + ((size_t)b * P.Hq + h * G + g) * D;
#pragma unroll
            for (int p = 0; p < Tr::VP; ++p) {
              const int d0 = (p * Tr::NCG + cg) * Tr::VEPP;
#pragma unroll
              for (int e = 0; e < Tr::VEPP; ++e) o[d0 + e] = f2bf(acc[g][p * Tr::VEPP + e] * inv);
            }
          }
        }
      } else {
        if (tsub == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float* pp = partial_ptr(P, D, (size_t)blockIdx.x, b, (size_t)h * G + g);
            if (cg == 0) {
              pp[0] = m[g];
              pp[1] = lsum[g];
            }
#pragma unroll
            for (int p = 0; p < Tr::VP; ++p) {
              const int d0 = (p * Tr::NCG + cg) * Tr::VEPP;
#pragma unroll
              for (int e = 0; e < Tr::VEPP; ++e) pp[kPartialHeader + d0 + e] = acc[g][p * Tr::VEPP + e];
            }
          }
        }
      }
    }
  }
}

// Shared-memory plan: T tokens per stage, NS stages (see plan_decode).
template <int FMT, int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a) {
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
  using Tr = DecodeTraits<FMT, D, G>;
  P.stage_bytes = P.T * a.lv.hkv * (Tr::KB + Tr::VB + 2 * Tr::MB);
  auto kern = decode_kernel<FMT, D, G>;
  // Raise the dynamic shared-memory limit once per instantiation (not per call, so
  // that launches can be captured into CUDA graphs without runtime attribute calls).
  static size_t smem_set = 0;
  if (a.smem_bytes > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    smem_set = 232448;
  }
  cudaError_t e = launch_with_pdl(kern, a.grid, (a.lv.hkv + 1) * 32, a.smem_bytes, a.stream, P);
  if (e != cudaSuccess) return e;
  return launch_combine<D>(P, a.grid, a.stream);
}

template <int FMT>
cudaError_t launch_decode_fmt(const DecodeArgs& a) {
#define PKV_CASE(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_decode_t<FMT, DD, GG>(a);
  PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
  PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv
