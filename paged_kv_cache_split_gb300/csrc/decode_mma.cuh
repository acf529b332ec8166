// decode_mma.cuh — native-bf16 paged decode attention on tensor-core tiles.
//
// Work partition: units of T tokens x all kv heads, split over one CTA per SM
// evenly in cost (Split, decode_common.cuh: a sequence start counts as part of a
// unit); a producer warp plus one consumer warp per kv head; split-K partials merged
// by the chained combine kernel (decode_common.cuh).  For bf16 K/V two choices cut
// the consumer's issue slots by several times against CUDA-core dot products:
//
//  * Staging: one 3-D tensor copy per 16 tokens and tensor (K, V) moves those
//    tokens' rows of all kv heads; they land as 128-byte-wide boxes [column
//    block][16 tokens][128 bytes] with the 128-byte swizzle (16-byte chunk c of
//    token row r at chunk c ^ (r & 7)), so ldmatrix reads of 8 tokens x 16 bytes
//    are conflict-free.  The producer's lane i issues every copy of unit i of a
//    batch of 32 units, after the tensor-map acquire fences it ran when it read
//    the batch.
//  * Math on mma.sync.m16n8k16 (bf16 in, fp32 accumulate):
//      S  = Q K^T  with M = the G query heads of the kv head (padded to 16),
//                  N = 8 tokens, K = 16 dims; Q is an A fragment held in registers
//                  for the whole sequence, K comes from ldmatrix;
//      O^T = V^T P^T with M = 16 output dims, N = the query heads, K = 16 tokens;
//                  V^T comes from ldmatrix.trans, and P^T's B fragment is exactly
//                  the accumulator fragment of S for those 16 tokens, so the
//                  probabilities never leave registers.
//    Logits are scaled by scale*log2(e) in fp32 after the QK product; the online
//    softmax runs in base 2 on the accumulator fragments; P is rounded to bf16 for
//    the PV product while the denominator sums the fp32 probabilities.
#pragma once

#include <type_traits>

#include "decode_common.cuh"

namespace pkv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A B for one m16n8k16 bf16 tile (A row-major 16x16, B col-major 16x8).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// NQ > 1 (chunked prefill): a virtual sequence carries NQ consecutive queries of one
// sequence's chunk, and the S tile's rows are (query, head) pairs, query-major: row
// r is query r / G and head r % G of the kv head.  Up to 8 rows ride in the rows
// decode leaves empty; with more (up to 16, head dims up to 128) rows 8..15 get a
// second softmax state and a second PV product per lane.  Query j of NQ sees the
// sequence's first L - (NQ - 1 - j) tokens (causal); P.Hq counts the NQ queries' heads.
template <int D, int G, int NQ = 1>
__global__ void __launch_bounds__(kMaxThreads, 1) decode_bf16_mma_kernel(const DecodeParams P) {
  static_assert(G >= 1 && G <= 8 && D % 16 == 0, "geometry");
  static_assert(NQ >= 1 && NQ * G <= 16 && (NQ * G <= 8 || D <= 128), "query rows of one kv head fit the tile");
  constexpr int R = NQ * G;      // rows in use
  constexpr bool TWO = R > 8;    // rows 8..15 in use
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = P.lv.hkv;
  const int NC = hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = P.T, NS = P.NS, B = P.B;
  int32_t* err = P.lv.err;
  const int ROW = hkv * D * 2;  // one token, all kv heads, in the slab (a multiple of 128 bytes)
  const int NX = ROW >> 7;      // 128-byte column blocks of a row

  // Stages start on a 1024-byte boundary (the 128-byte swizzle repeats every 1 KB).
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + (size_t)NS * P.stage_bytes);
  uint64_t* empty = full + NS;
  const uint8_t** tab = reinterpret_cast<const uint8_t**>(empty + NS);  // [kSmemTableEntries]
  int32_t* UP = reinterpret_cast<int32_t*>(tab + kSmemTableEntries);
  int32_t* LS = UP + (B + 1);
  uint64_t* tok = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(LS + B) + 7) & ~uintptr_t(7));

  uint64_t* spec = tok + 2;  // [kSpecUnits]
  const int offV = T * ROW;      // K region [T/16][NX][16][128], then V region
  const int offQ = 2 * T * ROW;  // q of the sequence, when the unit starts one
  const int QB = P.Hq * D * 2;
  // Arms `bar` with a unit's bytes and issues its copies.  A whole unit is always
  // copied (T tokens stay inside the block); tokens past the context are masked by
  // a zero probability.  A unit that starts a CTA's segment of a sequence also
  // brings that sequence's q.
  auto issue = [&](uint64_t* bar, uint8_t* st, const uint8_t* map, int y0, int ok, const uint8_t* qsrc) {
    const uint64_t kv_policy = P.kv_reuse ? l2_policy_evict_normal() : l2_policy_evict_first();
    mbar_arrive_expect_tx(bar, (ok ? (uint32_t)(2 * T * ROW) : 0u) + (qsrc ? (uint32_t)QB : 0u));
    if (qsrc) bulk_g2s(st + offQ, qsrc, (uint32_t)QB, bar);
    if (ok) {
      for (int cy = 0; cy < T / 16; ++cy) {
        tma_load_3d(st + cy * 16 * ROW, map, 0, y0 + 16 * cy, 0, bar, kv_policy);
        tma_load_3d(st + offV + cy * 16 * ROW, map + 128, 0, y0 + 16 * cy, 0, bar, kv_policy);
      }
    }
  };

  const FirstGuess fg = decode_prologue<D, true>(P, full, empty, NC, NC, UP, LS, tab, tok, spec, stages, issue);
  __syncthreads();
  const int32_t U = UP[B];
  const Split sp = make_split(U, B, (int)gridDim.x, P.seg_cost);  // this CTA's units: [u0, u1)
  zero_empty_sequences<D>(P, LS);
  const int32_t u0 = U == 0 ? 0 : sp.first_unit(UP, B, blockIdx.x);
  const int32_t u1 = U == 0 ? 0 : sp.first_unit(UP, B, (int64_t)blockIdx.x + 1);
  if (U == 0 || u0 >= u1) {
    if (warp == NC) finish_spec(fg, spec, err);
    return;
  }

  if (warp == NC) {
    // ----------------------------- producer ---------------------------------
    run_producer<D, 1>(P, 0, u0, u1, UP, tab, full, empty, tok, stages, fg, spec, issue);
    return;
  }

  // ------------------------------ consumers ---------------------------------
  const int h = warp;
  const int g = lane >> 2, t = lane & 3;
  // q head (within the virtual sequence's P.Hq) of row r
  auto qhead = [&](int r) -> size_t {
    if constexpr (NQ == 1) return (size_t)h * G + r;
    else return (size_t)(r / G) * (size_t)(P.Hq / NQ) + (size_t)h * G + (size_t)(r % G);
  };
  // ldmatrix row owned by this lane: matrix mi = lane/8, row ri = lane%8 covers
  // token 8*(mi/2)+ri and dims 8*(mi%2) .. +7 of the current 16-token x 16-dim tile.
  const int ld_tok = 8 * ((lane >> 3) >> 1) + (lane & 7);
  const int ld_dim = 8 * ((lane >> 3) & 1);
  // Its address in a 16-token box row: the head's first column block, token row
  // ld_tok; the 16-dim tile kk sits in column block kk / 4 at logical chunk
  // 2 (kk % 4) + ld_dim / 8, stored at that chunk XOR (ld_tok % 8).
  const uint32_t ld_base = (uint32_t)(((h * D * 2) >> 7) * 2048 + ld_tok * 128);
  uint32_t ld_chunk[4];
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) ld_chunk[q4] = (uint32_t)(((2 * q4 + (ld_dim >> 3)) ^ (ld_tok & 7)) << 4);
  uint32_t qa[D / 16][2];
  float o[D / 16][4];
  float m_run = -INFINITY, l_run = 0.f;
  uint32_t qa8[D / 16][2];  // rows g + 8 (TWO only)
  float o8[D / 16][4];
  float m_run8 = -INFINITY, l_run8 = 0.f;
  bool dead = false;
  const uint32_t smem_base = smem_u32(stages);

  int b = find_seq(UP, B, u0);
  int s = 0;           // stage of unit u
  uint32_t phase = 0;  // parity of its full barrier
  for (int32_t u = u0; u < u1; ++u, s = (s + 1 == NS) ? 0 : s + 1, phase ^= (s == 0)) {
    while (u >= UP[b + 1]) ++b;
    const bool seg_start = (u == u0) || (u == UP[b]);
    const bool seg_end = (u == u1 - 1) || (u == UP[b + 1] - 1);
    if (seg_start) {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
      if constexpr (TWO) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) o8[mt][i] = 0.f;
        m_run8 = -INFINITY;
        l_run8 = 0.f;
      }
    }

    const int32_t tok0 = (u - UP[b]) * T;
    const int nv = min(T, LS[b] - tok0);
    // tokens of this unit visible to the lane's row (its query's causal limit)
    const int nvr = NQ == 1 ? nv : min(T, LS[b] - tok0 - (NQ - 1 - (g < R ? g / G : NQ - 1)));
    const int nvr8 = TWO ? min(T, LS[b] - tok0 - (NQ - 1 - (g + 8 < R ? (g + 8) / G : NQ - 1))) : 0;
    if (!dead && !mbar_wait_bounded(&full[s], phase, err)) dead = true;
    dead = __shfl_sync(0xffffffffu, dead, 0);
    if (!dead && seg_start) {
      // A fragments of Q (rows = query heads of kv head h; rows >= G are zero),
      // from the copy of q that arrived with this stage.
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(stages + (size_t)s * P.stage_bytes + offQ +
                                                               qhead(g < R ? g : 0) * D * 2);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        qa[kk][0] = g < R ? qrow[(16 * kk + 2 * t) / 2] : 0u;
        qa[kk][1] = g < R ? qrow[(16 * kk + 2 * t + 8) / 2] : 0u;
      }
      if constexpr (TWO) {
        const uint32_t* qrow8 = reinterpret_cast<const uint32_t*>(stages + (size_t)s * P.stage_bytes + offQ +
                                                                  qhead(g + 8 < R ? g + 8 : 0) * D * 2);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          qa8[kk][0] = g + 8 < R ? qrow8[(16 * kk + 2 * t) / 2] : 0u;
          qa8[kk][1] = g + 8 < R ? qrow8[(16 * kk + 2 * t + 8) / 2] : 0u;
        }
      }
    }
    if (!dead) {
      const uint32_t kst = smem_base + (uint32_t)(s * P.stage_bytes);
      const uint32_t vst = kst + (uint32_t)offV;
      for (int kc = 0; kc * 16 < nv; ++kc) {
        // ---- S = Q K^T for 16 tokens (two n-tiles of 8) ----
        float sacc[2][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[0][i] = sacc[1][i] = 0.f;
        const uint32_t kaddr = kst + (uint32_t)(kc * NX * 2048) + ld_base;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kaddr + (kk >> 2) * 2048 + ld_chunk[kk & 3], r0, r1, r2, r3);
          if constexpr (TWO) {
            mma_bf16_16816(sacc[0], qa[kk][0], qa8[kk][0], qa[kk][1], qa8[kk][1], r0, r1);
            mma_bf16_16816(sacc[1], qa[kk][0], qa8[kk][0], qa[kk][1], qa8[kk][1], r2, r3);
          } else {
            mma_bf16_16816(sacc[0], qa[kk][0], 0u, qa[kk][1], 0u, r0, r1);
            mma_bf16_16816(sacc[1], qa[kk][0], 0u, qa[kk][1], 0u, r2, r3);
          }
        }
        // ---- online softmax for head g (row g), tokens 2t, 2t+1, 8+2t, 9+2t ----
        const int tb = kc * 16 + 2 * t;
        float x0 = tb < nvr ? sacc[0][0] * P.scale_log2 : -INFINITY;
        float x1 = tb + 1 < nvr ? sacc[0][1] * P.scale_log2 : -INFINITY;
        float x2 = tb + 8 < nvr ? sacc[1][0] * P.scale_log2 : -INFINITY;
        float x3 = tb + 9 < nvr ? sacc[1][1] * P.scale_log2 : -INFINITY;
        float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const bool grow = mx > m_run;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? exp2f(m_run - mx) : 1.0f;
          if (grow) m_run = mx;
          l_run *= alpha;
          // O^T columns of this lane are heads 2t and 2t+1, whose statistics live in
          // lanes 8t and 8t+4.
          const float ae = __shfl_sync(0xffffffffu, alpha, 8 * t);
          const float ao = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            o[mt][0] *= ae;
            o[mt][2] *= ae;
            o[mt][1] *= ao;
            o[mt][3] *= ao;
          }
        }
        float p0 = exp2f(x0 - m_run), p1 = exp2f(x1 - m_run);
        float p2 = exp2f(x2 - m_run), p3 = exp2f(x3 - m_run);
        if constexpr (NQ > 1) {
          // a row with no visible token yet in this segment keeps m_run = -inf
          if (m_run == -INFINITY) p0 = p1 = p2 = p3 = 0.f;
        }
        l_run += (p0 + p1) + (p2 + p3);
        const uint32_t pb0 = pack_bf16x2(p0, p1), pb1 = pack_bf16x2(p2, p3);
        uint32_t pb2 = 0u, pb3 = 0u;
        if constexpr (TWO) {
          // ---- the same for rows g + 8 (fragment elements 2 and 3) ----
          const float y0 = tb < nvr8 ? sacc[0][2] * P.scale_log2 : -INFINITY;
          const float y1 = tb + 1 < nvr8 ? sacc[0][3] * P.scale_log2 : -INFINITY;
          const float y2 = tb + 8 < nvr8 ? sacc[1][2] * P.scale_log2 : -INFINITY;
          const float y3 = tb + 9 < nvr8 ? sacc[1][3] * P.scale_log2 : -INFINITY;
          float my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
          my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
          my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
          const bool grow8 = my > m_run8;
          if (__any_sync(0xffffffffu, grow8)) {
            const float alpha = grow8 ? exp2f(m_run8 - my) : 1.0f;
            if (grow8) m_run8 = my;
            l_run8 *= alpha;
            const float ae = __shfl_sync(0xffffffffu, alpha, 8 * t);
            const float ao = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              o8[mt][0] *= ae;
              o8[mt][2] *= ae;
              o8[mt][1] *= ao;
              o8[mt][3] *= ao;
            }
          }
          float q0 = exp2f(y0 - m_run8), q1 = exp2f(y1 - m_run8);
          float q2 = exp2f(y2 - m_run8), q3 = exp2f(y3 - m_run8);
          if (m_run8 == -INFINITY) q0 = q1 = q2 = q3 = 0.f;
          l_run8 += (q0 + q1) + (q2 + q3);
          pb2 = pack_bf16x2(q0, q1);
          pb3 = pack_bf16x2(q2, q3);
        }
        // ---- O^T += V^T P^T over these 16 tokens ----
        // The lane's A fragments hold V of tokens tb, tb + 1 (a0, a1) and tb + 8,
        // tb + 9 (a2, a3).  In a chunk that ends past the context those tokens' slots
        // may hold stale bytes (an earlier owner of the row, an imported record): their
        // probability is 0, but 0 times a non-finite value is not, so their V halves
        // are replaced by zeros.
        const uint32_t vaddr = vst + (uint32_t)(kc * NX * 2048) + ld_base;
        auto pv_tile = [&](auto masked_c) {
          constexpr bool MASKED = decltype(masked_c)::value;
          uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
          if constexpr (MASKED) {
            m01 = (tb < nv ? 0x0000ffffu : 0u) | (tb + 1 < nv ? 0xffff0000u : 0u);
            m89 = (tb + 8 < nv ? 0x0000ffffu : 0u) | (tb + 9 < nv ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vaddr + (mt >> 2) * 2048 + ld_chunk[mt & 3], a0, a1, a2, a3);
            if constexpr (MASKED) {
              a0 &= m01;
              a1 &= m01;
              a2 &= m89;
              a3 &= m89;
            }
            mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            if constexpr (TWO) mma_bf16_16816(o8[mt], a0, a1, a2, a3, pb2, pb3);
          }
        };
        if (kc * 16 + 16 > nv)
          pv_tile(std::true_type{});
        else
          pv_tile(std::false_type{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    if (seg_end) {
      // rows rb + 2t and rb + 2t + 1 of the tile (this lane's O^T columns)
      auto finish = [&](const float (&ov)[D / 16][4], float mv, float lv, const int rb) {
        lv += __shfl_xor_sync(0xffffffffu, lv, 1);
        lv += __shfl_xor_sync(0xffffffffu, lv, 2);
        const float me = __shfl_sync(0xffffffffu, mv, 8 * t), mo = __shfl_sync(0xffffffffu, mv, 8 * t + 4);
        const float le = __shfl_sync(0xffffffffu, lv, 8 * t), lo = __shfl_sync(0xffffffffu, lv, 8 * t + 4);
        const int he = rb + 2 * t, ho = rb + 2 * t + 1;
        const int32_t c_lo = sp.c_lo(UP, b), c_hi = sp.c_hi(UP, b);
        if (c_lo == c_hi) {
          const float ie = 1.0f / le, io = 1.0f / lo;
          uint16_t* oe = P.out + ((size_t)b * P.Hq + qhead(he < R ? he : 0)) * D;
          uint16_t* oo = P.out + ((size_t)b * P.Hq + qhead(ho < R ? ho : 0)) * D;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            if (he < R) {
              oe[16 * mt + g] = f2bf(ov[mt][0] * ie);
              oe[16 * mt + g + 8] = f2bf(ov[mt][2] * ie);
            }
            if (ho < R) {
              oo[16 * mt + g] = f2bf(ov[mt][1] * io);
              oo[16 * mt + g + 8] = f2bf(ov[mt][3] * io);
            }
          }
        } else {
          float* pe = partial_ptr(P, D, (size_t)blockIdx.x, b, qhead(he < R ? he : 0));
          float* po = partial_ptr(P, D, (size_t)blockIdx.x, b, qhead(ho < R ? ho : 0));
          if (he < R) {
            if (g == 0) {
              pe[0] = me;
              pe[1] = le;
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              pe[kPartialHeader + 16 * mt + g] = ov[mt][0];
              pe[kPartialHeader + 16 * mt + g + 8] = ov[mt][2];
            }
          }
          if (ho < R) {
            if (g == 0) {
              po[0] = mo;
              po[1] = lo;
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              po[kPartialHeader + 16 * mt + g] = ov[mt][1];
              po[kPartialHeader + 16 * mt + g + 8] = ov[mt][3];
            }
          }
        }
      };
      finish(o, m_run, l_run, 0);
      if constexpr (TWO) finish(o8, m_run8, l_run8, 8);
    }
  }
}

template <int D, int G, int NQ = 1>
cudaError_t launch_decode_bf16_mma_t(const DecodeArgs& a) {
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
  P.kv_reuse = a.kv_reuse;
  P.nq = a.nq;
  P.seg_cost = a.seg_cost;
  P.T = a.tokens_per_stage;
  P.NS = a.n_stages;
  P.stage_bytes = 2 * P.T * (a.lv.hkv * D * 2) + ((a.Hq * D * 2 + 1023) & ~1023);
  auto kern = decode_bf16_mma_kernel<D, G, NQ>;
  {
    static unsigned long long smem_done = 0;  // this kernel (one per template instantiation)
    cudaError_t e = allow_max_dynamic_smem(kern, smem_done);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_with_pdl(kern, a.grid, (a.lv.hkv + 1) * 32, a.smem_bytes, a.stream, P);
  if (e != cudaSuccess) return e;
  return launch_combine<D, 2>(P, a.grid, a.nq, a.stream);
}


}  // namespace pkv
