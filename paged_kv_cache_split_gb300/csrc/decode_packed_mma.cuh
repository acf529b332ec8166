// decode_packed_mma.cuh — paged decode attention over packed K4/V4, K8/V4, K8/V8
// pages on tensor-core tiles (fp16 in, fp32 accumulate).
//
// Work partition and split-K epilogue are those of the bf16 kernel
// (decode_mma.cuh): units of T tokens x all kv heads split over one CTA per SM,
// evenly in cost (Split), two producer warps and one consumer warp per kv head (two
// with the dim split).
// Staging uses TMA tensor copies: each stored tensor of a slab (K codes, V codes, K
// meta, V meta) has a tensor map over [tokens][all-heads row bytes]; a stage holds
// T tokens of each tensor as boxes of 16 tokens x W bytes (W = 128, 64, 32 or 16,
// the largest dividing the row), written with the W-byte shared-memory swizzle (16-byte chunk c of box row r
// lands at chunk c ^ f(r)), so 16-byte chunks of 8 consecutive tokens sit in
// distinct banks and are read with ldmatrix.  q comes with the first unit of a
// sequence (one bulk copy; with 16 tile rows the consumers read it from global
// memory instead, QG).  The packed pages are consumed directly, never
// expanded in memory (mlx-swift-lm PR #142, Summary: direct attention on packed
// pages):
//
//  * q is rotated into K's signed Hadamard basis (q~ = H diag(s) q / sqrt(D), a fast
//    Walsh-Hadamard transform at each segment start, stored as fp16 in place of q in
//    the stage, or in a per-head scratch with QG) and kept as fp16 A fragments
//    (rows = the tile's (query, head) rows, rows 8..15 in the fragment's upper half
//    when more than 8 are in use; unused rows zero).
//  * Codes enter the tensor cores as fp16 subnormals: the bit pattern of a code c
//    (4 or 8 bits) in the low mantissa bits is the exact value c * 2^-24, so a code
//    becomes an operand with one AND (4-bit) or one byte permute (8-bit).  A 4-bit
//    code in the high nibble of its byte is taken as 16c * 2^-24 and the factor 16
//    is removed on the other operand (q / 16) or on the output (V).
//  * QK, one affine group of 32 dims at a time: the group's product
//    C = sum_k q~_k c_k * 2^-24, and the stored (scale s, offset o) of the token
//    and group fold in on the accumulator fragment:
//        logit = 2^24 * sum_groups [ s C + o * 2^-24 * sum(q~ over the group) ].
//    A consistent permutation of the 32 dims of a group is used on both operands
//    (the dot product does not depend on the order), chosen so that each lane's
//    B fragment comes from one 32-bit word of codes (an ldmatrix row).
//  * PV as O^T = V^T (P S)^T + (P O_v): the A operand holds raw V codes of two
//    tokens per register (ldmatrix.trans of the code rows), the B operand is
//    p_t * s_t (fp16) formed from the S accumulator fragments and the tokens'
//    scales, and the offsets add sum_t p_t o_t per head and group in fp32.  Each
//    16-row M tile covers 16 dims of one group; the order of dims inside a group
//    follows the ldmatrix.trans fragment (a lane's two dims per token come from one
//    half-word of codes) and the output store undoes the permutation.
//
// fp16 range.  The stored scales and offsets are FP32 (mlx-swift-lm PR #142,
// Summary), so q, K and V may have any magnitude; only the two operands rounded to
// fp16 need care, and both are kept in range by powers of two that are undone in
// fp32 (exact, so no rounding is added):
//  * q~ of each tile row is multiplied by 2^e, with e chosen once per sequence
//    segment so that the row's largest |q~| lies in [2^14, 2^15); the logits' fp32
//    scale carries 2^-e.
//  * p s uses an exponent f shared by all of a warp's groups: the softmax works
//    with the reference max m - f, so every probability (and with it the running
//    denominator and both accumulators) carries 2^f.  Before the products of a
//    chunk's groups are formed, their V scales are compared with 2^(15 - f) (p 2^f
//    never exceeds 2^f): the first nonzero scale of a segment, or one at or above
//    that bound, sets f from the chunk's largest scale s so that s 2^f lies in
//    [2^4, 2^5), and the state is multiplied by the matching power of two.  Partial
//    records store the state with 2^f removed.
// A token past the context (in the last unit of a sequence) gets probability 0
// and its V scale and offset are replaced by 0 before they meet it, so stale
// non-finite bytes in unused slots of a block never reach the output.
#pragma once

#include <cuda_fp16.h>

#include <type_traits>

#include "decode_common.cuh"

namespace pkv {

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t r) {
  return __half22float2(*reinterpret_cast<const __half2*>(&r));
}

template <int FMT, int D, int GS = kGroup>
struct PackedTraits {
  static constexpr int KBITS = FMT == PKV_FMT_K4V4 ? 4 : 8;
  static constexpr int VBITS = FMT == PKV_FMT_K8V8 ? 8 : 4;
  static constexpr int KB = D * KBITS / 8;   // K code bytes per (token, head)
  static constexpr int VB = D * VBITS / 8;
  static constexpr int NG = D / 32;          // 32-dim groups per row (the unit of the fold)
  static constexpr int SPP = GS / 32;        // 32-dim groups sharing one (scale, offset) pair
  static constexpr int MB = (D / GS) * 8;    // (scale, offset) bytes per (token, head)
  static constexpr int NKC = KB / 16;        // 16-byte chunks per (token, head)
  static constexpr int NVC = VB / 16;
  static constexpr int NMC = MB / 16;        // two pairs per chunk
  static constexpr int SPC = 2 * SPP;        // 32-dim groups per metadata chunk
  static_assert(GS == 32 || GS == 64, "group size");
  static_assert(MB % 16 == 0, "whole metadata chunks per (token, head)");
};

// B fragments of K for one group and one token (this lane's token of the n-tile),
// as fp16 subnormals: k-step ks in {0,1} of the group gets (b[ks][0], b[ks][1]).
// 4-bit: word t of the group holds elements 8t..8t+7 (element n in bits 4n..4n+3).
__device__ __forceinline__ void k_group_frags4(uint32_t w, uint32_t (&b)[2][2]) {
  const uint32_t w8 = w >> 8;
  b[0][0] = w & 0x000F000Fu;   // elements 0, 4      : c
  b[0][1] = w & 0x00F000F0u;   // elements 1, 5      : 16 c
  b[1][0] = w8 & 0x000F000Fu;  // elements 2, 6
  b[1][1] = w8 & 0x00F000F0u;  // elements 3, 7      : 16 c
}

// 8-bit: k-step ks uses word t of the group's chunk ks: elements 16 ks + 4t + j.
__device__ __forceinline__ void k_group_frags8(uint32_t w0, uint32_t w1, uint32_t (&b)[2][2]) {
  b[0][0] = __byte_perm(w0, 0u, 0x4140);  // (c0, c1)
  b[0][1] = __byte_perm(w0, 0u, 0x4342);  // (c2, c3)
  b[1][0] = __byte_perm(w1, 0u, 0x4140);
  b[1][1] = __byte_perm(w1, 0u, 0x4342);
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

// Output dim of M tile mi of group grp, row half hh (0: row g, 1: row g+8).  The
// A fragment of a 4-bit group comes from half-word g of its 16-byte chunk (dims
// 4g..4g+3 of the group): tile 0 takes the low nibbles of its bytes (dims 4g, 4g+2),
// tile 1 the high nibbles (dims 4g+1, 4g+3, read as 16c).  An 8-bit group spans two
// chunks, one per tile; half-word g holds dims 2g and 2g+1 of the chunk.
template <int VBITS>
__device__ __forceinline__ int v_out_dim(int grp, int mi, int hh, int g) {
  return VBITS == 4 ? 32 * grp + 4 * g + mi + 2 * hh : 32 * grp + 16 * mi + 2 * g + hh;
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

// 2^n as a float, for n in [-126, 127].
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

// floor(log2 x) of a positive float, read from its exponent field (fp32 subnormals
// give -127).
__device__ __forceinline__ int exponent_of(float x) { return (int)((__float_as_uint(x) >> 23) & 0xffu) - 127; }

// The p s exponent for a largest V scale smax > 0: smax 2^f lands in [2^4, 2^5).
__device__ __forceinline__ int v_exponent_for(float smax) {
  const int f = 4 - exponent_of(smax);
  return f < -40 ? -40 : (f > 80 ? 80 : f);
}


// Register split (RS): the block is laid out in warpgroups, ceil(Hkv / 4) of consumer
// warps and one whose first two warps are the producers.  At the role branch the producer warpgroup
// gives registers back (setmaxnreg.dec to kProdRegs) and the consumer warpgroups
// take them (setmaxnreg.inc to kConsRegs): per scheduler, two consumer warps and one
// producer-group warp fit in the three warps' launch allocation (2 x 224 + 56 = 3 x
// 168).  The launcher checks the kernel's launch register count before choosing it.
constexpr int kRsThreads = 384;
constexpr int kConsRegs = 224;
constexpr int kProdRegs = 56;

// W128: every stored tensor's all-heads row is a multiple of 128 bytes, so every box
// is 128 bytes wide; then every shared-memory address below is a per-lane constant
// plus a per-chunk uniform offset plus an immediate.
// DS (dim split, D = 256 with at most 4 kv heads): two consumer warps per kv head,
// each owning half of the head's affine groups (K dims for the logits, V dims for
// the output).  Per 16-token chunk the two halves of every logit are exchanged
// through shared memory and added in a fixed order, so both warps run the same
// softmax; each keeps the state of its own dims.
// NQ > 1 (chunked prefill): the S tile's rows are (query, head) pairs of NQ
// consecutive queries of one sequence, query-major (row r: query r / G, head r % G
// of the kv head; NQ x G <= 8), each masked at its query's causal limit; P.Hq counts
// the NQ queries' heads.
template <int FMT, int D, int G, bool W128, bool RS, bool DS, int GS, int NQ = 1>
__global__ void __launch_bounds__(RS ? kRsThreads : kMaxThreads, 1) decode_packed_mma_kernel(const DecodeParams P) {
  using Tr = PackedTraits<FMT, D, GS>;
  static_assert(G >= 1 && G <= 8 && D % 32 == 0, "geometry");
  static_assert(!DS || (W128 && D == 256), "dim split: 128-byte boxes, D = 256");
  constexpr int NG = Tr::NG;
  extern __shared__ __align__(128) uint8_t smem[];
  const int hkv = P.lv.hkv;
  const int NC = DS ? 2 * hkv : hkv;  // consumer warps
  constexpr int RW = NQ * G;          // tile rows in use
  constexpr bool TWO = RW > 8;        // rows 8..15 in use
  // QG: the consumers read q from global memory at each segment start (the producer
  // prefetches it into L2 with the segment's first unit) and rotate it into a per-head
  // scratch, so the stages carry no q region: used with 16 rows, whose q (16 rows x D
  // per kv head) would otherwise take a large share of every stage.
  constexpr bool QG = TWO;
  constexpr int QS = D + 8;  // QG scratch row stride (halves): rows 16 bytes apart in banks
  static_assert(RW <= 16 && (!TWO || (D <= 128 && !DS)), "query rows of one kv head fit the tile");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NCW = (NC + 3) >> 2;                // consumer warpgroups (register split)
  const int PW = RS ? 4 * NCW : NC;             // the first of the two producer warps
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
  const int QB = QG ? 0 : P.Hq * D * 2;  // q bytes a stage receives
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
  // the q~ exponent of each tile row, per kv head
  int32_t* qes = reinterpret_cast<int32_t*>((reinterpret_cast<uintptr_t>(LS + B) + 15) & ~uintptr_t(15));
  // QG: q~ of each kv head's RW rows (fp16, row stride QS)
  uint16_t* qg_scr = reinterpret_cast<uint16_t*>(qes + (size_t)hkv * 16);
  // dim split: per kv head, each half's partial logits (up to 32 tokens) of the last two exchanges, and
  // one mbarrier per kv head that pairs the two warps (bounded waits)
  float4* xbuf = reinterpret_cast<float4*>(qg_scr + (QG ? (size_t)hkv * RW * QS : 0));
  uint64_t* pbar = reinterpret_cast<uint64_t*>(xbuf + (size_t)hkv * 2 * 2 * 2 * 32);
  // the producers' issue token, one barrier per batch parity (after the dim-split
  // buffers, or where they would start)
  uint64_t* tok = DS ? pbar + hkv : reinterpret_cast<uint64_t*>(xbuf);

  uint64_t* spec = tok + 2;  // [kSpecUnits]

  // Producers: one 3-D tensor copy per 16 tokens and stored tensor, plus q when the
  // unit starts a CTA's segment of a sequence, all counted on barrier `bar`.
  auto issue = [&](uint64_t* bar, uint8_t* st, const uint8_t* map, int y0, int ok, const uint8_t* qsrc) {
    const uint64_t kv_policy = P.kv_reuse ? l2_policy_evict_normal() : l2_policy_evict_first();
    mbar_arrive_expect_tx(bar, (ok ? (uint32_t)(T * (KR + VR + 2 * MR)) : 0u) + (qsrc ? (uint32_t)QB : 0u));
    if (qsrc) {
      if constexpr (QG) bulk_prefetch_l2(qsrc, (uint32_t)(P.Hq * D * 2));
      else bulk_g2s(st + offQ, qsrc, (uint32_t)QB, bar);
    }
    if (ok) {
      for (int cy = 0; cy < T / 16; ++cy)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tma_load_3d(st + zr[k].off + ((cy * zr[k].nx) << (zr[k].lg + 4)), map + k * 128, 0, y0 + 16 * cy, 0,
                      bar, kv_policy);
    }
  };

  // every consumer lane arrives on empty
  const FirstGuess fg = decode_prologue<D, false>(P, full, empty, NC * 32, PW, UP, LS, tab, tok, spec, stages, issue);
  if (DS && threadIdx.x == 0) {
    for (int i = 0; i < hkv; ++i) mbar_init(&pbar[i], 64);
    fence_mbar_init();
  }
  __syncthreads();
  const int32_t U = UP[B];
  const Split sp = make_split(U, B, (int)gridDim.x, P.seg_cost);  // this CTA's units: [u0, u1)
  zero_empty_sequences<D>(P, LS);
  const int32_t u0 = U == 0 ? 0 : sp.first_unit(UP, B, blockIdx.x);
  const int32_t u1 = U == 0 ? 0 : sp.first_unit(UP, B, (int64_t)blockIdx.x + 1);
  if (U == 0 || u0 >= u1) {
    if (warp == PW) finish_spec(fg, spec, err);
    return;
  }

  // Register split at the role branch: the producer warpgroup gives registers back,
  // the consumer warpgroups take them; neither path rejoins the other.
  if constexpr (RS) {
    if (warp >= 4 * NCW) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProdRegs));
      if (warp <= PW + 1)
        run_producer<D, kProducerWarps>(P, warp - PW, u0, u1, UP, tab, full, empty, tok, stages, fg, spec, issue);
      return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsRegs));
  } else if (warp >= PW) {
    run_producer<D, kProducerWarps>(P, warp - PW, u0, u1, UP, tab, full, empty, tok, stages, fg, spec, issue);
    return;
  }

  if (warp >= NC) return;  // warps without a role in the register-split layout
  // ------------------------------ consumers ---------------------------------
  // the warp's share of the head: NGL groups from group gofs; chunk counts per row
  constexpr int NGL = DS ? NG / 2 : NG;
  constexpr int NKC = Tr::NKC / (DS ? 2 : 1), NVC = Tr::NVC / (DS ? 2 : 1), NMC = Tr::NMC / (DS ? 2 : 1);
  // row sets of the S tile: rows g (tile rows 0..7) and, with more than 8 rows in use,
  // rows g + 8, each with its own softmax state and PV product
  constexpr int NSET = TWO ? 2 : 1;
  const int h = DS ? warp % hkv : warp;
  const int half = DS ? warp / hkv : 0;
  const int gofs = half * NGL;
  const int g = lane >> 2, t = lane & 3;
  // q head (within the virtual sequence's P.Hq) of tile row r
  auto qhead = [&](int r) -> size_t {
    if constexpr (NQ == 1) return (size_t)h * G + r;
    else return (size_t)(r / G) * (size_t)(P.Hq / NQ) + (size_t)h * G + (size_t)(r % G);
  };
  uint32_t qa[NSET][NGL][2][2];  // A fragments per row set, group, k-step, register
  float qsum[NSET][NGL];         // 2^-24 * sum over the group of the q~ values the MMA sees
  float o[NSET][NGL][2][4];      // O^T accumulators, in units of 2^-24: set, group, M tile, fragment
  float corr[NSET][NGL];         // sum_t p_t o_t for the lane's row and each group, this lane's tokens
  uint32_t pphase = 0;           // dim split: phase of the pair barrier
  int xpar = 0;                  // dim split: which partial-logit buffer this chunk uses
  float m_run[NSET], l_run[NSET];
  float m_eff[NSET];  // m_run - vf: the reference of the probabilities (which carry 2^vf)
  float s24[NSET];    // the row's logit scale: scale * log2(e) * 2^24 * 2^-(q~ exponent)
  int vf = 0;         // p s exponent of this warp's groups (warp-uniform)
  float vlim = 0.f;   // V scales at or above this take p s 2^vf to 2^15 (below 2^-100: vf not chosen yet)
  // dim split: every lane of both warps of the pair arrives, then waits (bounded) for
  // the other warp.  False when the wait gave up: the warp then stops (returns), so
  // its partner gives up at its next wait and no wait is ever repeated.
  auto pair_sync = [&]() -> bool {
    if constexpr (DS) {
      mbar_arrive(&pbar[h]);
      const bool ok = mbar_wait_bounded(&pbar[h], pphase, err);
      pphase ^= 1;
      return !__any_sync(0xffffffffu, !ok);
    }
    return true;
  };

  // Shared-memory addresses.  ldmatrix: lane 8i + r gives row r of matrix i.  K codes
  // (non-transposed) and V codes (transposed) are read as 8 tokens x one 16-byte
  // chunk per matrix; a K matrix for (token half j, chunk c) hands lane (g, t) word t
  // of token 8j + g, a V matrix for (token half p, chunk c) hands it half-word g of
  // tokens 8p + 2t and 8p + 2t + 1.  With NKC == 2 one x4 load covers both halves
  // (matrix i = (j = i / 2, c = i % 2)); otherwise x4 load (j, cs) covers chunks
  // 4cs..4cs+3 of half j.  The (scale, offset) chunks are read 16 bytes per token.
  const int li = lane >> 3, lr = lane & 7;
  constexpr int KCS = NKC >= 4 ? NKC / 4 : 1, VCS = NVC >= 4 ? NVC / 4 : 1;
  constexpr int NMX = NMC >= 2 ? NMC : 2;
  int kofs[KCS], vofs[VCS], mofs[NMX];
  int KSTEP = 0, VSTEP = 0, MSTEP = 0;
  const int VMD = zr[3].off - zr[2].off;
  if constexpr (W128) {
    // 128-byte rows: box row r sits at r * 128 and its chunk c at c ^ (r & 7).  A
    // lane's rows differ only by multiples of 8 (same key), so each load is a
    // per-lane constant + the chunk's uniform offset + an immediate.  For the
    // (scale, offset) reads the row key is 2t ^ e and the chunk cm of the head is
    // hb + cm = hb ^ cm (hb is a multiple of NMC), so the address depends on cm ^ e.
#pragma unroll
    for (int cs = 0; cs < KCS; ++cs) {
      const int c = NKC == 2 ? (li & 1) : 4 * cs + li;
      const int row = NKC == 2 ? 8 * (li >> 1) + lr : lr;
      const int byte = h * Tr::KB + 16 * (c + half * NKC);
      kofs[cs] = zr[0].off + (byte >> 7) * 2048 + row * 128 + ((((byte >> 4) & 7) ^ lr) << 4);
    }
#pragma unroll
    for (int cs = 0; cs < VCS; ++cs) {
      const int c = NVC == 2 ? (li & 1) : 4 * cs + li;
      const int row = NVC == 2 ? 8 * (li >> 1) + lr : lr;
      const int byte = h * Tr::VB + 16 * (c + half * NVC);
      vofs[cs] = zr[1].off + (byte >> 7) * 2048 + row * 128 + ((((byte >> 4) & 7) ^ lr) << 4);
    }
    const int mb = h * Tr::MB + 16 * half * NMC;
#pragma unroll
    for (int x = 0; x < NMX; ++x)
      mofs[x] = zr[2].off + (mb >> 7) * 2048 + 2 * t * 128 + (((((mb >> 4) & 7) ^ (2 * t)) ^ x) << 4);
    KSTEP = zr[0].nx * 2048;
    VSTEP = zr[1].nx * 2048;
    MSTEP = zr[2].nx * 2048;
  }
  auto k_addr = [&](uint32_t sb, int kc, int j, int cs) -> uint32_t {
    if constexpr (W128) {
      return sb + kc * KSTEP + kofs[cs] + (NKC == 2 ? 0 : 1024 * j);
    } else {
      const int c = NKC == 2 ? (li & 1) : 4 * cs + li;
      const int row = NKC == 2 ? 8 * (li >> 1) + lr : 8 * j + lr;
      return sb + swz(zr[0], kc * 16 + row, h * Tr::KB + 16 * (c + half * NKC));
    }
  };
  auto v_addr = [&](uint32_t sb, int kc, int p, int cs) -> uint32_t {
    if constexpr (W128) {
      return sb + kc * VSTEP + vofs[cs] + (NVC == 2 ? 0 : 1024 * p);
    } else {
      const int c = NVC == 2 ? (li & 1) : 4 * cs + li;
      const int row = NVC == 2 ? 8 * (li >> 1) + lr : 8 * p + lr;
      return sb + swz(zr[1], kc * 16 + row, h * Tr::VB + 16 * (c + half * NVC));
    }
  };
  // (scale, offset) of groups 2cm, 2cm+1 for token 16kc + 8j + 2t + e; kind 2 = K, 3 = V
  auto m_addr = [&](uint32_t sb, int kind, int kc, int j, int e, int cm) -> uint32_t {
    if constexpr (W128) {
      return sb + (kind == 3 ? VMD : 0) + kc * MSTEP + mofs[cm ^ e] + 1024 * j + 128 * e;
    } else {
      return sb + swz(zr[kind], kc * 16 + 8 * j + 2 * t + e, h * Tr::MB + 16 * (cm + half * NMC));
    }
  };

  // ---- the CTA's units, one sequence segment at a time ----
  // Logits (unmasked, before the softmax scale) of NT n-tiles: tile jj holds tokens
  // 16 kc0 + 8 jj + 2t + e of row g (set 0) and row g + 8 (set 1).  One MMA serves both
  // row sets (their q~ fill the A fragment's rows g and g + 8); the (scale, offset) fold
  // is per row.  With the dim split both halves of every logit are added (in half
  // order, by both warps).  False: a pair wait gave up.
  auto logits = [&](auto nt_c, const uint32_t sb, const int kc0, auto& x) -> bool {
    constexpr int NT = decltype(nt_c)::value;
    uint32_t kw[4][NKC];  // word t of token 16kc + 8j + g, chunk c; tile jj = 2 (kc - kc0) + j
#pragma unroll
    for (int c2 = 0; c2 < NT / 2; ++c2) {
      if constexpr (NKC == 2) {
        uint32_t r4[4];
        ldsm4(k_addr(sb, kc0 + c2, 0, 0), r4);
        kw[2 * c2][0] = r4[0];
        kw[2 * c2][1] = r4[1];
        kw[2 * c2 + 1][0] = r4[2];
        kw[2 * c2 + 1][1] = r4[3];
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int cs = 0; cs < KCS; ++cs) {
            uint32_t r4[4];
            ldsm4(k_addr(sb, kc0 + c2, j, cs), r4);
#pragma unroll
            for (int m = 0; m < 4; ++m) kw[2 * c2 + j][4 * cs + m] = r4[m];
          }
      }
    }
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      const int kc = kc0 + (jj >> 1), j = jj & 1;
      float sa[NSET][2];
#pragma unroll
      for (int st2 = 0; st2 < NSET; ++st2) sa[st2][0] = sa[st2][1] = 0.f;
#pragma unroll
      for (int cm = 0; cm < NMC; ++cm) {
        const float4 m0 = lds128(m_addr(sb, 2, kc, j, 0, cm));  // token 8j + 2t
        const float4 m1 = lds128(m_addr(sb, 2, kc, j, 1, cm));  // token 8j + 2t + 1
        // per (scale, offset) pair of the chunk: the products of the groups sharing it
        // (one group, or two with groups of 64) accumulate in one fragment, folded once
        // (qsum of the pair's first group holds the pair's sum)
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          float cacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int gi = 0; gi < Tr::SPP; ++gi) {
            const int grp = Tr::SPC * cm + Tr::SPP * pr + gi;
            uint32_t bfr[2][2];
            if constexpr (Tr::KBITS == 4) {
              k_group_frags4(kw[jj][grp], bfr);
            } else {
              k_group_frags8(kw[jj][2 * grp], kw[jj][2 * grp + 1], bfr);
            }
            mma_f16_16816(cacc, qa[0][grp][0][0], TWO ? qa[NSET - 1][grp][0][0] : 0u, qa[0][grp][0][1],
                          TWO ? qa[NSET - 1][grp][0][1] : 0u, bfr[0][0], bfr[0][1]);
            mma_f16_16816(cacc, qa[0][grp][1][0], TWO ? qa[NSET - 1][grp][1][0] : 0u, qa[0][grp][1][1],
                          TWO ? qa[NSET - 1][grp][1][1] : 0u, bfr[1][0], bfr[1][1]);
          }
          const int lead = Tr::SPC * cm + Tr::SPP * pr;
          const float sc0 = pr ? m0.z : m0.x, of0 = pr ? m0.w : m0.y;
          const float sc1 = pr ? m1.z : m1.x, of1 = pr ? m1.w : m1.y;
#pragma unroll
          for (int st2 = 0; st2 < NSET; ++st2) {
            sa[st2][0] = fmaf(sc0, cacc[2 * st2], fmaf(of0, qsum[st2][lead], sa[st2][0]));
            sa[st2][1] = fmaf(sc1, cacc[2 * st2 + 1], fmaf(of1, qsum[st2][lead], sa[st2][1]));
          }
        }
      }
#pragma unroll
      for (int st2 = 0; st2 < NSET; ++st2) {
        x[st2][jj][0] = sa[st2][0];
        x[st2][jj][1] = sa[st2][1];
      }
    }
    if constexpr (DS) {
#pragma unroll
      for (int q4 = 0; q4 < NT / 2; ++q4)
        xbuf[((((size_t)h * 2 + half) * 2 + xpar) * 2 + q4) * 32 + lane] =
            make_float4(x[0][2 * q4][0], x[0][2 * q4][1], x[0][2 * q4 + 1][0], x[0][2 * q4 + 1][1]);
      if (!pair_sync()) return false;
#pragma unroll
      for (int q4 = 0; q4 < NT / 2; ++q4) {
        const float4 pr = xbuf[((((size_t)h * 2 + (half ^ 1)) * 2 + xpar) * 2 + q4) * 32 + lane];
        float* x0 = x[0][2 * q4];
        float* x1 = x[0][2 * q4 + 1];
        x0[0] = half ? pr.x + x0[0] : x0[0] + pr.x;
        x0[1] = half ? pr.y + x0[1] : x0[1] + pr.y;
        x1[0] = half ? pr.z + x1[0] : x1[0] + pr.z;
        x1[1] = half ? pr.w + x1[1] : x1[1] + pr.w;
      }
      xpar ^= 1;
    }
    return true;
  };
  // Online softmax of each row set over NT tiles: x (scaled, masked) -> probabilities p.
  auto softmax = [&](auto nt_c, auto& x, auto& p) {
    constexpr int NT = decltype(nt_c)::value;
#pragma unroll
    for (int st2 = 0; st2 < NSET; ++st2) {
      float mx = fmaxf(x[st2][0][0], x[st2][0][1]);
#pragma unroll
      for (int jj = 1; jj < NT; ++jj) mx = fmaxf(mx, fmaxf(x[st2][jj][0], x[st2][jj][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const bool grow = mx > m_run[st2];
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? ex2(m_run[st2] - mx) : 1.0f;
        if (grow) m_run[st2] = mx;
        m_eff[st2] = m_run[st2] - (float)vf;
        l_run[st2] *= alpha;
#pragma unroll
        for (int grp = 0; grp < NGL; ++grp) corr[st2][grp] *= alpha;
        const float ae = __shfl_sync(0xffffffffu, alpha, 8 * t);
        const float ao = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
        for (int grp = 0; grp < NGL; ++grp)
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            o[st2][grp][mi][0] *= ae;
            o[st2][grp][mi][2] *= ae;
            o[st2][grp][mi][1] *= ao;
            o[st2][grp][mi][3] *= ao;
          }
      }
#pragma unroll
      for (int jj = 0; jj < NT; ++jj)
#pragma unroll
        for (int e = 0; e < 2; ++e) p[st2][jj][e] = ex2(x[st2][jj][e] - m_eff[st2]);
      if constexpr (NQ > 1) {
        // a row with no visible token yet in this segment keeps m_run = -inf
        if (m_run[st2] == -INFINITY)
#pragma unroll
          for (int jj = 0; jj < NT; ++jj) p[st2][jj][0] = p[st2][jj][1] = 0.f;
      }
      float ls = p[st2][0][0] + p[st2][0][1];
#pragma unroll
      for (int jj = 1; jj < NT; ++jj) ls += p[st2][jj][0] + p[st2][jj][1];
      l_run[st2] += ls;
    }
  };
  // The p s exponent moves by d: the state (both accumulators, the denominator and
  // the probabilities in flight) of every row set is multiplied by 2^d, exactly.
  auto v_rescale = [&](int d, auto& p) {
    const float a = pow2i(d);
#pragma unroll
    for (int st2 = 0; st2 < NSET; ++st2) {
#pragma unroll
      for (int grp = 0; grp < NGL; ++grp) {
        corr[st2][grp] *= a;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[st2][grp][mi][i] *= a;
      }
      l_run[st2] *= a;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        p[st2][jj][0] *= a;
        p[st2][jj][1] *= a;
      }
      m_eff[st2] = m_run[st2] - (float)(vf + d);
    }
    vf += d;
    vlim = pow2i(15 - vf);
  };
  // O^T += V^T (P S)^T over the 16 tokens of chunk kc (tiles p[.][jp], p[.][jp + 1]);
  // offsets into corr.  The V fragment of each M tile serves every row set.
  // MASK: only the chunk's first nvc tokens hold data (the last unit of a sequence);
  // the others' scale and offset are taken as 0.
  auto pv = [&](auto mask_c, const uint32_t sb, const int kc, auto& p, const int jp, const int nvc) {
    constexpr bool MASK = decltype(mask_c)::value;
    uint32_t vx[2][NVC];  // half-word g of tokens 16kc + 8pp + 2t, +1; chunk c
    if constexpr (NVC == 2) {
      uint32_t r4[4];
      ldsm4_t(v_addr(sb, kc, 0, 0), r4);
      vx[0][0] = r4[0];
      vx[0][1] = r4[1];
      vx[1][0] = r4[2];
      vx[1][1] = r4[3];
    } else {
#pragma unroll
      for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int cs = 0; cs < VCS; ++cs) {
          uint32_t r4[4];
          ldsm4_t(v_addr(sb, kc, pp, cs), r4);
#pragma unroll
          for (int m = 0; m < 4; ++m) vx[pp][4 * cs + m] = r4[m];
        }
    }
    auto tok_ok = [&](int pp, int e) { return !MASK || 8 * pp + 2 * t + e < nvc; };
    float4 mva[NMC][2][2];
    float sm4 = 0.f;
#pragma unroll
    for (int cm = 0; cm < NMC; ++cm)
#pragma unroll
      for (int pp = 0; pp < 2; ++pp)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mva[cm][pp][e] = lds128(m_addr(sb, 3, kc, pp, e, cm));
          if (!tok_ok(pp, e)) mva[cm][pp][e] = make_float4(0.f, 0.f, 0.f, 0.f);
          sm4 = fmaxf(sm4, fmaxf(mva[cm][pp][e].x, mva[cm][pp][e].z));
        }
    if (__any_sync(0xffffffffu, sm4 >= vlim && sm4 > 0.f)) {
      float sm = fmaxf(sm4, __shfl_xor_sync(0xffffffffu, sm4, 1));
      sm = fmaxf(sm, __shfl_xor_sync(0xffffffffu, sm, 2));
      const int nf = v_exponent_for(sm);
      if (vlim < 1e-30f || nf < vf) v_rescale(nf - vf, p);
    }
#pragma unroll
    for (int cm = 0; cm < NMC; ++cm) {
      float4 (&mv)[2][2] = mva[cm];
#pragma unroll
      for (int q = 0; q < Tr::SPC; ++q) {
        const int grp = Tr::SPC * cm + q;
        const bool q2 = q >= Tr::SPP;  // second pair of the chunk
        const float sv00 = q2 ? mv[0][0].z : mv[0][0].x, sv01 = q2 ? mv[0][1].z : mv[0][1].x;
        const float sv10 = q2 ? mv[1][0].z : mv[1][0].x, sv11 = q2 ? mv[1][1].z : mv[1][1].x;
        const float ov00 = q2 ? mv[0][0].w : mv[0][0].y, ov01 = q2 ? mv[0][1].w : mv[0][1].y;
        const float ov10 = q2 ? mv[1][0].w : mv[1][0].y, ov11 = q2 ? mv[1][1].w : mv[1][1].y;
        uint32_t pb[NSET][2];
#pragma unroll
        for (int st2 = 0; st2 < NSET; ++st2) {
          const float* p0 = p[st2][jp];
          const float* p1 = p[st2][jp + 1];
          pb[st2][0] = pack_f16x2(p0[0] * sv00, p0[1] * sv01);
          pb[st2][1] = pack_f16x2(p1[0] * sv10, p1[1] * sv11);
          // the offsets term, once per (scale, offset) pair (in its first group's slot)
          if (q % Tr::SPP == 0)
            corr[st2][grp] =
                fmaf(p0[0], ov00, fmaf(p0[1], ov01, fmaf(p1[0], ov10, fmaf(p1[1], ov11, corr[st2][grp]))));
        }
        if constexpr (Tr::VBITS == 4) {
          const uint32_t x01 = vx[0][grp], x23 = vx[1][grp];
          const uint32_t y01 = x01 >> 8, y23 = x23 >> 8;
#pragma unroll
          for (int st2 = 0; st2 < NSET; ++st2) {
            mma_f16_16816(o[st2][grp][0], x01 & 0x000F000Fu, y01 & 0x000F000Fu, x23 & 0x000F000Fu,
                          y23 & 0x000F000Fu, pb[st2][0], pb[st2][1]);
            mma_f16_16816(o[st2][grp][1], x01 & 0x00F000F0u, y01 & 0x00F000F0u, x23 & 0x00F000F0u,
                          y23 & 0x00F000F0u, pb[st2][0], pb[st2][1]);
          }
        } else {
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            const uint32_t x01 = vx[0][2 * grp + mi], x23 = vx[1][2 * grp + mi];
#pragma unroll
            for (int st2 = 0; st2 < NSET; ++st2)
              mma_f16_16816(o[st2][grp][mi], __byte_perm(x01, 0u, 0x4240), __byte_perm(x01, 0u, 0x4341),
                            __byte_perm(x23, 0u, 0x4240), __byte_perm(x23, 0u, 0x4341), pb[st2][0], pb[st2][1]);
          }
        }
      }
    }
  };
  // A whole 32-token unit (both chunks, one softmax, no masks) where registers allow it
  // (with 16 rows, in the register-split variant: a few spilled registers, one softmax
  // step per 32 tokens instead of two).
  constexpr bool kUnit32 = (!TWO && (D <= 64 || (RS && D <= 128) || DS)) || (TWO && RS);

  int b = find_seq(UP, B, u0);
  int s = 0;           // stage of the next unit
  uint32_t phase = 0;  // parity of its full barrier
  for (int32_t ua = u0; ua < u1;) {
    while (ua >= UP[b + 1]) ++b;
    const int32_t ue = min(u1, UP[b + 1]);  // this segment: units [ua, ue) of sequence b
    const int32_t Lb = LS[b];
#pragma unroll
    for (int st2 = 0; st2 < NSET; ++st2) {
#pragma unroll
      for (int grp = 0; grp < NGL; ++grp) {
        corr[st2][grp] = 0.f;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[st2][grp][mi][i] = 0.f;
      }
      m_run[st2] = -INFINITY;
      m_eff[st2] = -INFINITY;
      l_run[st2] = 0.f;
    }
    vf = 0;
    vlim = 0.f;
    for (int32_t u = ua; u < ue; ++u) {
      {
        const bool ok = mbar_wait_bounded(&full[s], phase, err);
        if (__any_sync(0xffffffffu, !ok)) return;  // a wait gave up: stop (no wait is repeated)
      }
      const uint8_t* st = stages + (size_t)s * P.stage_bytes;
      const uint32_t sb = smem_u32(st);
      if (u == ua) {
        // q~ rows of this kv head (fp16): without QG, q of the segment's sequence sits in
        // the stage (bf16) and each row becomes q~ in place (same two bytes per element),
        // read back below as the A fragments before the stage is released; with QG, q is
        // read from global memory and q~ goes to the head's scratch
        uint16_t* qst = reinterpret_cast<uint16_t*>(stages + (size_t)s * P.stage_bytes + offQ);
        const uint16_t* qglob = P.q + (size_t)b * P.Hq * D;
        auto qrow = [&](int r) -> uint16_t* { return QG ? qg_scr + ((size_t)h * RW + r) * QS : qst + qhead(r) * D; };
        // Rotation layout: with at least 16 lanes' worth of rows (rows x lanes per row)
        // the rows are spread over the lanes (short chains, two or three exchange
        // steps); with fewer the whole warp works on each row in turn.
        constexpr bool kRowLanes = RW * (D <= 128 ? 4 : 8) >= 16;
        if (half == 0 && kRowLanes) {
          // q~ = H diag(s) q / sqrt(D) for the tile rows of this kv head by a fast Walsh-
          // Hadamard transform, RPP rows at a time: LPR lanes per row, lane k of a row
          // holding its VPL consecutive dims from k VPL (butterfly spans below VPL in
          // registers, the longer ones across the row's lanes).  The row's q~ exponent e
          // puts its largest |q~| times 2^e in [2^14, 2^15); the stored fp16 value is
          // q~ 2^e, divided by 16 where the K code is read as 16c (odd dims of 4-bit K).
          constexpr int LPR = D <= 128 ? 4 : 8;  // lanes per row
          constexpr int VPL = D / LPR;            // dims per lane
          constexpr int RPP = 32 / LPR;           // rows per pass
          const int k = lane % LPR;
          const int d0 = k * VPL;
#pragma unroll 1
          for (int g0 = 0; g0 < RW; g0 += RPP) {
            const int row = g0 + lane / LPR;
            const bool live = row < RW;
            const uint16_t* src = (QG ? qglob + qhead(live ? row : 0) * D : qrow(live ? row : 0)) + d0;
            float v[VPL];
#pragma unroll
            for (int i = 0; i < VPL; i += 8) {
              const uint4 w = live ? *reinterpret_cast<const uint4*>(src + i) : make_uint4(0u, 0u, 0u, 0u);
              const float4 s0 = *reinterpret_cast<const float4*>(P.signs + d0 + i);
              const float4 s1 = *reinterpret_cast<const float4*>(P.signs + d0 + i + 4);
              v[i + 0] = __uint_as_float(w.x << 16) * s0.x;
              v[i + 1] = __uint_as_float(w.x & 0xffff0000u) * s0.y;
              v[i + 2] = __uint_as_float(w.y << 16) * s0.z;
              v[i + 3] = __uint_as_float(w.y & 0xffff0000u) * s0.w;
              v[i + 4] = __uint_as_float(w.z << 16) * s1.x;
              v[i + 5] = __uint_as_float(w.z & 0xffff0000u) * s1.y;
              v[i + 6] = __uint_as_float(w.w << 16) * s1.z;
              v[i + 7] = __uint_as_float(w.w & 0xffff0000u) * s1.w;
            }
#pragma unroll
            for (int hs = 1; hs < VPL; hs <<= 1)
#pragma unroll
              for (int i = 0; i < VPL; ++i)
                if ((i & hs) == 0) {
                  const float x = v[i], y = v[i + hs];
                  v[i] = x + y;
                  v[i + hs] = x - y;
                }
#pragma unroll
            for (int lb = 1; lb < LPR; lb <<= 1) {
              const float sgn = (k & lb) ? -1.f : 1.f;  // upper element: x - y; lower: x + y
#pragma unroll
              for (int i = 0; i < VPL; ++i) v[i] = fmaf(sgn, v[i], __shfl_xor_sync(0xffffffffu, v[i], lb));
            }
            float qm = fabsf(v[0]);
#pragma unroll
            for (int i = 1; i < VPL; ++i) qm = fmaxf(qm, fabsf(v[i]));
#pragma unroll
            for (int lb = 1; lb < LPR; lb <<= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, lb));
            qm *= P.inv_sqrt_d;
            int qe = 0;
            if (qm > 0.f) {
              qe = 14 - exponent_of(qm);
              qe = qe < -100 ? -100 : (qe > 126 ? 126 : qe);
            }
            const float qf = P.inv_sqrt_d * pow2i(qe);
            if (live) {
              uint16_t* dst = qrow(row) + d0;
              constexpr float kOdd = Tr::KBITS == 4 ? 0.0625f : 1.0f;  // odd dims of 4-bit K
#pragma unroll
              for (int i = 0; i < VPL; i += 8) {
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = pack_f16x2(v[i + 2 * j] * qf, v[i + 2 * j + 1] * qf * kOdd);
                *reinterpret_cast<uint4*>(dst + i) = make_uint4(w[0], w[1], w[2], w[3]);
              }
              if (k == 0) qes[h * 16 + row] = qe;
            }
          }
        } else if (half == 0) {
          // The same transform for few rows (RB at a time), lane l holding dims l + 32 r of
          // a row (butterfly spans 1..16 across lanes, 32.. in registers), so every lane
          // works on every row.
          constexpr int R = D / 32;
          constexpr int RB = RW < 4 ? RW : 4;
          float sg[R];
#pragma unroll
          for (int r = 0; r < R; ++r) sg[r] = P.signs[lane + 32 * r];
#pragma unroll 1
          for (int g0 = 0; g0 < RW; g0 += RB) {
            float v[RB][R];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
              const uint16_t* src = QG ? qglob + qhead(g0 + i) * D : qrow(g0 + i);
#pragma unroll
              for (int r = 0; r < R; ++r) v[i][r] = __uint_as_float((uint32_t)src[lane + 32 * r] << 16) * sg[r];
            }
#pragma unroll
            for (int hs = 1; hs < 32; hs <<= 1) {
              const float sgn = (lane & hs) ? -1.f : 1.f;  // upper element: x - y; lower: x + y
#pragma unroll
              for (int i = 0; i < RB; ++i)
#pragma unroll
                for (int r = 0; r < R; ++r) v[i][r] = fmaf(sgn, v[i][r], __shfl_xor_sync(0xffffffffu, v[i][r], hs));
            }
#pragma unroll
            for (int i = 0; i < RB; ++i) {
#pragma unroll
              for (int hr = 1; hr < R; hr <<= 1)
#pragma unroll
                for (int r = 0; r < R; ++r)
                  if ((r & hr) == 0) {
                    const float x = v[i][r], y = v[i][r + hr];
                    v[i][r] = x + y;
                    v[i][r + hr] = x - y;
                  }
            }
            float qm[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) {
              qm[i] = fabsf(v[i][0]);
#pragma unroll
              for (int r = 1; r < R; ++r) qm[i] = fmaxf(qm[i], fabsf(v[i][r]));
            }
#pragma unroll
            for (int hs = 16; hs >= 1; hs >>= 1)
#pragma unroll
              for (int i = 0; i < RB; ++i) qm[i] = fmaxf(qm[i], __shfl_xor_sync(0xffffffffu, qm[i], hs));
#pragma unroll
            for (int i = 0; i < RB; ++i) {
              const float qmi = qm[i] * P.inv_sqrt_d;
              int qe = 0;
              if (qmi > 0.f) {
                qe = 14 - exponent_of(qmi);
                qe = qe < -100 ? -100 : (qe > 126 ? 126 : qe);
              }
              const float qf = P.inv_sqrt_d * pow2i(qe);
              uint16_t* dst = qrow(g0 + i);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const float qv = v[i][r] * qf;
                dst[lane + 32 * r] = __half_as_ushort(__float2half_rn(Tr::KBITS == 4 && (lane & 1) ? qv * 0.0625f : qv));
              }
              if (lane == 0) qes[h * 16 + g0 + i] = qe;
            }
          }
        }
        // q~ of this segment is in place (dim split: written by the pair's first warp)
        if (!pair_sync()) return;
        __syncwarp();
#pragma unroll
        for (int st2 = 0; st2 < NSET; ++st2) {
          const int row = g + 8 * st2;
          const bool live = row < RW;  // rows >= RW are zero
          s24[st2] = P.scale_log2 * pow2i(live ? -qes[h * 16 + row] : 0) * 16777216.0f;
          const uint16_t* qr = qrow(live ? row : 0);
#pragma unroll
          for (int grp = 0; grp < NGL; ++grp) {
            float tsum = 0.f;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                uint32_t hv[2];
                bool d16 = false;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const int dd = 32 * (gofs + grp) + k_dim<Tr::KBITS>(t, ks, r, hh, d16);
                  hv[hh] = live ? (uint32_t)qr[dd] : 0u;
                }
                qa[st2][grp][ks][r] = hv[0] | (hv[1] << 16);
                const float2 back = unpack_f16x2(qa[st2][grp][ks][r]);  // the values the MMA sees
                tsum += d16 ? 16.f * (back.x + back.y) : (back.x + back.y);
              }
            tsum += __shfl_xor_sync(0xffffffffu, tsum, 1);
            tsum += __shfl_xor_sync(0xffffffffu, tsum, 2);
            qsum[st2][grp] = tsum * 5.9604644775390625e-08f;  // 2^-24
          }
          if constexpr (Tr::SPP == 2) {
            // groups sharing a (scale, offset) pair fold together: the pair's sum of q~
            // in its first group's slot
#pragma unroll
            for (int grp = 0; grp < NGL; grp += 2) qsum[st2][grp] += qsum[st2][grp + 1];
          }
        }
        __syncwarp();
      }
      const int nv = min(T, Lb - (u - UP[b]) * T);
      const int tleft = Lb - (u - UP[b]) * T;  // the sequence's tokens from this unit's first
      if (kUnit32 && T == 32 && nv == 32 && (NQ == 1 || tleft - (NQ - 1) >= 32)) {
        float x[NSET][4][2], p[NSET][4][2];
        if (!logits(std::integral_constant<int, 4>{}, sb, 0, x)) return;
#pragma unroll
        for (int st2 = 0; st2 < NSET; ++st2)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            x[st2][jj][0] *= s24[st2];
            x[st2][jj][1] *= s24[st2];
          }
        softmax(std::integral_constant<int, 4>{}, x, p);
        pv(std::false_type{}, sb, 0, p, 0, 16);
        pv(std::false_type{}, sb, 1, p, 2, 16);
      } else {
        // tokens of this unit visible to each of the lane's rows (its query's causal limit)
        int nvr[NSET];
#pragma unroll
        for (int st2 = 0; st2 < NSET; ++st2) {
          const int row = g + 8 * st2;
          nvr[st2] = NQ == 1 ? nv : min(T, tleft - (NQ - 1 - (row < RW ? row / G : NQ - 1)));
        }
        const bool whole = TWO && nv == T && tleft - (NQ - 1) >= T;  // every row sees every token
        for (int kc = 0; kc * 16 < nv; ++kc) {
          float x[NSET][4][2], p[NSET][4][2] = {};
          if (!logits(std::integral_constant<int, 2>{}, sb, kc, x)) return;
#pragma unroll
          for (int st2 = 0; st2 < NSET; ++st2)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int tk = kc * 16 + 8 * j + 2 * t;
              x[st2][j][0] = whole || tk < nvr[st2] ? x[st2][j][0] * s24[st2] : -INFINITY;
              x[st2][j][1] = whole || tk + 1 < nvr[st2] ? x[st2][j][1] * s24[st2] : -INFINITY;
            }
          softmax(std::integral_constant<int, 2>{}, x, p);
          if (whole) pv(std::false_type{}, sb, kc, p, 0, 16);
          else pv(std::true_type{}, sb, kc, p, 0, nv - 16 * kc);
        }
      }
      mbar_arrive(&empty[s]);  // every lane: its reads of the stage are done
      if (++s == NS) {
        s = 0;
        phase ^= 1;
      }
    }

    // ---- end of the segment: output rows, or a partial record for the combine ----
    const int32_t c_lo = sp.c_lo(UP, b), c_hi = sp.c_hi(UP, b);
#pragma unroll
    for (int st2 = 0; st2 < NSET; ++st2) {
      float lr2 = l_run[st2];
      lr2 += __shfl_xor_sync(0xffffffffu, lr2, 1);
      lr2 += __shfl_xor_sync(0xffffffffu, lr2, 2);
      const float me = __shfl_sync(0xffffffffu, m_run[st2], 8 * t), mo = __shfl_sync(0xffffffffu, m_run[st2], 8 * t + 4);
      const float le = __shfl_sync(0xffffffffu, lr2, 8 * t), lo = __shfl_sync(0xffffffffu, lr2, 8 * t + 4);
      // Offsets term of the row summed over its four lanes, then moved to the lanes
      // that hold rows 2t and 2t+1 (of the set) in the O^T fragments.
      float ce[NGL], co[NGL];
#pragma unroll
      for (int grp = 0; grp < NGL; ++grp) {
        float c = corr[st2][grp - grp % Tr::SPP];  // a pair's offsets term sits in its first group
        c += __shfl_xor_sync(0xffffffffu, c, 1);
        c += __shfl_xor_sync(0xffffffffu, c, 2);
        ce[grp] = __shfl_sync(0xffffffffu, c, 8 * t);
        co[grp] = __shfl_sync(0xffffffffu, c, 8 * t + 4);
      }
      // 2^24 undoes the subnormal code scale; tile 1 of a 4-bit group read 16c.
      const float fs[2] = {16777216.0f, Tr::VBITS == 4 ? 1048576.0f : 16777216.0f};
      const int he = 2 * t + 8 * st2, ho = 2 * t + 1 + 8 * st2;
      if (c_lo == c_hi) {
        const float ie = 1.0f / le, io = 1.0f / lo;
        uint16_t* oe = P.out + ((size_t)b * P.Hq + qhead(he < RW ? he : 0)) * D;
        uint16_t* oo = P.out + ((size_t)b * P.Hq + qhead(ho < RW ? ho : 0)) * D;
#pragma unroll
        for (int grp = 0; grp < NGL; ++grp)
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            const int d0 = v_out_dim<Tr::VBITS>(gofs + grp, mi, 0, g), d1 = v_out_dim<Tr::VBITS>(gofs + grp, mi, 1, g);
            if (he < RW) {
              oe[d0] = f2bf(fmaf(o[st2][grp][mi][0], fs[mi], ce[grp]) * ie);
              oe[d1] = f2bf(fmaf(o[st2][grp][mi][2], fs[mi], ce[grp]) * ie);
            }
            if (ho < RW) {
              oo[d0] = f2bf(fmaf(o[st2][grp][mi][1], fs[mi], co[grp]) * io);
              oo[d1] = f2bf(fmaf(o[st2][grp][mi][3], fs[mi], co[grp]) * io);
            }
          }
      } else {
        // the record holds the state without the p s exponent's 2^vf (exact), so the
        // two warps of a dim-split pair, each with its own exponent, agree
        const float iv = pow2i(-vf);
        const float fsv[2] = {fs[0] * iv, fs[1] * iv};
        float* pe = partial_ptr(P, D, (size_t)blockIdx.x, b, qhead(he < RW ? he : 0));
        float* po = partial_ptr(P, D, (size_t)blockIdx.x, b, qhead(ho < RW ? ho : 0));
        if (he < RW && g == 0 && half == 0) {
          pe[0] = me;
          pe[1] = le * iv;
        }
        if (ho < RW && g == 0 && half == 0) {
          po[0] = mo;
          po[1] = lo * iv;
        }
#pragma unroll
        for (int grp = 0; grp < NGL; ++grp) {
          const float cev = ce[grp] * iv, cov = co[grp] * iv;
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            const int d0 = v_out_dim<Tr::VBITS>(gofs + grp, mi, 0, g), d1 = v_out_dim<Tr::VBITS>(gofs + grp, mi, 1, g);
            if (he < RW) {
              pe[kPartialHeader + d0] = fmaf(o[st2][grp][mi][0], fsv[mi], cev);
              pe[kPartialHeader + d1] = fmaf(o[st2][grp][mi][2], fsv[mi], cev);
            }
            if (ho < RW) {
              po[kPartialHeader + d0] = fmaf(o[st2][grp][mi][1], fsv[mi], cov);
              po[kPartialHeader + d1] = fmaf(o[st2][grp][mi][3], fsv[mi], cov);
            }
          }
        }
      }
    }
    ua = ue;
  }
}

template <int FMT, int D, int G, bool W128, bool RS, bool DS, int GS, int NQ = 1>
cudaError_t launch_decode_packed_mma_t(const DecodeArgs& a) {
  using Tr = PackedTraits<FMT, D, GS>;
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
  const int hkv = a.lv.hkv;
  P.stage_bytes = packed_stage_bytes(P.T, hkv * Tr::KB, hkv * Tr::VB, hkv * Tr::MB, G * NQ > 8 ? 0 : a.Hq * D * 2);
  auto kern = decode_packed_mma_kernel<FMT, D, G, W128, RS, DS, GS, NQ>;
  {
    static unsigned long long smem_done = 0;  // this kernel (one per template instantiation)
    cudaError_t e = allow_max_dynamic_smem(kern, smem_done);
    if (e != cudaSuccess) return e;
  }
  const int ncons = DS ? 2 * hkv : hkv;
  const int threads = RS ? 128 * (((ncons + 3) >> 2) + 1) : (ncons + kProducerWarps) * 32;
  cudaError_t e = launch_with_pdl(kern, a.grid, threads, a.smem_bytes, a.stream, P);
  if (e != cudaSuccess) return e;
  return launch_combine<D>(P, a.grid, NQ, a.stream);
}

// The register split needs the launch allocation to cover the split: per scheduler
// 2 x kConsRegs + kProdRegs <= 3 x (registers per thread at launch); otherwise
// setmaxnreg.inc could never be satisfied.  Checked once per kernel.
template <auto Kern>
bool register_split_fits() {
  static int verdict = -1;  // one per kernel
  if (verdict < 0) {
    cudaFuncAttributes fa;
    verdict = cudaFuncGetAttributes(&fa, Kern) == cudaSuccess && fa.maxThreadsPerBlock >= kRsThreads &&
              2 * kConsRegs + kProdRegs <= 3 * fa.numRegs;
  }
  return verdict == 1;
}

template <int FMT, int GS = kGroup>
cudaError_t launch_decode_packed_mma(const DecodeArgs& a) {
  const bool w128 = a.lv.box_bytes[0] == 128 && a.lv.box_bytes[1] == 128 && a.lv.box_bytes[2] == 128 &&
                    a.lv.box_bytes[3] == 128;
#define PKV_CASE(DD, GG)                                                                                      \
  if (a.D == DD && a.G == GG) {                                                                               \
    if (DD == 256 && a.dim_split) {                                                                           \
      if (register_split_fits<decode_packed_mma_kernel<FMT, 256, GG, true, true, true, GS>>())                 \
        return launch_decode_packed_mma_t<FMT, 256, GG, true, true, true, GS>(a);                             \
      return launch_decode_packed_mma_t<FMT, 256, GG, true, false, true, GS>(a);                              \
    }                                                                                                         \
    if (w128 && DD >= 128 && register_split_fits<decode_packed_mma_kernel<FMT, DD, GG, true, true, false, GS>>()) \
      return launch_decode_packed_mma_t<FMT, DD, GG, true, true, false, GS>(a);                               \
    return w128 ? launch_decode_packed_mma_t<FMT, DD, GG, true, false, false, GS>(a)                          \
                : launch_decode_packed_mma_t<FMT, DD, GG, false, false, false, GS>(a);                        \
  }
  if constexpr (GS == kGroup) {
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
  }
  PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
  PKV_CASE(256, 1) PKV_CASE(256, 2) PKV_CASE(256, 4) PKV_CASE(256, 8)
#undef PKV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pkv

namespace pkv {

// Chunked prefill in the packed formats: NQ queries per tile, NQ x G = 8 rows
// (ROWS16 false) or 16 rows (true; head dims up to 128).  Head dim 128 with
// 128-byte rows takes the register split; other geometries the plain variants.
template <int FMT, int GS, bool ROWS16>
cudaError_t launch_decode_packed_mma_mq(const DecodeArgs& a) {
  const bool w128 = a.lv.box_bytes[0] == 128 && a.lv.box_bytes[1] == 128 && a.lv.box_bytes[2] == 128 &&
                    a.lv.box_bytes[3] == 128;
  const int G = a.G / a.nq;
#define PKV_MQ(DD, GG, NN)                                                                                    \
  if (a.D == DD && G == GG && a.nq == NN) {                                                                   \
    if constexpr (DD == 128) {                                                                                \
      if (w128 && register_split_fits<decode_packed_mma_kernel<FMT, DD, GG, true, true, false, GS, NN>>())      \
        return launch_decode_packed_mma_t<FMT, DD, GG, true, true, false, GS, NN>(a);                         \
    } else {                                                                                                  \
      if (w128) return launch_decode_packed_mma_t<FMT, DD, GG, true, false, false, GS, NN>(a);                \
    }                                                                                                         \
    return launch_decode_packed_mma_t<FMT, DD, GG, false, false, false, GS, NN>(a);                           \
  }
  if constexpr (ROWS16) {
    if constexpr (GS == kGroup) {
      PKV_MQ(64, 1, 16) PKV_MQ(64, 2, 8) PKV_MQ(64, 4, 4) PKV_MQ(64, 8, 2)
    }
    PKV_MQ(128, 1, 16) PKV_MQ(128, 2, 8) PKV_MQ(128, 4, 4) PKV_MQ(128, 8, 2)
  } else {
    if constexpr (GS == kGroup) {
      PKV_MQ(64, 1, 8) PKV_MQ(64, 2, 4) PKV_MQ(64, 4, 2)
    }
    PKV_MQ(128, 1, 8) PKV_MQ(128, 2, 4) PKV_MQ(128, 4, 2)
    PKV_MQ(256, 1, 8) PKV_MQ(256, 2, 4) PKV_MQ(256, 4, 2)
  }
#undef PKV_MQ
  return cudaErrorInvalidValue;
}

}  // namespace pkv
