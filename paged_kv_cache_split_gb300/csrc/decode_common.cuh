// decode_common.cuh — pieces shared by the decode-attention kernels: launch
// parameters, the prologue (unit prefix over sequences, guessed and speculatively
// copied first units), the producer side of the stage ring, and the split-K merge
// kernel (in-order merge of the partials).
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
  int kv_reuse;     // 1: K/V are read again soon (chunked prefill): normal L2 priority, else evict-first
  int nq;           // queries per (virtual) sequence: 1 for decode
  int seg_cost;     // cost of a sequence start in quarter units (see Split)
};

constexpr int kMaxConsumerWarps = 8;
constexpr int kProducerWarps = 2;
constexpr int kMaxThreads = (kMaxConsumerWarps + kProducerWarps) * 32;

// 2^x with the hardware approximation (relative error below 2^-22; results below
// 2^-126 flush to zero, which a softmax weight can drop).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

// Split of the units over the CTAs.  A CTA pays for each sequence segment it starts
// (q staging or rotation at the start, the output or partial record at the end),
// about seg_cost / kCostScale units, so the split is even in cost, not in units:
// unit u of sequence b sits at position kCostScale u + seg_cost (b + 1), and CTA c
// holds the units whose positions lie in [c VC, (c + 1) VC), VC = ceil((kCostScale
// U + seg_cost B) / grid) but at least kCostScale.  seg_cost 0 gives the plain even
// split.  The attention kernels (each CTA's unit range, and whether a sequence needs
// a split-K merge) and the combine (the CTAs holding a sequence's parts) use the
// same positions.
constexpr int kCostScale = 4;

struct Split {
  int64_t VC = 0;   // positions per CTA (0: no units)
  int32_t a = 0;    // seg_cost
  __device__ __forceinline__ int32_t cta_of(int32_t u, int b) const {
    return (int32_t)(((int64_t)kCostScale * u + (int64_t)a * (b + 1)) / VC);
  }
  // first and last CTA holding units of a non-empty sequence b
  __device__ __forceinline__ int32_t c_lo(const int32_t* UP, int b) const { return cta_of(UP[b], b); }
  __device__ __forceinline__ int32_t c_hi(const int32_t* UP, int b) const { return cta_of(UP[b + 1] - 1, b); }
  // first unit of CTA c, UP[B] when it has none: the first sequence whose last unit
  // reaches position c VC, from the first of its units that does
  __device__ __forceinline__ int32_t first_unit(const int32_t* UP, int B, int64_t c) const {
    const int64_t pos = c * VC;
    int lo = 0, hi = B;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)kCostScale * (UP[mid + 1] - 1) + (int64_t)a * (mid + 1) >= pos) hi = mid;
      else lo = mid + 1;
    }
    if (lo == B) return UP[B];
    const int64_t x = pos - (int64_t)a * (lo + 1);
    const int64_t u = x <= 0 ? 0 : (x + kCostScale - 1) / kCostScale;
    return (int32_t)(u > UP[lo] ? u : UP[lo]);
  }
};

__device__ __forceinline__ Split make_split(int32_t U, int B, int grid, int seg_cost) {
  Split sp;
  sp.a = seg_cost;
  const int64_t tot = (int64_t)kCostScale * U + (int64_t)seg_cost * B;
  // at least one unit's step per CTA, so the CTAs holding a sequence's units are
  // consecutive (no CTA in between is left without a unit of it)
  const int64_t vc = (tot + grid - 1) / grid;
  sp.VC = U == 0 ? 0 : (vc > kCostScale ? vc : kCostScale);
  return sp;
}

// Prologue of every decode kernel: thread 0 initialises the stage barriers (full:
// one producer arrival plus the copied bytes; empty: NC consumer arrivals, one per
// consumer warp or lane as the kernel counts them) and the producers' two issue-token
// barriers, and warp 0 builds the unit prefix UP[0..B] over sequences (unit = T tokens
// of one sequence) and LS[b], the context length clamped to the block table.  The
// caller runs __syncthreads() afterwards.
//
// Programmatic dependent launch: the kernel waits for the previous kernel of the
// stream to complete and publish its memory (wait) before it reads any input or
// writes any output, and only then lets the next kernel of the stream be scheduled
// (launch_dependents).  So when a dependent kernel starts, everything that preceded
// this kernel on the stream has completed: the combine kernel relies on that to
// read the context lengths before its own wait.
//
// Before the wait the kernel relies only on what no kernel writes: it copies this
// layer's slab base pointers into shared memory (`tab`, when they fit; the table
// changes only through stream-ordered copies issued by append_slab), issues L2
// prefetch hints for the context lengths and the block table, prefetches the
// guessed first units' K/V and acquires their tensor maps (guess_first_units).
constexpr int kSmemTableEntries = 1024;

__device__ __forceinline__ int smem_table_entries(const DecodeParams& P) {
  const int64_t n = (P.lv.rows_capacity / P.lv.slab_blocks) * P.lv.n_kinds;
  return n <= kSmemTableEntries ? (int)n : 0;
}

// Before the dependency wait the first producer warp guesses this CTA's first units
// from the context lengths and block table as they are now (an earlier kernel may
// still be writing them: every address the guess forms is a pool row checked
// against the pool, and nothing read here is used after the wait except as a
// hint).  Lane l takes unit u0 + l while it lies in the CTA's first sequence: it
// acquires that unit's tensor maps and, for l < nprefetch, prefetches the unit's
// K/V rows into L2, so that the copies issued after the wait hit L2.  The maps'
// contents were final before this kernel started (they are written by
// stream-ordered copies when a slab is appended), and lane l of this warp is the
// thread that reads unit u0 + l's maps after the wait (the producer's first
// batch), so it may skip its own acquire when the real unit uses the same maps.
// Returns the lane's guess (map == nullptr when there is none).
struct FirstGuess {
  const uint8_t* map = nullptr;   // tensor maps of the unit's slab, acquired by this lane
  const uint8_t* qsrc = nullptr;  // q copied with the unit (it starts the CTA's segment)
  int32_t u = -1, row = -1;       // unit index and its pool row
  int b = -1, y0 = 0, j = -1;     // sequence; first slab row of the unit; block-table column
  bool spec = false;              // its copies were issued right after the wait
  int32_t row_now = -1;           // the same block-table entry read after the wait (spec lanes)
};

// The context length the kernels work with: clamped into [0, max_blocks x block
// size]; with nq > 1 queries per (virtual) sequence a length in (0, nq) is too short
// for the chunk (its first query would see no token) and counts as empty.  The
// caller flags both cases as context errors where it reads the lengths first.
__device__ __forceinline__ int32_t usable_ctx(int32_t L, int32_t lim, int nq) {
  L = L < 0 ? 0 : (L > lim ? lim : L);
  return (nq > 1 && L < nq) ? 0 : L;
}

template <int D>
__device__ __forceinline__ FirstGuess guess_first_units(const DecodeParams& P, int nprefetch) {
  FirstGuess g;
  const int lane = threadIdx.x & 31;
  const int lim = P.max_blocks * kBlockTokens;
  auto units_of = [&](int b) -> int32_t {
    const int32_t L = usable_ctx(b < P.B ? P.ctx[b] : 0, lim, P.nq);
    return (L + P.T - 1) / P.T;
  };
  int32_t tot = 0;
  for (int base = 0; base < P.B; base += 32) {
    int32_t n = units_of(base + lane);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    tot += n;
  }
  if (tot == 0) return g;
  const Split sp = make_split(tot, P.B, (int)gridDim.x, P.seg_cost);
  // the first sequence whose units reach this CTA's first position, and the CTA's
  // first unit (Split::first_unit over the guessed lengths, one lane per sequence)
  const int64_t pos = (int64_t)blockIdx.x * sp.VC;
  const int64_t pos1 = pos + sp.VC;
  int32_t carry = 0;
  int bsel = -1, nsel = 0;
  int32_t ubase = 0;
  for (int base = 0; base < P.B && bsel < 0; base += 32) {
    const int32_t n = units_of(base + lane);
    int32_t inc = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    const int bb = base + lane;
    const unsigned hit = __ballot_sync(
        0xffffffffu, bb < P.B && (int64_t)kCostScale * (carry + inc - 1) + (int64_t)sp.a * (bb + 1) >= pos);
    if (hit) {
      const int l = __ffs(hit) - 1;
      bsel = base + l;
      nsel = __shfl_sync(0xffffffffu, n, l);
      ubase = carry + __shfl_sync(0xffffffffu, inc - n, l);
    }
    carry += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (bsel < 0) return g;
  const int64_t x0 = pos - (int64_t)sp.a * (bsel + 1);
  const int64_t uf = x0 <= 0 ? 0 : (x0 + kCostScale - 1) / kCostScale;
  const int32_t u0 = (int32_t)(uf > ubase ? uf : ubase);
  const int32_t u = u0 + lane;
  // inside the first sequence and inside this CTA (position below the next CTA's first)
  if (u >= ubase + nsel || (int64_t)kCostScale * u + (int64_t)sp.a * (bsel + 1) >= pos1) return g;
  const int32_t tok0 = (u - ubase) * P.T;
  const int j = tok0 / kBlockTokens, slot0 = tok0 % kBlockTokens;
  if (j >= P.max_blocks) return g;
  const int32_t row = P.bt[(size_t)bsel * P.max_blocks + j];
  if (row < 0 || (int64_t)row >= P.lv.rows_capacity) return g;
  const int32_t slab = row / P.lv.slab_blocks, r = row - slab * P.lv.slab_blocks;
  const uint8_t* ent0 = P.lv.tab.base[(size_t)slab * P.lv.tab.stride];
  if (!ent0) return g;
  if (lane < nprefetch) {
    for (int k = 0; k < P.lv.n_kinds; ++k) {
      const uint8_t* base = P.lv.tab.base[(size_t)slab * P.lv.tab.stride + k];
      const int rowk = P.lv.row_bytes[k] * P.lv.hkv;
      if (base) bulk_prefetch_l2(base + (size_t)(r * kBlockTokens + slot0) * rowk, (uint32_t)(P.T * rowk));
    }
  }
  const uint8_t* map = ent0 + P.lv.map_delta;
  for (int k = 0; k < P.lv.n_kinds; ++k) tensormap_acquire(map + k * 128);
  g.map = map;
  g.u = u;
  g.row = row;
  g.b = bsel;
  g.j = j;
  g.y0 = r * kBlockTokens + slot0;
  if (u == u0) g.qsrc = reinterpret_cast<const uint8_t*>(P.q + (size_t)bsel * P.Hq * D);
  return g;
}

// Speculative copies: right after the dependency wait, lane l < kSpecUnits of the
// first producer warp issues the copies of its guessed unit into stage l, counted
// on spec[l] instead of full[l] (reads issued after the wait see every earlier
// write; only the choice of rows is a guess).  The producer's first batch then
// compares the guess with the real unit: when they agree it waits for the copies
// and completes full[l] with a plain arrival, otherwise it waits for them and
// issues the real unit's copies into the stage.  This takes the context-length and
// block-table reads after the wait off the path to the first data.
// The bf16 kernel uses this (SPEC); the packed kernels measured slower with it and
// issue their first units after the wait.
constexpr int kSpecUnits = 2;

// A lane that issued speculative copies waits for them (a CTA left without work,
// or a producer that stopped) before its CTA may exit.
__device__ __forceinline__ void finish_spec(const FirstGuess& g, uint64_t* spec, int32_t* err) {
  if (g.spec) mbar_wait_bounded(&spec[threadIdx.x & 31], 0, err);
}

template <int D, bool SPEC, typename IssueFn>
__device__ __forceinline__ FirstGuess decode_prologue(const DecodeParams& P, uint64_t* full, uint64_t* empty, int NC,
                                                      int PW, int32_t* UP, int32_t* LS, const uint8_t** tab,
                                                      uint64_t* tok, uint64_t* spec, uint8_t* stages,
                                                      IssueFn&& issue) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = smem_table_entries(P);
  for (int i = threadIdx.x; i < nt; i += blockDim.x) {
    const int slab = i / P.lv.n_kinds, kind = i - slab * P.lv.n_kinds;
    tab[i] = P.lv.tab.base[(size_t)slab * P.lv.tab.stride + kind];
  }
  for (int i = threadIdx.x * 32; i < P.B; i += blockDim.x * 32) prefetch_l2(P.ctx + i);
  for (int64_t i = (int64_t)threadIdx.x * 32; i < (int64_t)P.B * P.max_blocks; i += (int64_t)blockDim.x * 32)
    prefetch_l2(P.bt + i);
  FirstGuess g;
  if (warp == PW) {
    if (lane == 0) {
      for (int i = 0; i < kSpecUnits; ++i) mbar_init(&spec[i], 1);
      fence_mbar_init();
    }
    __syncwarp();
    g = guess_first_units<D>(P, P.NS < 2 ? P.NS : 2);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (SPEC && warp == PW && g.map && lane < kSpecUnits && lane < P.NS) {
    issue(&spec[lane], stages + (size_t)lane * P.stage_bytes, g.map, g.y0, 1, g.qsrc);
    g.spec = true;
    // the guessed entry as it is after the wait, read while warp 0 reads the context
    // lengths, so that validating the guess costs one round trip instead of two
    g.row_now = P.bt[(size_t)g.b * P.max_blocks + g.j];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    mbar_init(&tok[0], 1);
    mbar_init(&tok[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    const int lim = P.max_blocks * kBlockTokens;
    int32_t carry = 0;
    for (int base = 0; base < P.B; base += 32) {
      const int b = base + lane;
      int32_t n = 0;
      if (b < P.B) {
        const int32_t L0 = P.ctx[b];
        const int32_t L = usable_ctx(L0, lim, P.nq);
        if (L != L0) atomicOr(P.lv.err, ERR_CTX);
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
  return g;
}

// Producer side of the stage ring, run by NPW (1 or 2) warps that take turns over
// batches of 32 units (warp pw takes batches pw, pw + NPW, ...).  For its batch a
// warp reads the block table lane by lane and acquires each unit's tensor maps in
// the lane that will issue that unit's copies.  With two warps it then takes the
// issue token from the other warp (one mbarrier per batch parity, so units enter the
// ring in order and never more than one round ahead of the consumers), issues the
// batch in unit order and hands the token on: while one warp issues, the other
// prepares its next batch, which keeps the table reads and the fence latency off
// the issue path.  issue(bar, stage, map, y0, ok, qsrc) arms barrier `bar` with the
// unit's bytes and issues its copies.  `g` is this lane's guess of its first-batch
// unit (guess_first_units; first warp only): a unit whose maps are the guessed
// ones skips the acquire, and the stages of speculatively copied units are settled
// as described at kSpecUnits.  Every wait is bounded: a warp that gives up stops,
// so the other gives up at its next token wait.
template <int D, int NPW, typename IssueFn>
__device__ __forceinline__ void run_producer(const DecodeParams& P, const int pw, const int32_t u0, const int32_t u1,
                                             const int32_t* UP, const uint8_t* const* tab, uint64_t* full,
                                             uint64_t* empty, uint64_t* tok, uint8_t* stages,
                                             const FirstGuess& g, uint64_t* spec, IssueFn&& issue) {
  const int lane = threadIdx.x & 31;
  const int NS = P.NS, B = P.B, T = P.T;
  int32_t* err = P.lv.err;
  const bool use_stab = smem_table_entries(P) > 0;
  const int n_batches = (u1 - u0 + 31) >> 5;
  int issued = 0;  // units in the ring when this warp stopped as the last issuer (0: not the last)
  for (int k = pw; k < n_batches; k += NPW) {
    const int32_t ub = u0 + 32 * k;
    const int32_t u = ub + lane;
    const uint8_t* map = nullptr;   // tensor maps of the unit's slab (kind k at + 128 k)
    const uint8_t* qsrc = nullptr;  // q of its sequence when the unit starts a CTA's segment
    int y0 = 0, ok = 0;             // first slab row of the unit; row valid
    bool reuse = false;             // the speculative copies of this stage hold exactly this unit
    if (u < u1) {
      const int bb = find_seq(UP, B, u);
      if (u == u0 || u == UP[bb]) qsrc = reinterpret_cast<const uint8_t*>(P.q + (size_t)bb * P.Hq * D);
      const int32_t t0 = (u - UP[bb]) * T;
      const int j = t0 / kBlockTokens, slot0 = t0 % kBlockTokens;
      int32_t row;
      if (k == 0 && g.spec && g.u == u && g.b == bb && g.j == j)
        row = g.row_now;  // already read after the wait
      else
        row = P.bt[(size_t)bb * P.max_blocks + j];
      if (row >= 0 && (int64_t)row < P.lv.rows_capacity) {
        const int32_t slab = row / P.lv.slab_blocks;
        const int32_t r = row - slab * P.lv.slab_blocks;
        const uint8_t* ent0 =
            use_stab ? tab[(size_t)slab * P.lv.n_kinds] : P.lv.tab.base[(size_t)slab * P.lv.tab.stride];
        map = ent0 + P.lv.map_delta;
        y0 = r * kBlockTokens + slot0;
        ok = 1;
        if (k != 0 || map != g.map)
          for (int kk = 0; kk < P.lv.n_kinds; ++kk) tensormap_acquire(map + kk * 128);
        reuse = k == 0 && g.spec && g.u == u && g.b == bb && g.row == row && g.map == map && g.qsrc == qsrc;
      } else {
        atomicOr(err, ERR_ROW);
      }
    }
    if (NPW == 2 && k > 0) {
      const bool got = mbar_wait_bounded(&tok[k & 1], ((k - 1) >> 1) & 1, err);
      if (__any_sync(0xffffffffu, !got)) return;  // the other warp stopped; nothing of this warp is in flight
    }
    const int cnt = min(32, u1 - ub);
    int i0 = 0;  // first unit of the batch left to the in-order loop below
    bool dead = false;
    if (k == 0) {
      // First round of the ring (no stage in use yet): units without speculative
      // copies are issued first, then each speculative stage is settled by its lane
      // once its copies have landed.
      const unsigned smask = __ballot_sync(0xffffffffu, g.spec);
      i0 = min(cnt, NS);
      for (int i = 0; i < i0; ++i)
        if (lane == i && !((smask >> i) & 1u)) issue(&full[i], stages + (size_t)i * P.stage_bytes, map, y0, ok, qsrc);
      int bad = 0;
      if (g.spec) {
        if (!mbar_wait_bounded(&spec[lane], 0, err))
          bad = 1;
        else if (lane < cnt) {
          if (reuse)
            mbar_arrive(&full[lane]);
          else
            issue(&full[lane], stages + (size_t)lane * P.stage_bytes, map, y0, ok, qsrc);
        }
      }
      dead = __any_sync(0xffffffffu, bad);
    }
    int n = 32 * k + i0;         // ring position of unit ub + i0
    int s = n % NS;              // its stage
    uint32_t ph = (n / NS) & 1;  // parity of that stage's round
    for (int i = i0; i < cnt && !dead; ++i, ++n) {
      int bad = 0;
      if (lane == i) {
        if (n >= NS && !mbar_wait_bounded(&empty[s], ph ^ 1, err))
          bad = 1;
        else
          issue(&full[s], stages + (size_t)s * P.stage_bytes, map, y0, ok, qsrc);
      }
      if (__any_sync(0xffffffffu, bad)) {
        dead = true;
        break;
      }
      if (++s == NS) {
        s = 0;
        ph ^= 1;
      }
    }
    if (dead || k + 1 >= n_batches) {
      issued = n;
      break;
    }
    if (NPW == 2) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&tok[(k + 1) & 1]);
    }
  }
  // The last issuer (or the warp that gave up while holding the token) leaves no
  // copy in flight into a stage that is no longer waited on.
  if (issued > 0 && lane == 0) {
    const int first = issued > NS ? issued - NS : 0;
    for (int m = first; m < issued; ++m) mbar_wait_bounded(&full[m % NS], (m / NS) & 1, err);
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

// Partial record of one (CTA, sequence, query head), 16-byte aligned:
//   [m (running max, base 2), l (sum of probabilities), 0, 0, acc[D]]
// in slot (CTA + sequence); CTAs c and c+1 of one sequence use consecutive slots.
constexpr int kPartialHeader = 4;

__host__ __device__ constexpr int partial_floats(int D) { return D + kPartialHeader; }

__device__ __forceinline__ float* partial_ptr(const DecodeParams& P, int D, size_t cta, int b, size_t head) {
  return P.partials + (((cta + (size_t)b) * P.Hq) + head) * (size_t)partial_floats(D);
}

template <int V>
struct VecF;
template <>
struct VecF<1> {
  using T = float;
};
template <>
struct VecF<2> {
  using T = float2;
};
template <>
struct VecF<4> {
  using T = float4;
};

// The combine gives each (sequence, query head) to S warps, one per slice of the
// head's dims (S = 1: the whole head); a lane holds V = D / (32 S) consecutive dims.
// Decode uses S = 1; chunked prefill, with many more (virtual sequence, head) pairs
// each spread over as many CTAs, uses S = 4, which shortens each warp's chain.
template <int D, int S>
struct CombineShape {
  static constexpr int V = D / (32 * S);                   // dims per lane: 1..8
  static constexpr int NV = V > 4 ? 2 : 1;                 // vector loads per part
  static constexpr int VW = V / NV;                        // floats per load
  static constexpr int N = S == 1 ? (D <= 128 ? 10 : 5) : 12;  // parts per load round
};

// Merge of up to N parts of one (sequence, query head, slice), parts i0 .. i0+cnt-1
// of the records at `base` (one every `pstride` floats; `dofs` the slice's first
// dim), into the running (M, den, num): lane k holds part k's (m, l) for the max
// and the denominator, every lane its V dims of each part for the numerator.  All
// loads are issued before any is used.  `first` (no earlier round) skips the
// rescale of an empty state, which would multiply zeros by zero.
template <int D, int S>
__device__ __forceinline__ void merge_chunk(const float* base, size_t pstride, int dofs, int i0, int cnt, int lane,
                                            bool first, float& M, float& den, float (&num)[CombineShape<D, S>::V]) {
  using Sh = CombineShape<D, S>;
  constexpr int V = Sh::V, NV = Sh::NV, N = Sh::N;
  using Vec = typename VecF<Sh::VW>::T;
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < cnt) ml = __ldcg(reinterpret_cast<const float2*>(base + (size_t)(i0 + lane) * pstride));
  Vec v[N][NV];
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (k < cnt)
#pragma unroll
      for (int x = 0; x < NV; ++x)
        v[k][x] = __ldcg(reinterpret_cast<const Vec*>(base + (size_t)(i0 + k) * pstride + kPartialHeader + dofs +
                                                      lane * V) + x);
  // Lanes = parts: the round's max, weights, denominator.
  float Mc = ml.x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, off));
  Mc = fmaxf(Mc, M);
  const float wgt = exp2f(ml.x - Mc);
  float dc = wgt * ml.y;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dc += __shfl_xor_sync(0xffffffffu, dc, off);
  if (first) {
    den = dc;
  } else {
    const float a = exp2f(M - Mc);  // rescales earlier rounds
    den = fmaf(den, a, dc);
#pragma unroll
    for (int j = 0; j < V; ++j) num[j] *= a;
  }
  M = Mc;
  // Lanes = dims: add the round's parts in order.
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (k < cnt) {
      const float wk = __shfl_sync(0xffffffffu, wgt, k);
      const float* vf = reinterpret_cast<const float*>(&v[k][0]);
#pragma unroll
      for (int j = 0; j < V; ++j) num[j] = fmaf(wk, vf[j], num[j]);
    }
  }
}

// Split-K merge, a separate kernel chained after the attention kernel: for every
// (sequence, query head) of a sequence that more than one CTA worked on, S warps
// (one per slice of the head's dims, CombineShape) merge the parts one after
// another in CTA order with the online-softmax rule (running max, rescaled
// denominator and numerator), so the result does not depend on which CTA finished
// first.  Parts are loaded in rounds of CombineShape::N, all loads of a round issued
// before any is used.
//
// The kernel is latency-bound (a few hundred dependent instructions per warp
// around one L2 round trip), so everything that does not need the partials (the
// unit prefix, the CTA share, each warp's first (sequence, head) and its part
// range) is computed before the dependency wait.  The attention kernel signals its
// dependents only after its own wait, so the context lengths (inputs of the
// attention call, never written by it) are final when this kernel starts.
//
// This kernel releases its own dependents before its wait: the next kernel
// (typically the next call's attention kernel) may then be scheduled onto SMs
// that the tail of this call's attention grid has left, and run its prologue and
// L2 prefetches there; its own wait still covers this kernel's completion, and
// this kernel completes only after the attention grid has.
//
// One warp per CTA (W warps for bf16 prefill), at most 80 registers a thread (launch
// bounds): the block scheduler packs up to eight of these CTAs onto an SM that the
// attention grid has left, and an attention CTA of the next call (about 44k
// registers, 219 KB of shared memory) still fits beside eight one-warp CTAs (8 x 80 x
// 32 registers, 1 KB of shared memory each), so the next call's CTAs are not held
// back until the merge ends.
// With 256-thread CTAs of 176 registers a thread, such CTAs filled the SM's
// registers and the next call's CTAs on about 16 SMs started 4-5 us late.
template <int D, int S, int W = 1>
__global__ void __launch_bounds__(32 * W, 25 / W) combine_kernel(const DecodeParams P, int main_grid) {
  extern __shared__ int32_t cup[];  // unit prefix UP[0..B]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const int lim = P.max_blocks * kBlockTokens;
    int32_t carry = 0;
    for (int base = 0; base < P.B; base += 32) {
      const int b = base + lane;
      int32_t n = 0;
      if (b < P.B) {
        const int32_t L = usable_ctx(P.ctx[b], lim, P.nq);
        n = (L + P.T - 1) / P.T;
      }
      int32_t inc = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
      }
      if (b < P.B) cup[b] = carry + inc - n;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) cup[P.B] = carry;
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int V = CombineShape<D, S>::V;  // dims per lane of the warp's slice
  constexpr int NC = CombineShape<D, S>::N;
  const int32_t U = cup[P.B];
  const Split sp = make_split(U, P.B, main_grid, P.seg_cost);
  const size_t pstride = (size_t)P.Hq * partial_floats(D);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int items = S * P.B * P.Hq;  // (sequence, head, slice)
  // this warp's first item and its part range, before the wait
  int item = blockIdx.x * (blockDim.x >> 5) + warp;
  int b = (item / S) / P.Hq;
  int32_t c_lo = 0, c_hi = 0;
  if (U > 0 && item < items && cup[b + 1] > cup[b]) {
    c_lo = sp.c_lo(cup, b);
    c_hi = sp.c_hi(cup, b);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (U == 0) return;
  while (item < items) {
    const size_t head = (size_t)(item / S - b * P.Hq);
    const int dofs = S > 1 ? (item % S) * (D / S) : 0;
    const int nparts = c_hi - c_lo + 1;
    // empty sequences (zeros written by the attention kernel) and sequences of one
    // CTA (output written directly) have c_hi == c_lo
    if (nparts > 1) {
      const float* base = partial_ptr(P, D, (size_t)c_lo, b, head);
      float M = -INFINITY, den = 0.f, num[V];
#pragma unroll
      for (int j = 0; j < V; ++j) num[j] = 0.f;
#pragma unroll 1
      for (int i0 = 0; i0 < nparts; i0 += NC)
        merge_chunk<D, S>(base, pstride, dofs, i0, min(NC, nparts - i0), lane, i0 == 0, M, den, num);
      const float inv = 1.0f / den;
      uint16_t* o = P.out + ((size_t)b * P.Hq + head) * D + dofs + lane * V;
      if constexpr (V == 1) {
        *o = f2bf(num[0] * inv);
      } else {
        uint32_t w[V / 2];
#pragma unroll
        for (int j = 0; j < V / 2; ++j)
          w[j] = (uint32_t)f2bf(num[2 * j] * inv) | ((uint32_t)f2bf(num[2 * j + 1] * inv) << 16);
        if constexpr (V == 2) {
          *reinterpret_cast<uint32_t*>(o) = w[0];
        } else if constexpr (V == 4) {
          *reinterpret_cast<uint2*>(o) = make_uint2(w[0], w[1]);
        } else {
          *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    item += nwarps;
    if (item >= items) break;
    b = (item / S) / P.Hq;
    c_lo = c_hi = 0;
    if (cup[b + 1] > cup[b]) {
      c_lo = sp.c_lo(cup, b);
      c_hi = sp.c_hi(cup, b);
    }
  }
}

// Opt `kern` in to the largest dynamic shared memory a block may use (227 KB).  The
// attribute belongs to the current device, so it is set once per device; `done` is
// the caller's record for this kernel (bit d: set on device d).
template <typename Kern>
inline cudaError_t allow_max_dynamic_smem(Kern kern, unsigned long long& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && ((done >> dev) & 1ull)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  if (e == cudaSuccess && dev < 64) done |= 1ull << dev;
  return e;
}

// Launch `kern` with programmatic stream serialization enabled (see above).
template <typename Kern>
inline cudaError_t launch_with_pdl(Kern kern, int grid, int threads, size_t smem, cudaStream_t stream,
                                   const DecodeParams& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int D, int S, int W = 1>
inline cudaError_t launch_combine_s(const DecodeParams& P, int main_grid, cudaStream_t stream) {
  const int pairs = P.B * P.Hq;
  // one warp per (sequence, head, slice), W warps (consecutive items) per CTA; see
  // combine_kernel
  int grid = (S * pairs + W - 1) / W;
  if (grid > 8192) grid = 8192;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(32 * W);
  cfg.dynamicSmemBytes = (size_t)(P.B + 1) * sizeof(int32_t);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, S, W>, P, main_grid);
}

// Decode: one warp per (sequence, head); chunked prefill (nq > 1 queries per virtual
// sequence, so nq times the heads): two warps per head, each merging half of its dims
// (at head_dim 128, four warps per head merged the bf16 chunk of 8 as fast and the
// K4/V4 one 2% slower; one warp per head was 8% slower on bf16).  WP: warps per CTA
// for prefill (the two warps of a head in one CTA: bf16 prefill +4%, K4/V4 -1%).
template <int D, int WP = 1>
inline cudaError_t launch_combine(const DecodeParams& P, int main_grid, int nq, cudaStream_t stream) {
  return nq > 1 ? launch_combine_s<D, 2, WP>(P, main_grid, stream) : launch_combine_s<D, 1>(P, main_grid, stream);
}

}  // namespace pkv
