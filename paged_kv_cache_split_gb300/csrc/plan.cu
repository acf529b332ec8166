// plan.cu — shared-memory plan of the decode kernel (host side).
#include "pkv_internal.cuh"

namespace pkv {

// The kernels keep NS stages of T tokens x all kv heads in shared memory (T = 32
// or 16, NS <= 8), leaving room for the barriers, the staged slab table, the
// per-sequence unit prefix and, for packed formats, the q~ exponent of each tile row
// (the rotated q~ itself replaces q in its stage).
bool plan_decode(int fmt, int D, int G, int hkv, int B, int group, DecodePlan* plan) {
  const FormatBits fb = format_bits(fmt);
  if (fb.k == 0 || hkv < 1 || hkv > 8 || B < 1 || B > 4096) return false;
  const bool packed = fmt != PKV_FMT_BF16;
  if (packed && (group <= 0 || D % group)) return false;
  const size_t meta = packed ? (size_t)(D / group) * 8 : 0;
  const size_t budget = 232448;  // 227 KB opt-in shared memory per block on sm_100-class parts
  // + staged slab table (kSmemTableEntries) + the producers' two token barriers
  size_t fixed = (size_t)(2 * B + 1 + 4) * 4 + 16 + 128 + 1024 * sizeof(void*) + 32;
  if (packed) fixed += (size_t)hkv * 16 * 4 + 16;  // the q~ exponent of each tile row
  // packed with more than 8 tile rows: q is read by the consumers (no q region in the
  // stages) and rotated into a per-kv-head scratch of G rows, D + 8 halves apart
  const bool q_global = packed && G > 8;
  if (q_global) fixed += (size_t)hkv * G * (D + 8) * 2;
  // packed D = 256 with at most 4 kv heads and 128-byte rows: the dim split's partial
  // logit buffers and pair barriers
  const bool dim_split = packed && D == 256 && hkv <= 4 && (hkv * D * fb.k / 8) % 128 == 0 &&
                         (hkv * D * fb.v / 8) % 128 == 0 && (hkv * (int)meta) % 128 == 0;
  if (dim_split) fixed += (size_t)hkv * (4096 + 8);
  if (fixed >= budget) return false;
  if (!packed) {
    // Native bf16 (tensor-core kernel): T tokens of K and of V for all kv heads, as
    // swizzled 128-byte-wide boxes, plus q of one sequence (rounded up to 1 KB so
    // every stage starts on a 1024-byte boundary); T is 32 or 16 (the PV product
    // consumes 16 tokens at a time).  Prefer T = 32 with >= 3 stages.
    const size_t row = (size_t)hkv * D * 2;
    const int cand_bf16[2] = {32, 16};
    for (int pass = 0; pass < 2; ++pass) {
      for (int T : cand_bf16) {
        const size_t stage = 2 * (size_t)T * row + (((size_t)hkv * G * D * 2 + 1023) & ~(size_t)1023);
        // + 1024: the kernel aligns the first stage to a 1024-byte boundary
        if (fixed + 1024 >= budget) return false;
        size_t ns = (budget - fixed - 1024) / (stage + 16);
        if (ns > 8) ns = 8;
        if ((pass == 0 && ns >= 3) || (pass == 1 && ns >= 2)) {
          plan->tokens_per_stage = T;
          plan->n_stages = (int)ns;
          plan->stage_bytes = stage;
          plan->smem_bytes = ns * stage + ns * 16 + fixed + 1024;
          plan->threads = (hkv + 1) * 32;
          plan->dim_split = 0;
          return true;
        }
      }
    }
    return false;
  }
  {
    // Packed formats (tensor-core kernel): T tokens of K codes, V codes, K meta and
    // V meta for all kv heads, each in a 1024-byte-aligned region of swizzled TMA
    // boxes, plus q of one sequence per stage; T = 32 (or 16 when 3 stages would
    // not fit).
    const int kr = hkv * D * fb.k / 8, vr = hkv * D * fb.v / 8, mr = hkv * (int)meta;
    const int cand_p[2] = {32, 16};
    for (int pass = 0; pass < 2; ++pass) {
      for (int T : cand_p) {
        // + 1024: the kernel aligns the first stage to a 1024-byte boundary
        const size_t stage = (size_t)packed_stage_bytes(T, kr, vr, mr, q_global ? 0 : hkv * G * D * 2);
        if (fixed + 1024 >= budget) return false;
        size_t ns = (budget - fixed - 1024) / (stage + 16);
        if (ns > 8) ns = 8;
        if ((pass == 0 && ns >= 3) || (pass == 1 && ns >= 2)) {
          plan->tokens_per_stage = T;
          plan->n_stages = (int)ns;
          plan->stage_bytes = stage;
          plan->smem_bytes = ns * stage + ns * 16 + fixed + 1024;
          plan->dim_split = dim_split;
          plan->threads = ((dim_split ? 2 * hkv : hkv) + 2) * 32;
          return true;
        }
      }
    }
    return false;
  }
}

}  // namespace pkv
