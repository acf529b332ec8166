/*
 * pkv_oracle.c — the oracle for paged decode attention over a chunked-slab KV pool.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously-correct CPU
 * statement of what the GPU library computes.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it; the library never
 * does, and it shares no source, header, table or constant with the CUDA code.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (no FMA contraction, so every float operation below is one IEEE-rounded step).
 *
 * Sources followed (cited by page title and section):
 *  [SLAB]  mlxcel issue #235, "chunked slab storage for the paged pool":
 *          Proposed solution (bullets 1-3) and touch points 1-3, 5.
 *  [PACK]  mlx-swift-lm PR #142, "packed paged KV formats with bounded workspace
 *          admission": Summary; After flowchart (new K/V quantised a single
 *          time on write; attention reads the packed pages directly).
 *  [ATTN]  mlxcel issue #2171, "one KV storage abstraction with dense and paged
 *          backends": Proposed Solution (attend = update storage, then attention)
 *          and Implementation Notes / Edge cases (single token, no mask).
 *
 * Readings taken where the pages are silent (each is also listed in the design
 * notes):
 *  - affine groups are 32 consecutive values of one (token, head) row, with an
 *    FP32 (scale, offset) pair; scale = (max-min)/(2^bits-1), offset = min,
 *    code = round-half-even((x-min)/scale) clamped to [0, 2^bits-1]; a constant
 *    group (scale 0) stores code 0;
 *  - 4-bit codes pack element 2j in the low nibble and 2j+1 in the high nibble;
 *  - the signed Hadamard basis is R = H_D diag(s) with H_D the Sylvester matrix
 *    scaled by 1/sqrt(D) and s_i = -1 iff the top bit of splitmix64(seed+i) is set;
 *    it rotates the whole head_dim of K (before quantising) and of Q; V and the
 *    native bf16 format are not rotated;
 *  - the rotated K value is (float)( (sum_j H_ij s_j k_j) * (1/sqrt(D)) ) with
 *    the +-1 sum exact in FP64 (checked, see rotate_k) and two roundings after it
 *    (FP64 product, then FP32);
 *  - query head h reads KV head h / (Hq/Hkv);
 *  - a sequence of length 0 attends to nothing and returns zeros.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FMT_BF16 0
#define OR_FMT_K4V4 1
#define OR_FMT_K8V4 2
#define OR_FMT_K8V8 3

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_RANGE (-5)
#define OR_ERR_MEM (-2)

/* ------------------------------------------------------------------------- */
/* Scalars                                                                   */
/* ------------------------------------------------------------------------- */

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014; the 64-bit finaliser constants as published by
 * Vigna).  Returns the output for state x, i.e. mix(x + golden gamma). */
uint64_t oracle_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Signs of the fixed signed Hadamard basis [PACK, Summary]: s_i in {+1,-1}. */
void oracle_hadamard_signs(uint64_t seed, int D, double* s) {
  for (int i = 0; i < D; ++i) s[i] = (oracle_splitmix64(seed + (uint64_t)i) >> 63) ? -1.0 : 1.0;
}

static int popcount32(uint32_t v) { return __builtin_popcount(v); }

/* Entry (i, j) of the orthonormal Sylvester Hadamard matrix of order D. */
double oracle_hadamard_entry(int i, int j, int D) {
  double sgn = (popcount32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
  return sgn / sqrt((double)D);
}

static int ilog2(int v) {
  int r = 0;
  while ((1 << r) < v) ++r;
  return r;
}

/* Largest binary exponent E with 2^E <= |x| (x != 0, finite). */
static int exponent_of(double x) {
  int e;
  frexp(x, &e); /* x = m * 2^e, 0.5 <= |m| < 1 */
  return e - 1;
}

/* Rotated K for one (token, head) row [PACK, Summary: signed Hadamard basis for
 * Q/K].  y_i = (float)( (sum_j (-1)^popcount(i&j) s_j k_j) * (1/sqrt(D)) ).
 * Returns 1 when the FP64 sum is exact for every i (every nonzero input is a
 * multiple of 2^(Emin-7) and |sum| < D*2^(Emax+1), so the sum is exact when
 * Emax - Emin <= 45 - log2(D)); 0 otherwise (the result is still produced). */
/* The same rotation with the +-1 entries of sqrt(D) * H_D taken from a table
 * (hs[i * D + j] = (-1)^popcount(i&j)); used by the pool image for speed. */
static int rotate_k_table(const uint16_t* k_bf16, int D, const double* signs, const double* hs, float* out) {
  int emin = 100000, emax = -100000;
  double x[512];
  for (int j = 0; j < D; ++j) {
    double v = bf16_to_double(k_bf16[j]);
    x[j] = signs[j] * v;
    if (v != 0.0) {
      int e = exponent_of(v);
      if (e < emin) emin = e;
      if (e > emax) emax = e;
    }
  }
  int exact = (emax < emin) || (emax - emin <= 45 - ilog2(D));
  const double inv = 1.0 / sqrt((double)D);
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int j = 0; j < D; ++j) acc += hs[(size_t)i * D + j] * x[j];
    double prod = acc * inv;
    out[i] = (float)prod;
  }
  return exact;
}

int oracle_rotate_k(const uint16_t* k_bf16, int D, const double* signs, float* out) {
  int emin = 100000, emax = -100000;
  for (int j = 0; j < D; ++j) {
    double v = bf16_to_double(k_bf16[j]);
    if (v != 0.0) {
      int e = exponent_of(v);
      if (e < emin) emin = e;
      if (e > emax) emax = e;
    }
  }
  int exact = (emax < emin) || (emax - emin <= 45 - ilog2(D));
  const double inv = 1.0 / sqrt((double)D);
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int j = 0; j < D; ++j) {
      double h = (popcount32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
      acc += h * signs[j] * bf16_to_double(k_bf16[j]);
    }
    double prod = acc * inv;
    out[i] = (float)prod;
  }
  return exact;
}

/* Rotated Q in FP64 (no rounding to FP32): q~ = H diag(s) q. */
void oracle_rotate_q(const double* q, int D, const double* signs, double* out) {
  for (int i = 0; i < D; ++i) {
    double acc = 0.0;
    for (int j = 0; j < D; ++j) acc += oracle_hadamard_entry(i, j, D) * signs[j] * q[j];
    out[i] = acc;
  }
}

/* ------------------------------------------------------------------------- */
/* Token-local affine quantiser [PACK, Summary]                              */
/* ------------------------------------------------------------------------- */

/* Quantise one group of n values to `bits`-bit codes (one code per byte in
 * codes[]), writing (scale, offset). */
static void quantize_group(const float* x, int n, int bits, uint8_t* codes, float* scale_out,
                           float* offset_out) {
  float mn = x[0], mx = x[0];
  for (int i = 1; i < n; ++i) {
    if (x[i] < mn) mn = x[i];
    if (x[i] > mx) mx = x[i];
  }
  const int top = (1 << bits) - 1;
  float range = mx - mn;
  float scale = range / (float)top;
  for (int i = 0; i < n; ++i) {
    long c = 0;
    if (scale != 0.0f) {
      float d = x[i] - mn;
      float r = d / scale;
      c = lrintf(r); /* round half to even in the default rounding mode */
      if (c < 0) c = 0;
      if (c > top) c = top;
    }
    codes[i] = (uint8_t)c;
  }
  *scale_out = scale;
  *offset_out = mn;
}

/* Quantise a row of D values with groups of `group` (D % group == 0).
 * codes_packed: D/2 bytes (bits=4, element 2j in the low nibble of byte j) or
 * D bytes (bits=8).  meta: D/group pairs (scale, offset). */
int oracle_quantize(const float* x, int D, int bits, int group, uint8_t* codes_packed, float* meta) {
  if ((bits != 4 && bits != 8) || group <= 0 || D % group) return OR_ERR_ARG;
  uint8_t* codes = (uint8_t*)malloc((size_t)D);
  if (!codes) return OR_ERR_MEM;
  for (int g = 0; g < D / group; ++g)
    quantize_group(x + g * group, group, bits, codes + g * group, &meta[2 * g], &meta[2 * g + 1]);
  if (bits == 8) {
    memcpy(codes_packed, codes, (size_t)D);
  } else {
    for (int j = 0; j < D / 2; ++j)
      codes_packed[j] = (uint8_t)((codes[2 * j] & 0xF) | ((codes[2 * j + 1] & 0xF) << 4));
  }
  free(codes);
  return OR_OK;
}

/* x^_i = code_i * scale + offset, in FP64. */
int oracle_dequantize(const uint8_t* codes_packed, const float* meta, int D, int bits, int group,
                      double* out) {
  if ((bits != 4 && bits != 8) || group <= 0 || D % group) return OR_ERR_ARG;
  for (int i = 0; i < D; ++i) {
    int c = (bits == 8) ? codes_packed[i]
                        : ((i & 1) ? (codes_packed[i / 2] >> 4) : (codes_packed[i / 2] & 0xF));
    int g = i / group;
    out[i] = (double)c * (double)meta[2 * g] + (double)meta[2 * g + 1];
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Host image of the chunked-slab pool [SLAB, Proposed solution]             */
/* ------------------------------------------------------------------------- */

typedef struct oracle_pool {
  int n_layers, n_kv_heads, head_dim, block_size, slab_blocks, group_size, format;
  int k_bits, v_bits; /* 16 for native bf16 */
  int n_kinds;        /* 2 (K, V) or 4 (K, V, K meta, V meta) */
  size_t row_bytes[4];
  double* signs;
  double* hs; /* [D * D] entries of sqrt(D) * H_D */
  int n_slabs, cap_slabs;
  uint8_t** slab; /* slab[(s * n_layers + layer) * n_kinds + kind] */
  long inexact_rotations;
} oracle_pool;

static int format_bits(int format, int* kb, int* vb) {
  switch (format) {
    case OR_FMT_BF16: *kb = 16; *vb = 16; return 1;
    case OR_FMT_K4V4: *kb = 4; *vb = 4; return 1;
    case OR_FMT_K8V4: *kb = 8; *vb = 4; return 1;
    case OR_FMT_K8V8: *kb = 8; *vb = 8; return 1;
    default: return 0;
  }
}

oracle_pool* oracle_pool_new(int n_layers, int n_kv_heads, int head_dim, int format, uint64_t seed,
                             int block_size, int slab_blocks, int group_size) {
  int kb, vb;
  if (n_layers <= 0 || n_kv_heads <= 0 || head_dim <= 0 || head_dim > 512 || block_size <= 0 ||
      slab_blocks <= 0)
    return NULL;
  if (!format_bits(format, &kb, &vb)) return NULL;
  if (format != OR_FMT_BF16 && (group_size <= 0 || head_dim % group_size)) return NULL;
  oracle_pool* p = (oracle_pool*)calloc(1, sizeof *p);
  if (!p) return NULL;
  p->n_layers = n_layers;
  p->n_kv_heads = n_kv_heads;
  p->head_dim = head_dim;
  p->block_size = block_size;
  p->slab_blocks = slab_blocks;
  p->group_size = group_size;
  p->format = format;
  p->k_bits = kb;
  p->v_bits = vb;
  p->n_kinds = (format == OR_FMT_BF16) ? 2 : 4;
  p->row_bytes[0] = (size_t)head_dim * (size_t)kb / 8;
  p->row_bytes[1] = (size_t)head_dim * (size_t)vb / 8;
  if (p->n_kinds == 4) {
    p->row_bytes[2] = (size_t)(head_dim / group_size) * 2 * sizeof(float);
    p->row_bytes[3] = p->row_bytes[2];
  }
  p->signs = (double*)malloc(sizeof(double) * (size_t)head_dim);
  if (!p->signs) { free(p); return NULL; }
  oracle_hadamard_signs(seed, head_dim, p->signs);
  p->hs = (double*)malloc(sizeof(double) * (size_t)head_dim * (size_t)head_dim);
  if (!p->hs) { free(p->signs); free(p); return NULL; }
  for (int i = 0; i < head_dim; ++i)
    for (int j = 0; j < head_dim; ++j)
      p->hs[(size_t)i * head_dim + j] = (popcount32((uint32_t)(i & j)) & 1) ? -1.0 : 1.0;
  return p;
}

void oracle_pool_free(oracle_pool* p) {
  if (!p) return;
  for (long i = 0; i < (long)p->n_slabs * p->n_layers * p->n_kinds; ++i) free(p->slab[i]);
  free(p->slab);
  free(p->signs);
  free(p->hs);
  free(p);
}

static size_t slab_bytes(const oracle_pool* p, int kind) {
  return (size_t)p->slab_blocks * (size_t)p->block_size * (size_t)p->n_kv_heads * p->row_bytes[kind];
}

/* Grow to at least `rows` rows by appending zero-filled slabs; existing slabs are
 * never touched [SLAB, Proposed solution, bullet 2]. */
int oracle_pool_reserve_rows(oracle_pool* p, int64_t rows) {
  int need = (int)((rows + p->slab_blocks - 1) / p->slab_blocks);
  if (need <= p->n_slabs) return OR_OK;
  long per = (long)p->n_layers * p->n_kinds;
  uint8_t** ns = (uint8_t**)realloc(p->slab, sizeof(uint8_t*) * (size_t)(need * per));
  if (!ns) return OR_ERR_MEM;
  p->slab = ns;
  for (int s = p->n_slabs; s < need; ++s)
    for (int l = 0; l < p->n_layers; ++l)
      for (int k = 0; k < p->n_kinds; ++k) {
        uint8_t* b = (uint8_t*)calloc(1, slab_bytes(p, k));
        if (!b) return OR_ERR_MEM;
        p->slab[((long)s * p->n_layers + l) * p->n_kinds + k] = b;
      }
  p->n_slabs = need;
  return OR_OK;
}

int64_t oracle_pool_rows(const oracle_pool* p) { return (int64_t)p->n_slabs * p->slab_blocks; }
long oracle_pool_inexact_rotations(const oracle_pool* p) { return p->inexact_rotations; }

/* Address of (layer, kind, row, slot, head): slab = row / slab_blocks,
 * row_in_slab = row % slab_blocks [SLAB, Proposed solution, bullet 1]; inside a
 * slab shaped [slab_blocks, block_size, n_kv_heads, row] the element sits at
 * ((row_in_slab * block_size + slot) * n_kv_heads + head) * row_bytes. */
static uint8_t* addr(const oracle_pool* p, int layer, int kind, int32_t row, int slot, int head) {
  int s = row / p->slab_blocks;
  int r = row % p->slab_blocks;
  uint8_t* base = p->slab[((long)s * p->n_layers + layer) * p->n_kinds + kind];
  size_t off = (((size_t)r * p->block_size + (size_t)slot) * p->n_kv_heads + (size_t)head) *
               p->row_bytes[kind];
  return base + off;
}

static int row_ok(const oracle_pool* p, int32_t row) {
  return row >= 0 && (int64_t)row < oracle_pool_rows(p);
}

/* write_block [SLAB, touch point 1], new K/V quantised a single time [PACK, After]:
 * token i of k/v ([n, Hkv, D] bf16) goes to (rows[i], slots[i]). */
int oracle_write_block(oracle_pool* p, int layer, int n, const int32_t* rows, const int32_t* slots,
                       const uint16_t* k, const uint16_t* v) {
  if (layer < 0 || layer >= p->n_layers || n < 0) return OR_ERR_ARG;
  const int D = p->head_dim, H = p->n_kv_heads;
  int rc = OR_OK;
  long inexact = 0;
  /* Tokens are independent; rows written by two tokens of one call must differ. */
#pragma omp parallel for schedule(static) reduction(+ : inexact)
  for (int i = 0; i < n; ++i) {
    float xr[512];
    if (!row_ok(p, rows[i]) || slots[i] < 0 || slots[i] >= p->block_size) {
#pragma omp atomic write
      rc = OR_ERR_RANGE;
      continue;
    }
    for (int h = 0; h < H; ++h) {
      const uint16_t* kr = k + ((size_t)i * H + h) * D;
      const uint16_t* vr = v + ((size_t)i * H + h) * D;
      if (p->format == OR_FMT_BF16) {
        memcpy(addr(p, layer, 0, rows[i], slots[i], h), kr, p->row_bytes[0]);
        memcpy(addr(p, layer, 1, rows[i], slots[i], h), vr, p->row_bytes[1]);
        continue;
      }
      if (!rotate_k_table(kr, D, p->signs, p->hs, xr)) inexact++;
      oracle_quantize(xr, D, p->k_bits, p->group_size, addr(p, layer, 0, rows[i], slots[i], h),
                      (float*)addr(p, layer, 2, rows[i], slots[i], h));
      for (int d = 0; d < D; ++d) xr[d] = bf16_to_float(vr[d]);
      oracle_quantize(xr, D, p->v_bits, p->group_size, addr(p, layer, 1, rows[i], slots[i], h),
                      (float*)addr(p, layer, 3, rows[i], slots[i], h));
    }
  }
  p->inexact_rotations += inexact;
  return rc;
}

/* copy_on_write_block [SLAB, touch point 2]: every byte of block src[i] (every
 * layer, every stored tensor) is copied to block dst[i]. */
int oracle_copy_block(oracle_pool* p, int n, const int32_t* src, const int32_t* dst) {
  int rc = OR_OK;
  for (int i = 0; i < n; ++i) {
    if (!row_ok(p, src[i]) || !row_ok(p, dst[i])) { rc = OR_ERR_RANGE; continue; }
    for (int l = 0; l < p->n_layers; ++l)
      for (int kind = 0; kind < p->n_kinds; ++kind) {
        size_t blk = (size_t)p->block_size * p->n_kv_heads * p->row_bytes[kind];
        memmove(addr(p, l, kind, dst[i], 0, 0), addr(p, l, kind, src[i], 0, 0), blk);
      }
  }
  return rc;
}

/* Maximal same-slab runs of a block-table row list, in logical order
 * [SLAB, touch point 3].  Writes the start index of each run; returns the count. */
int oracle_slab_runs(const int32_t* rows, int n, int slab_blocks, int32_t* starts) {
  int runs = 0;
  for (int i = 0; i < n; ++i) {
    if (i == 0 || rows[i] / slab_blocks != rows[i - 1] / slab_blocks) starts[runs++] = i;
  }
  return runs;
}

/* gather_visible [SLAB, touch point 3]: the visible context of one sequence as
 * dense [Hkv, ctx, row] arrays, built run by run: each maximal same-slab run of
 * the block-table row list is taken from its slab and the runs are concatenated
 * in logical order. meta outputs are ignored for the native format. */
int oracle_gather_visible(const oracle_pool* p, int layer, const int32_t* bt_row, int ctx,
                          uint8_t* k_out, uint8_t* v_out, uint8_t* km_out, uint8_t* vm_out) {
  if (layer < 0 || layer >= p->n_layers || ctx < 0) return OR_ERR_ARG;
  const int bs = p->block_size;
  int nblk = (ctx + bs - 1) / bs;
  for (int j = 0; j < nblk; ++j)
    if (!row_ok(p, bt_row[j])) return OR_ERR_RANGE;
  int32_t* starts = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nblk + 1));
  if (!starts) return OR_ERR_MEM;
  int nruns = oracle_slab_runs(bt_row, nblk, p->slab_blocks, starts);
  starts[nruns] = nblk;
  uint8_t* outs[4] = {k_out, v_out, km_out, vm_out};
  for (int kind = 0; kind < p->n_kinds; ++kind) {
    size_t rb = p->row_bytes[kind];
    for (int run = 0; run < nruns; ++run) {
      /* one "take" of rows starts[run]..starts[run+1]-1 from a single slab */
      for (int j = starts[run]; j < starts[run + 1]; ++j)
        for (int slot = 0; slot < bs; ++slot) {
          int t = j * bs + slot;
          if (t >= ctx) break;
          for (int h = 0; h < p->n_kv_heads; ++h)
            memcpy(outs[kind] + ((size_t)h * ctx + t) * rb, addr(p, layer, kind, bt_row[j], slot, h), rb);
        }
    }
  }
  free(starts);
  return OR_OK;
}

/* Dequantised (FP64) K and V of one (layer, row, slot, head), in the stored basis
 * (rotated for packed K). */
static void load_kv(const oracle_pool* p, int layer, int32_t row, int slot, int head, double* kd,
                    double* vd) {
  const int D = p->head_dim;
  if (p->format == OR_FMT_BF16) {
    const uint16_t* kr = (const uint16_t*)addr(p, layer, 0, row, slot, head);
    const uint16_t* vr = (const uint16_t*)addr(p, layer, 1, row, slot, head);
    for (int d = 0; d < D; ++d) { kd[d] = bf16_to_double(kr[d]); vd[d] = bf16_to_double(vr[d]); }
    return;
  }
  oracle_dequantize(addr(p, layer, 0, row, slot, head), (const float*)addr(p, layer, 2, row, slot, head),
                    D, p->k_bits, p->group_size, kd);
  oracle_dequantize(addr(p, layer, 1, row, slot, head), (const float*)addr(p, layer, 3, row, slot, head),
                    D, p->v_bits, p->group_size, vd);
}

/* One (sequence, query head) of paged decode attention, in FP64.  Single query
 * token, no mask, over tokens [0, L) [ATTN, Edge cases].  Plain two-pass softmax:
 *   z_t = scale * (q~ . k^_t), m = max z, p_t = exp(z_t - m),
 *   out = sum_t p_t v^_t / sum_t p_t.
 * For packed formats q~ = R q with the same basis as K, so q~.k~ = q.k. */
static void attend_one(const oracle_pool* p, int layer, const double* qrot, const int32_t* bt_row,
                       int L, int kvh, double scale, double* out) {
  const int D = p->head_dim, bs = p->block_size;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0) return;
  double* z = (double*)malloc(sizeof(double) * (size_t)L);
  double* kd = (double*)malloc(sizeof(double) * (size_t)D);
  double* vd = (double*)malloc(sizeof(double) * (size_t)D);
  double m = -INFINITY;
  for (int t = 0; t < L; ++t) {
    load_kv(p, layer, bt_row[t / bs], t % bs, kvh, kd, vd);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qrot[d] * kd[d];
    z[t] = scale * dot;
    if (z[t] > m) m = z[t];
  }
  double den = 0.0;
  for (int t = 0; t < L; ++t) {
    double pt = exp(z[t] - m);
    den += pt;
    load_kv(p, layer, bt_row[t / bs], t % bs, kvh, kd, vd);
    for (int d = 0; d < D; ++d) out[d] += pt * vd[d];
  }
  for (int d = 0; d < D; ++d) out[d] /= den;
  free(z);
  free(kd);
  free(vd);
}

/* Batched paged decode attention with GQA [ATTN, Current Behavior /
 * Proposed Solution: paged_batch_decode_attention behind KVCache::attend].
 * q: [B, Hq, D] bf16 (un-rotated); bt: [B, max_blocks]; ctx: [B];
 * out: [B, Hq, D] FP64.  n_threads <= 0 means the OpenMP default. */
int oracle_decode_attention(const oracle_pool* p, int layer, int B, int Hq, const uint16_t* q,
                            const int32_t* bt, int max_blocks, const int32_t* ctx, double scale,
                            double* out, int n_threads) {
  if (layer < 0 || layer >= p->n_layers || B < 0 || Hq <= 0 || Hq % p->n_kv_heads) return OR_ERR_ARG;
  const int D = p->head_dim, G = Hq / p->n_kv_heads;
  for (int b = 0; b < B; ++b) {
    if (ctx[b] < 0 || ctx[b] > max_blocks * p->block_size) return OR_ERR_RANGE;
    for (int j = 0; j < (ctx[b] + p->block_size - 1) / p->block_size; ++j)
      if (!row_ok(p, bt[(size_t)b * max_blocks + j])) return OR_ERR_RANGE;
  }
  long total = (long)B * Hq;
#ifdef _OPENMP
  if (n_threads > 0) {
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
    for (long i = 0; i < total; ++i) {
      int b = (int)(i / Hq), h = (int)(i % Hq);
      double qd[512], qr[512];
      for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[((size_t)b * Hq + h) * D + d]);
      if (p->format == OR_FMT_BF16) memcpy(qr, qd, sizeof(double) * (size_t)D);
      else oracle_rotate_q(qd, D, p->signs, qr);
      attend_one(p, layer, qr, bt + (size_t)b * max_blocks, ctx[b], h / G, scale,
                 out + ((size_t)b * Hq + h) * D);
    }
    return OR_OK;
  }
#endif
  for (long i = 0; i < total; ++i) {
    int b = (int)(i / Hq), h = (int)(i % Hq);
    double qd[512], qr[512];
    for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[((size_t)b * Hq + h) * D + d]);
    if (p->format == OR_FMT_BF16) memcpy(qr, qd, sizeof(double) * (size_t)D);
    else oracle_rotate_q(qd, D, p->signs, qr);
    attend_one(p, layer, qr, bt + (size_t)b * max_blocks, ctx[b], h / G, scale,
               out + ((size_t)b * Hq + h) * D);
  }
  return OR_OK;
}

/* Causal chunked-prefill attention [ATTN, Proposed Solution: attend = update the
 * storage, then attention over it; Implementation Notes, edge cases: a masked
 * (prefill) step runs attention with a causal mask, not the single-token path].
 * Sequence b holds ctx[b] tokens, the last n_q of which are the chunk's new tokens
 * (already written); query i of the chunk (position ctx[b] - n_q + i) attends to
 * tokens [0, ctx[b] - n_q + i] of its sequence, with the same softmax(q K^T scale) V
 * as decode.  q: [B, n_q, Hq, D] bf16; out: [B, n_q, Hq, D] FP64.  A sequence with
 * fewer than n_q tokens is an argument error. */
int oracle_prefill_attention(const oracle_pool* p, int layer, int B, int n_q, int Hq, const uint16_t* q,
                             const int32_t* bt, int max_blocks, const int32_t* ctx, double scale, double* out) {
  if (layer < 0 || layer >= p->n_layers || B < 0 || n_q <= 0 || Hq <= 0 || Hq % p->n_kv_heads) return OR_ERR_ARG;
  const int D = p->head_dim, G = Hq / p->n_kv_heads;
  for (int b = 0; b < B; ++b) {
    if (ctx[b] < n_q || ctx[b] > max_blocks * p->block_size) return OR_ERR_RANGE;
    for (int j = 0; j < (ctx[b] + p->block_size - 1) / p->block_size; ++j)
      if (!row_ok(p, bt[(size_t)b * max_blocks + j])) return OR_ERR_RANGE;
  }
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < n_q; ++i) {
      const int visible = ctx[b] - n_q + i + 1;
      for (int h = 0; h < Hq; ++h) {
        double qd[512], qr[512];
        const size_t row = (((size_t)b * n_q + i) * Hq + h) * D;
        for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(q[row + d]);
        if (p->format == OR_FMT_BF16) memcpy(qr, qd, sizeof(double) * (size_t)D);
        else oracle_rotate_q(qd, D, p->signs, qr);
        attend_one(p, layer, qr, bt + (size_t)b * max_blocks, visible, h / G, scale, out + row);
      }
    }
  return OR_OK;
}

/* Block record [SLAB, touch point 6 (serde block content, restore path); PACK,
 * Summary (a full checkpoint keeps the packed bytes unchanged)]: every stored byte of one
 * block, for each layer in order and, within a layer, for each stored tensor in
 * the order K, V, K meta, V meta, the block's [block_size][n_kv_heads][row]
 * bytes as stored.  Nothing is converted. */
size_t oracle_record_bytes(const oracle_pool* p) {
  size_t per_layer = 0;
  for (int kind = 0; kind < p->n_kinds; ++kind) per_layer += (size_t)p->block_size * p->n_kv_heads * p->row_bytes[kind];
  return per_layer * (size_t)p->n_layers;
}

/* export: the records of rows[0..n) one after another in list order. */
int oracle_export_blocks(const oracle_pool* p, int n, const int32_t* rows, uint8_t* out) {
  for (int i = 0; i < n; ++i)
    if (!row_ok(p, rows[i])) return OR_ERR_RANGE;
  uint8_t* o = out;
  for (int i = 0; i < n; ++i)
    for (int l = 0; l < p->n_layers; ++l)
      for (int kind = 0; kind < p->n_kinds; ++kind) {
        size_t blk = (size_t)p->block_size * p->n_kv_heads * p->row_bytes[kind];
        memcpy(o, addr(p, l, kind, rows[i], 0, 0), blk);
        o += blk;
      }
  return OR_OK;
}

/* import (restore): record i is written back into block rows[i]. */
int oracle_import_blocks(oracle_pool* p, int n, const int32_t* rows, const uint8_t* in) {
  for (int i = 0; i < n; ++i)
    if (!row_ok(p, rows[i])) return OR_ERR_RANGE;
  const uint8_t* r = in;
  for (int i = 0; i < n; ++i)
    for (int l = 0; l < p->n_layers; ++l)
      for (int kind = 0; kind < p->n_kinds; ++kind) {
        size_t blk = (size_t)p->block_size * p->n_kv_heads * p->row_bytes[kind];
        memcpy(addr(p, l, kind, rows[i], 0, 0), r, blk);
        r += blk;
      }
  return OR_OK;
}

/* Raw bytes of one (layer, kind, row) block, for tests. */
int oracle_read_block(const oracle_pool* p, int layer, int kind, int32_t row, uint8_t* out) {
  if (layer < 0 || layer >= p->n_layers || kind < 0 || kind >= p->n_kinds || !row_ok(p, row))
    return OR_ERR_ARG;
  memcpy(out, addr(p, layer, kind, row, 0, 0),
         (size_t)p->block_size * p->n_kv_heads * p->row_bytes[kind]);
  return OR_OK;
}

/* Raw bytes of one whole slab (layer, kind, slab index), for layout tests. */
int oracle_read_slab(const oracle_pool* p, int layer, int kind, int slab, uint8_t* out) {
  if (layer < 0 || layer >= p->n_layers || kind < 0 || kind >= p->n_kinds || slab < 0 ||
      slab >= p->n_slabs)
    return OR_ERR_ARG;
  memcpy(out, p->slab[((long)slab * p->n_layers + layer) * p->n_kinds + kind], slab_bytes(p, kind));
  return OR_OK;
}
