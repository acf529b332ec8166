// write.cu — write_block (native copy or quantise-once), copy_on_write_block and
// gather_visible kernels.
//
//  write_block: mlxcel #235 touch point 1 (the row's slab is the target);
//    packed formats follow mlx-swift-lm #142 (Summary: token-local affine groups
//    with FP32 scale/offset, fixed signed Hadamard basis on K; After flowchart:
//    new K/V quantised a single time, when written).
//  copy_on_write_block: mlxcel #235 touch point 2.
//  gather_visible: mlxcel #235 touch point 3.  The page splits the row list into
//    maximal same-slab runs because one gather op cannot span tensors; here every
//    block's source slab comes from the per-slab pointer table, so one launch
//    produces the concatenation of all runs in logical order.
#include <cuda_runtime.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

__device__ __forceinline__ uint8_t* row_addr(const LayerView& lv, int kind, int32_t row, int slot, int head) {
  const int32_t slab = row / lv.slab_blocks;
  const int32_t r = row - slab * lv.slab_blocks;
  uint8_t* base = lv.tab.base[(size_t)slab * lv.tab.stride + kind];
  return base + ((size_t)(r * kBlockTokens + slot) * lv.hkv + head) * (size_t)lv.row_bytes[kind];
}

__device__ __forceinline__ bool row_ok(const LayerView& lv, int32_t row) {
  return row >= 0 && (int64_t)row < lv.rows_capacity;
}

// Native bf16: copy one (token, head) K and V row; one warp per (token, head).
template <int D>
__global__ void __launch_bounds__(256) write_bf16_kernel(LayerView lv, int n, const int32_t* __restrict__ rows,
                                                         const int32_t* __restrict__ slots,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (int64_t)n * lv.hkv) return;
  const int i = (int)(wid / lv.hkv), h = (int)(wid % lv.hkv);
  const int32_t row = rows[i], slot = slots[i];
  if (!row_ok(lv, row) || slot < 0 || slot >= kBlockTokens) {
    if (lane == 0) atomicOr(lv.err, row_ok(lv, row) ? ERR_SLOT : ERR_ROW);
    return;
  }
  constexpr int CH = D * 2 / 16;  // 16-byte chunks per row
  const uint4* ks = reinterpret_cast<const uint4*>(k + ((size_t)i * lv.hkv + h) * D);
  const uint4* vs = reinterpret_cast<const uint4*>(v + ((size_t)i * lv.hkv + h) * D);
  uint4* kd = reinterpret_cast<uint4*>(row_addr(lv, PKV_KIND_K, row, slot, h));
  uint4* vd = reinterpret_cast<uint4*>(row_addr(lv, PKV_KIND_V, row, slot, h));
  for (int c = lane; c < CH; c += 32) {
    kd[c] = ks[c];
    vd[c] = vs[c];
  }
}

// Quantise E consecutive values per lane (lane owns dims [lane*E, lane*E+E)) to
// `BITS`-bit codes with groups of GS dims (GS/E lanes per group) and store codes
// and (scale, offset).  All arithmetic is IEEE single precision, one rounding per
// operation, so the codes match a plain sequential CPU statement bit for bit.
template <int E, int BITS, int GS>
__device__ __forceinline__ void quantise_store(const float (&x)[E], uint8_t* code_row, float* meta_row, int lane) {
  constexpr int LPG = GS / E;  // lanes per group
  static_assert(LPG >= 1 && LPG <= 32, "group geometry");
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int e = 1; e < E; ++e) {
    mn = fminf(mn, x[e]);
    mx = fmaxf(mx, x[e]);
  }
#pragma unroll
  for (int off = 1; off < LPG; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  constexpr int TOP = (1 << BITS) - 1;
  const float scale = __fdiv_rn(__fsub_rn(mx, mn), (float)TOP);
  int c[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int q = 0;
    if (scale != 0.0f) {
      q = __float2int_rn(__fdiv_rn(__fsub_rn(x[e], mn), scale));
      q = q < 0 ? 0 : (q > TOP ? TOP : q);
    }
    c[e] = q;
  }
  if (BITS == 8) {
#pragma unroll
    for (int e = 0; e < E; ++e) code_row[lane * E + e] = (uint8_t)c[e];
  } else {
#pragma unroll
    for (int e = 0; e < E; e += 2) code_row[(lane * E + e) / 2] = (uint8_t)((c[e] & 15) | ((c[e + 1] & 15) << 4));
  }
  if ((lane % LPG) == 0) {
    const int g = lane / LPG;
    meta_row[2 * g] = scale;
    meta_row[2 * g + 1] = mn;
  }
}

// Packed formats: one warp per (token, head).  K is rotated by R = H diag(s) /
// sqrt(D) with a fast Walsh-Hadamard transform in FP64 (the +-1 sums are exact for
// bf16 rows whose binary-exponent spread is at most 45 - log2(D), so the order of
// the butterflies does not matter), multiplied by 1/sqrt(D) in FP64 and rounded
// once to FP32; V is quantised as stored.
template <int D, int KBITS, int VBITS, int GS>
__global__ void __launch_bounds__(256) write_packed_kernel(LayerView lv, int n, const int32_t* __restrict__ rows,
                                                           const int32_t* __restrict__ slots,
                                                           const uint16_t* __restrict__ k,
                                                           const uint16_t* __restrict__ v,
                                                           const float* __restrict__ signs, double inv_sqrt_d) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (wid >= (int64_t)n * lv.hkv) return;
  const int i = (int)(wid / lv.hkv), h = (int)(wid % lv.hkv);
  const int32_t row = rows[i], slot = slots[i];
  if (!row_ok(lv, row) || slot < 0 || slot >= kBlockTokens) {
    if (lane == 0) atomicOr(lv.err, row_ok(lv, row) ? ERR_SLOT : ERR_ROW);
    return;
  }
  const uint16_t* kr = k + ((size_t)i * lv.hkv + h) * D + lane * E;
  const uint16_t* vr = v + ((size_t)i * lv.hkv + h) * D + lane * E;
  double xd[E];
#pragma unroll
  for (int e = 0; e < E; ++e) xd[e] = (double)__uint_as_float((uint32_t)kr[e] << 16) * (double)signs[lane * E + e];
  // In-lane butterflies (stride h < E).
#pragma unroll
  for (int hs = 1; hs < E; hs <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & hs) == 0) {
        const double a = xd[e], b = xd[e + hs];
        xd[e] = a + b;
        xd[e + hs] = a - b;
      }
    }
  }
  // Cross-lane butterflies (stride h = E * m, partner lane ^ m).
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const double other = __shfl_xor_sync(0xffffffffu, xd[e], m);
      xd[e] = upper ? (other - xd[e]) : (xd[e] + other);
    }
  }
  float xk[E], xv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    xk[e] = __double2float_rn(__dmul_rn(xd[e], inv_sqrt_d));
    xv[e] = __uint_as_float((uint32_t)vr[e] << 16);
  }
  quantise_store<E, KBITS, GS>(xk, row_addr(lv, PKV_KIND_K, row, slot, h),
                           reinterpret_cast<float*>(row_addr(lv, PKV_KIND_KMETA, row, slot, h)), lane);
  quantise_store<E, VBITS, GS>(xv, row_addr(lv, PKV_KIND_V, row, slot, h),
                           reinterpret_cast<float*>(row_addr(lv, PKV_KIND_VMETA, row, slot, h)), lane);
}

template <int D>
cudaError_t launch_write_d(const LayerView& lv, int fmt, int group, int n, const int32_t* rows, const int32_t* slots,
                           const uint16_t* k, const uint16_t* v, const float* signs, double inv, cudaStream_t s) {
  const int64_t warps = (int64_t)n * lv.hkv;
  // A step's write (a few tokens) runs one warp per CTA, so its warps spread over
  // the SMs: the packed kernel's FP64 butterflies are throughput-bound per SM.
  const int threads = warps < 4096 ? 32 : 256;
  const unsigned grid = (unsigned)((warps * 32 + threads - 1) / threads);
  switch (fmt) {
    case PKV_FMT_BF16: write_bf16_kernel<D><<<grid, threads, 0, s>>>(lv, n, rows, slots, k, v); break;
    case PKV_FMT_K4V4:
      if (D >= 128 && group == kGroupWide)
        write_packed_kernel<D, 4, 4, (D >= 128 ? kGroupWide : kGroup)><<<grid, threads, 0, s>>>(lv, n, rows, slots, k,
                                                                                               v, signs, inv);
      else
        write_packed_kernel<D, 4, 4, kGroup><<<grid, threads, 0, s>>>(lv, n, rows, slots, k, v, signs, inv);
      break;
    case PKV_FMT_K8V4: write_packed_kernel<D, 8, 4, kGroup><<<grid, threads, 0, s>>>(lv, n, rows, slots, k, v, signs, inv); break;
    default: write_packed_kernel<D, 8, 8, kGroup><<<grid, threads, 0, s>>>(lv, n, rows, slots, k, v, signs, inv); break;
  }
  return cudaGetLastError();
}

// copy_on_write_block: CTAs stride over (pair, layer, kind) pieces; each thread
// keeps four 16-byte loads in flight before storing them.
__global__ void __launch_bounds__(256) copy_blocks_kernel(const uint8_t* const* __restrict__ table, int n_layers,
                                                          int n_kinds, int64_t b0, int64_t b1, int64_t b2, int64_t b3,
                                                          int slab_blocks, int64_t rows_capacity, int n,
                                                          const int32_t* __restrict__ src,
                                                          const int32_t* __restrict__ dst, int32_t* err) {
  const int ppb = n_layers * n_kinds;  // pieces per pair; also the pointer-table stride per slab
  const int64_t pieces = (int64_t)n * ppb;
  constexpr int U = 4;
  for (int64_t pc = blockIdx.x; pc < pieces; pc += gridDim.x) {
    const int pair = (int)(pc / ppb), lk = (int)(pc - (int64_t)pair * ppb);
    const int kind = lk % n_kinds;
    const int64_t bytes = kind == 0 ? b0 : kind == 1 ? b1 : kind == 2 ? b2 : b3;
    const int32_t rs = src[pair], rd = dst[pair];
    if (rs < 0 || rd < 0 || (int64_t)rs >= rows_capacity || (int64_t)rd >= rows_capacity) {
      if (threadIdx.x == 0 && lk == 0) atomicOr(err, ERR_ROW);
      continue;
    }
    const uint4* sp = reinterpret_cast<const uint4*>(table[(size_t)(rs / slab_blocks) * ppb + (size_t)lk] +
                                                     (int64_t)(rs % slab_blocks) * bytes);
    uint4* dp = reinterpret_cast<uint4*>(const_cast<uint8_t*>(table[(size_t)(rd / slab_blocks) * ppb + (size_t)lk]) +
                                         (int64_t)(rd % slab_blocks) * bytes);
    const int64_t chunks = bytes / 16;
    int64_t c = threadIdx.x;
    for (; c + (U - 1) * (int64_t)blockDim.x < chunks; c += U * (int64_t)blockDim.x) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = sp[c + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) dp[c + u * blockDim.x] = v[u];
    }
    for (; c < chunks; c += blockDim.x) dp[c] = sp[c];
  }
}

// export / import of block records.  A record holds every stored byte of one
// block, layer-major, then kind (K, V, K meta, V meta), each the block's
// [32 tokens][Hkv][row] bytes as stored.  Work item = one (block, layer, kind)
// piece; CTAs stride over the pieces, and each thread keeps four 16-byte loads in
// flight before storing them.
__global__ void __launch_bounds__(256) serde_blocks_kernel(const uint8_t* const* __restrict__ table, int n_layers,
                                                           int n_kinds, int64_t b0, int64_t b1, int64_t b2,
                                                           int64_t b3, int slab_blocks, int64_t rows_capacity,
                                                           int n, const int32_t* __restrict__ rows, uint8_t* buf,
                                                           int64_t rec_bytes, int to_pool, int32_t* err) {
  const int64_t per_layer = b0 + b1 + (n_kinds == 4 ? b2 + b3 : 0);
  const int ppb = n_layers * n_kinds;  // pieces per block; also the pointer-table stride per slab
  const int64_t pieces = (int64_t)n * ppb;
  constexpr int U = 4;
  for (int64_t pc = blockIdx.x; pc < pieces; pc += gridDim.x) {
    const int i = (int)(pc / ppb), lk = (int)(pc - (int64_t)i * ppb);
    const int layer = lk / n_kinds, kind = lk - layer * n_kinds;
    const int32_t r = rows[i];
    if (r < 0 || (int64_t)r >= rows_capacity) {
      if (threadIdx.x == 0 && lk == 0) atomicOr(err, ERR_ROW);
      continue;
    }
    const int64_t bytes = kind == 0 ? b0 : kind == 1 ? b1 : kind == 2 ? b2 : b3;
    const int64_t koff = kind == 0 ? 0 : kind == 1 ? b0 : kind == 2 ? b0 + b1 : b0 + b1 + b2;
    uint8_t* blk = const_cast<uint8_t*>(table[(size_t)(r / slab_blocks) * ppb + (size_t)lk]) +
                   (int64_t)(r % slab_blocks) * bytes;
    uint8_t* rec = buf + (int64_t)i * rec_bytes + (int64_t)layer * per_layer + koff;
    uint4* dp = reinterpret_cast<uint4*>(to_pool ? blk : rec);
    const uint4* sp = reinterpret_cast<const uint4*>(to_pool ? rec : blk);
    const int64_t chunks = bytes / 16;
    int64_t c = threadIdx.x;
    for (; c + (U - 1) * (int64_t)blockDim.x < chunks; c += U * (int64_t)blockDim.x) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = sp[c + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) dp[c + u * blockDim.x] = v[u];
    }
    for (; c < chunks; c += blockDim.x) dp[c] = sp[c];
  }
}

// Chunked prefill as decode of virtual sequences: queries nq s .. nq s + nq - 1 of
// sequence b's chunk of n_q new tokens become virtual sequence b * (n_q / nq) + s,
// holding the first ctx[b] - n_q + nq (s + 1) tokens of b through b's block-table
// row (the last of those queries' causal limit; the kernel masks the earlier ones).
// A sequence with fewer than n_q tokens sets the error word (context bit) and its
// queries see no token.
__global__ void expand_prefill_kernel(int B, int n_q, int nq, int max_blocks, const int32_t* __restrict__ bt,
                                      const int32_t* __restrict__ ctx, int32_t* __restrict__ bt_out,
                                      int32_t* __restrict__ ctx_out, int32_t* err) {
  const int S = n_q / nq;  // virtual sequences per sequence
  const int64_t nv = (int64_t)B * S;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t first = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t idx = first; idx < nv * max_blocks; idx += stride) {
    const int64_t v = idx / max_blocks, j = idx - v * max_blocks;
    bt_out[idx] = bt[(v / S) * max_blocks + j];
  }
  for (int64_t v = first; v < nv; v += stride) {
    const int b = (int)(v / S), sub = (int)(v - (int64_t)b * S);
    const int32_t L = ctx[b];
    int32_t vis = L - n_q + nq * (sub + 1);
    if (L < n_q) {
      atomicOr(err, ERR_CTX);
      vis = 0;
    }
    ctx_out[v] = vis;
  }
}

// gather_visible: blockIdx.y = kind; grid-stride over (head, token, 16-B chunk).
__global__ void gather_kernel(LayerView lv, const int32_t* __restrict__ bt_row, int ctx, uint8_t* o0, uint8_t* o1,
                              uint8_t* o2, uint8_t* o3) {
  const int kind = blockIdx.y;
  uint8_t* out = kind == 0 ? o0 : kind == 1 ? o1 : kind == 2 ? o2 : o3;
  const int rb = lv.row_bytes[kind];
  const int ch = rb / 16;
  const int64_t total = (int64_t)lv.hkv * ctx * ch;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % ch);
    const int64_t ht = idx / ch;
    const int t = (int)(ht % ctx);
    const int h = (int)(ht / ctx);
    const int32_t row = bt_row[t / kBlockTokens];
    if (!row_ok(lv, row)) {
      if (c == 0) atomicOr(lv.err, ERR_ROW);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(row_addr(lv, kind, row, t % kBlockTokens, h));
    reinterpret_cast<uint4*>(out + ((int64_t)h * ctx + t) * rb)[c] = src[c];
  }
}

}  // namespace

cudaError_t launch_write(const LayerView& lv, int fmt, int D, int group, int n, const int32_t* rows,
                         const int32_t* slots, const uint16_t* k, const uint16_t* v, const float* signs,
                         double inv_sqrt_d, cudaStream_t s) {
  switch (D) {
    case 64: return launch_write_d<64>(lv, fmt, group, n, rows, slots, k, v, signs, inv_sqrt_d, s);
    case 128: return launch_write_d<128>(lv, fmt, group, n, rows, slots, k, v, signs, inv_sqrt_d, s);
    default: return launch_write_d<256>(lv, fmt, group, n, rows, slots, k, v, signs, inv_sqrt_d, s);
  }
}

static int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  return sms;
}

cudaError_t launch_copy_blocks(const uint8_t* const* table, int n_layers, int n_kinds, const int64_t* block_bytes,
                               int slab_blocks, int64_t rows_capacity, int n, const int32_t* src,
                               const int32_t* dst, int32_t* err, cudaStream_t s) {
  const int64_t pieces = (int64_t)n * n_layers * n_kinds;
  const int64_t cap = 8LL * sm_count();  // eight 256-thread CTAs per SM
  const int64_t grid = pieces < cap ? pieces : cap;
  copy_blocks_kernel<<<(unsigned)grid, 256, 0, s>>>(table, n_layers, n_kinds, block_bytes[0], block_bytes[1],
                                                    block_bytes[2], block_bytes[3], slab_blocks, rows_capacity, n,
                                                    src, dst, err);
  return cudaGetLastError();
}

cudaError_t launch_serde_blocks(const uint8_t* const* table, int n_layers, int n_kinds, const int64_t* block_bytes,
                               int slab_blocks, int64_t rows_capacity, int n, const int32_t* rows, uint8_t* buf,
                               int64_t rec_bytes, int to_pool, int32_t* err, cudaStream_t s) {
  const int64_t pieces = (int64_t)n * n_layers * n_kinds;
  const int64_t cap = 8LL * sm_count();  // eight 256-thread CTAs per SM
  const int64_t grid = pieces < cap ? pieces : cap;
  serde_blocks_kernel<<<(unsigned)grid, 256, 0, s>>>(table, n_layers, n_kinds, block_bytes[0], block_bytes[1],
                                                     block_bytes[2], block_bytes[3], slab_blocks, rows_capacity, n,
                                                     rows, buf, rec_bytes, to_pool, err);
  return cudaGetLastError();
}

cudaError_t launch_expand_prefill(int B, int n_q, int nq, int max_blocks, const int32_t* bt, const int32_t* ctx,
                                  int32_t* bt_out, int32_t* ctx_out, int32_t* err, cudaStream_t s) {
  const int64_t work = (int64_t)B * (n_q / nq) * (max_blocks > 1 ? max_blocks : 1);
  int64_t grid = (work + 255) / 256;
  if (grid > 8LL * sm_count()) grid = 8LL * sm_count();
  if (grid < 1) grid = 1;
  expand_prefill_kernel<<<(unsigned)grid, 256, 0, s>>>(B, n_q, nq, max_blocks, bt, ctx, bt_out, ctx_out, err);
  return cudaGetLastError();
}

cudaError_t launch_gather(const LayerView& lv, const int32_t* bt_row, int ctx, uint8_t* const* outs, cudaStream_t s) {
  const int threads = 256;
  const int64_t total = (int64_t)lv.hkv * ctx * (lv.row_bytes[0] / 16);
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  dim3 grid((unsigned)blocks, (unsigned)lv.n_kinds);
  gather_kernel<<<grid, threads, 0, s>>>(lv, bt_row, ctx, outs[0], outs[1], outs[2], outs[3]);
  return cudaGetLastError();
}

}  // namespace pkv
