// pool.cu — host runtime of the chunked-slab pool and the C ABI entry points.
//
// Storage follows mlxcel issue #235 ("chunked slab storage for the paged pool"):
// per layer and stored tensor a vector of fixed-size slabs
// [slab_blocks, block_size, n_kv_heads, row]; row -> (row / slab_blocks,
// row % slab_blocks); growth appends fresh zeroed slabs, never copying or
// freeing existing ones (Proposed solution, bullets 1-2), and the slab-append
// counter and reserved bytes are sums over slabs (touch point 5).  Block ids,
// refcounts and free-row reuse stay row-level concepts (Behavioral invariants).
//
// One allocation ("slab group") holds slab s of every layer and tensor; the
// device pointer table still has one entry per (slab, layer, tensor), which is
// what every kernel reads (touch point 4: per-slab base pointers; touch point 7:
// one mapping helper).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "pkv_internal.cuh"

using namespace pkv;

struct pkv_pool {
  pkv_pool_config cfg{};
  pkv_allocator alloc{};
  bool default_alloc = true;
  int device = 0;
  int n_sm = 0;
  size_t smem_optin = 0;
  int n_kinds = 2;
  int64_t row_bytes[4] = {0, 0, 0, 0};
  int64_t slab_bytes[4] = {0, 0, 0, 0};  // one slab of one layer, per kind
  int64_t group_bytes = 0;               // one slab index across layers and kinds
  int64_t layer_bytes = 0;               // one slab of one layer, all kinds
  int64_t maps_offset = 0;               // tensor maps at the group's tail
  std::vector<void*> groups;             // allocation per slab index
  uint8_t** table_host = nullptr;        // pinned [max_slabs][n_layers][n_kinds]
  uint8_t** table_dev = nullptr;
  int32_t* err_dev = nullptr;
  float* signs_dev = nullptr;            // [head_dim] +-1
  double inv_sqrt_d = 0.0;
  std::vector<int32_t> refcount;
  std::vector<int32_t> free_rows;        // LIFO
  int64_t rows_in_use = 0;
  int64_t append_events = 0;
  int decode_ctas = 0;
  cudaStream_t last_stream = nullptr;
};

static thread_local std::string g_last_error;

namespace pkv {
// Defined in write.cu.
cudaError_t launch_expand_prefill(int B, int n_q, int nq, int max_blocks, const int32_t* bt, const int32_t* ctx,
                                  int32_t* bt_out, int32_t* ctx_out, int32_t* err, cudaStream_t s);
cudaError_t launch_serde_blocks(const uint8_t* const* table, int n_layers, int n_kinds, const int64_t* block_bytes,
                               int slab_blocks, int64_t rows_capacity, int n, const int32_t* rows, uint8_t* buf,
                               int64_t rec_bytes, int to_pool, int32_t* err, cudaStream_t s);
void set_last_error(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace pkv

static pkv_status cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return PKV_ERR_CUDA;
}

#define PKV_CUDA(call, where)                      \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

// splitmix64 (Steele, Lea & Flood 2014): output for state x.
static uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static LayerView layer_view(const pkv_pool* p, int layer) {
  LayerView lv;
  lv.tab.base = p->table_dev + (size_t)layer * p->n_kinds;
  lv.tab.stride = p->cfg.n_layers * p->n_kinds;
  lv.n_kinds = p->n_kinds;
  lv.hkv = p->cfg.n_kv_heads;
  lv.slab_blocks = p->cfg.slab_blocks;
  lv.rows_capacity = (int64_t)p->groups.size() * p->cfg.slab_blocks;
  for (int k = 0; k < 4; ++k) lv.row_bytes[k] = (int)p->row_bytes[k];
  lv.err = p->err_dev;
  lv.map_delta = p->maps_offset - (int64_t)layer * p->layer_bytes + (int64_t)layer * p->n_kinds * 128;
  for (int k = 0; k < 4; ++k)
    lv.box_bytes[k] = k < p->n_kinds ? tma_box_bytes(p->row_bytes[k] * p->cfg.n_kv_heads) : 0;
  return lv;
}

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  }
  return fn;
}

// Tensor maps of one slab group: for every layer and stored tensor, the slab
// [slab_blocks * 32 tokens][Hkv * row] bytes viewed in 3-D as [column block][token]
// [W bytes] (W = box_bytes), read in boxes of 16 tokens x the whole row, which land
// as row/W boxes of 16 x W bytes with the matching shared-memory swizzle.
static bool encode_group_maps(const pkv_pool* p, uint8_t* group, std::vector<CUtensorMap>& maps) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const int L = p->cfg.n_layers, K = p->n_kinds;
  maps.resize((size_t)L * K);
  int64_t off = 0;
  for (int l = 0; l < L; ++l)
    for (int k = 0; k < K; ++k) {
      const int64_t row = p->row_bytes[k] * p->cfg.n_kv_heads;
      const int box = tma_box_bytes(row);
      const CUtensorMapSwizzle sw = box == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                    : box == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                    : box == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
      // 3-D view [column block][token][W bytes] of the [token][row] tensor: one copy
      // moves 16 tokens of the whole row and lands as nx boxes of 16 x W bytes.
      const cuuint64_t nx = (cuuint64_t)(row / box);
      const cuuint64_t dims[3] = {(cuuint64_t)box, (cuuint64_t)p->cfg.slab_blocks * kBlockTokens, nx};
      const cuuint64_t strides[2] = {(cuuint64_t)row, (cuuint64_t)box};
      const cuuint32_t boxd[3] = {(cuuint32_t)box, 16u, (cuuint32_t)nx};
      const cuuint32_t estr[3] = {1u, 1u, 1u};
      if (enc(&maps[(size_t)l * K + k], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, group + off, dims, strides, boxd, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
      off += p->slab_bytes[k];
    }
  return true;
}

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_OOM: return "allocation failed (pool unchanged)";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_FORMAT: return "storage identity / format mismatch";
    case PKV_ERR_RANGE: return "index out of range";
    case PKV_ERR_DEVICE: return "device error word set";
  }
  return "unknown status";
}

const char* pkv_last_error(void) { return g_last_error.c_str(); }

pkv_status pkv_pool_create(const pkv_pool_config* cfg, const pkv_allocator* alloc, void* stream,
                           pkv_pool** out) {
  if (!cfg || !out) return PKV_ERR_INVALID;
  *out = nullptr;
  const FormatBits fb = format_bits(cfg->format);
  const int D = cfg->head_dim;
  if (fb.k == 0 || cfg->n_layers < 1 || cfg->n_kv_heads < 1 || cfg->n_kv_heads > 8 ||
      !(D == 64 || D == 128 || D == 256) || cfg->block_size != kBlockTokens || cfg->slab_blocks < 1 ||
      cfg->slab_blocks > 4096 || cfg->max_slabs < 1)
    return PKV_ERR_INVALID;
  // Groups of 32 for every packed format; groups of 64 (the five-bit K4/V4 layout)
  // for K4/V4 with head_dim >= 128, so a (token, head) metadata row stays a whole
  // number of 16-byte chunks.
  if (cfg->format != PKV_FMT_BF16 && cfg->group_size != kGroup &&
      !(cfg->group_size == kGroupWide && cfg->format == PKV_FMT_K4V4 && D >= 128))
    return PKV_ERR_INVALID;
  if (alloc && (!alloc->alloc || !alloc->release)) return PKV_ERR_INVALID;

  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_ERR_OOM;
  p->cfg = *cfg;
  if (cfg->format == PKV_FMT_BF16) p->cfg.group_size = cfg->group_size;
  if (alloc) {
    p->alloc = *alloc;
    p->default_alloc = false;
  }
  p->last_stream = (cudaStream_t)stream;
  auto fail = [&](pkv_status st) {
    pkv_pool_destroy(p);
    return st;
  };
  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaGetDevice"));
  e = cudaDeviceGetAttribute(&p->n_sm, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaDeviceGetAttribute(SM count)"));
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaDeviceGetAttribute(smem)"));
  p->smem_optin = (size_t)optin;

  p->n_kinds = (cfg->format == PKV_FMT_BF16) ? 2 : 4;
  p->row_bytes[PKV_KIND_K] = (int64_t)D * fb.k / 8;
  p->row_bytes[PKV_KIND_V] = (int64_t)D * fb.v / 8;
  if (p->n_kinds == 4) {
    p->row_bytes[PKV_KIND_KMETA] = (int64_t)(D / cfg->group_size) * 2 * sizeof(float);
    p->row_bytes[PKV_KIND_VMETA] = p->row_bytes[PKV_KIND_KMETA];
  }
  const int64_t per_row_tokens = (int64_t)cfg->slab_blocks * kBlockTokens * cfg->n_kv_heads;
  p->layer_bytes = 0;
  for (int k = 0; k < p->n_kinds; ++k) {
    p->slab_bytes[k] = per_row_tokens * p->row_bytes[k];
    p->layer_bytes += p->slab_bytes[k];
  }
  p->group_bytes = p->layer_bytes * cfg->n_layers;
  // Tensor maps (128 bytes each, 64-byte aligned) after the slab data.
  p->maps_offset = (p->group_bytes + 127) / 128 * 128;
  p->group_bytes = p->maps_offset + (int64_t)cfg->n_layers * p->n_kinds * 128;
  for (int k = 0; k < p->n_kinds; ++k)
    if (tma_box_bytes(p->row_bytes[k] * cfg->n_kv_heads) == 0) return fail(PKV_ERR_INVALID);

  const size_t table_entries = (size_t)cfg->max_slabs * cfg->n_layers * p->n_kinds;
  e = cudaMallocHost((void**)&p->table_host, table_entries * sizeof(uint8_t*));
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMallocHost(slab table)"));
  memset(p->table_host, 0, table_entries * sizeof(uint8_t*));
  e = cudaMalloc((void**)&p->table_dev, table_entries * sizeof(uint8_t*));
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMalloc(slab table)"));
  e = cudaMemset(p->table_dev, 0, table_entries * sizeof(uint8_t*));
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMemset(slab table)"));
  e = cudaMalloc((void**)&p->err_dev, 64);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMalloc(error word)"));
  e = cudaMemset(p->err_dev, 0, 64);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMemset(error word)"));

  // Fixed signed Hadamard basis: s_i = -1 iff the top bit of splitmix64(seed + i)
  // is set (mlx-swift-lm #142, Summary: Q and K share one signed Hadamard basis that
  // never changes).
  std::vector<float> signs((size_t)D);
  for (int i = 0; i < D; ++i) signs[i] = (splitmix64(cfg->hadamard_seed + (uint64_t)i) >> 63) ? -1.f : 1.f;
  e = cudaMalloc((void**)&p->signs_dev, sizeof(float) * (size_t)D);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMalloc(signs)"));
  e = cudaMemcpy(p->signs_dev, signs.data(), sizeof(float) * (size_t)D, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail(cuda_fail(e, "cudaMemcpy(signs)"));
  p->inv_sqrt_d = 1.0 / std::sqrt((double)D);
  *out = p;
  return PKV_OK;
}

void pkv_pool_destroy(pkv_pool* p) {
  if (!p) return;
  // Work enqueued on any stream may still read the slabs: wait for the device.
  if (!p->groups.empty()) cudaDeviceSynchronize();
  for (size_t i = 0; i < p->groups.size(); ++i) {
    if (!p->groups[i]) continue;
    if (p->default_alloc)
      cudaFree(p->groups[i]);
    else
      p->alloc.release(p->alloc.ctx, p->groups[i], (void*)p->last_stream);
  }
  if (p->table_dev) cudaFree(p->table_dev);
  if (p->table_host) cudaFreeHost(p->table_host);
  if (p->err_dev) cudaFree(p->err_dev);
  if (p->signs_dev) cudaFree(p->signs_dev);
  delete p;
}

pkv_status pkv_append_slab(pkv_pool* p, int n_slabs, void* stream) {
  if (!p || n_slabs < 0) return PKV_ERR_INVALID;
  if (n_slabs == 0) return PKV_OK;
  const int have = (int)p->groups.size();
  if (have + n_slabs > p->cfg.max_slabs) return PKV_ERR_RANGE;
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<void*> fresh;
  fresh.reserve((size_t)n_slabs);
  for (int i = 0; i < n_slabs; ++i) {
    void* ptr = nullptr;
    if (p->default_alloc) {
      if (cudaMallocAsync(&ptr, (size_t)p->group_bytes, s) != cudaSuccess) {
        cudaGetLastError();
        ptr = nullptr;
      }
    } else {
      ptr = p->alloc.alloc(p->alloc.ctx, (size_t)p->group_bytes, stream);
    }
    if (!ptr) {
      for (void* q : fresh) {
        if (p->default_alloc)
          cudaFreeAsync(q, s);
        else
          p->alloc.release(p->alloc.ctx, q, stream);
      }
      return PKV_ERR_OOM;
    }
    fresh.push_back(ptr);
  }
  // Tensor maps of the new slabs, encoded before anything is enqueued so that a
  // failure leaves the pool unchanged.
  std::vector<std::vector<CUtensorMap>> maps(fresh.size());
  for (size_t i = 0; i < maps.size(); ++i) {
    if (!encode_group_maps(p, (uint8_t*)fresh[i], maps[i])) {
      for (void* q : fresh) {
        if (p->default_alloc)
          cudaFreeAsync(q, s);
        else
          p->alloc.release(p->alloc.ctx, q, stream);
      }
      g_last_error = "cuTensorMapEncodeTiled unavailable or rejected a slab";
      return PKV_ERR_CUDA;
    }
  }
  // Zero the new slabs (a fresh zeros slab), then publish their base pointers.
  for (void* ptr : fresh) PKV_CUDA(cudaMemsetAsync(ptr, 0, (size_t)p->group_bytes, s), "cudaMemsetAsync(slab)");
  // The maps are copied from pageable memory: the call stages the bytes before it
  // returns, so the vectors may go out of scope at once.
  for (size_t i = 0; i < maps.size(); ++i)
    PKV_CUDA(cudaMemcpyAsync((uint8_t*)fresh[i] + p->maps_offset, maps[i].data(),
                             maps[i].size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s),
             "cudaMemcpyAsync(tensor maps)");
  const int L = p->cfg.n_layers, K = p->n_kinds;
  for (int i = 0; i < n_slabs; ++i) {
    uint8_t* g = (uint8_t*)fresh[(size_t)i];
    int64_t off = 0;
    for (int l = 0; l < L; ++l)
      for (int k = 0; k < K; ++k) {
        p->table_host[((size_t)(have + i) * L + l) * K + k] = g + off;
        off += p->slab_bytes[k];
      }
  }
  // The pinned host entries of these slabs are never rewritten, so the copy may
  // run asynchronously.
  const size_t first = (size_t)have * L * K, count = (size_t)n_slabs * L * K;
  PKV_CUDA(cudaMemcpyAsync(p->table_dev + first, p->table_host + first, count * sizeof(uint8_t*),
                           cudaMemcpyHostToDevice, s),
           "cudaMemcpyAsync(slab table)");
  for (int i = 0; i < n_slabs; ++i) p->groups.push_back(fresh[(size_t)i]);
  const int64_t old_rows = (int64_t)have * p->cfg.slab_blocks;
  const int64_t new_rows = (int64_t)p->groups.size() * p->cfg.slab_blocks;
  p->refcount.resize((size_t)new_rows, 0);
  // The free list is a stack: released rows sit on top and are reused first
  // (LIFO).  Fresh rows go underneath them, in descending order, so that once the
  // released rows are used up the fresh rows come out in ascending order.
  std::vector<int32_t> fresh_rows;
  for (int64_t r = new_rows - 1; r >= old_rows; --r) fresh_rows.push_back((int32_t)r);
  p->free_rows.insert(p->free_rows.begin(), fresh_rows.begin(), fresh_rows.end());
  p->append_events += n_slabs;
  p->last_stream = s;
  return PKV_OK;
}

pkv_status pkv_alloc_rows(pkv_pool* p, int n, int32_t* rows_host, void* stream) {
  if (!p || n < 0 || (n > 0 && !rows_host)) return PKV_ERR_INVALID;
  if ((int64_t)p->free_rows.size() < n) {
    const int64_t deficit = n - (int64_t)p->free_rows.size();
    const int need = (int)((deficit + p->cfg.slab_blocks - 1) / p->cfg.slab_blocks);
    pkv_status st = pkv_append_slab(p, need, stream);
    if (st != PKV_OK) return st;
  }
  for (int i = 0; i < n; ++i) {
    int32_t r = p->free_rows.back();
    p->free_rows.pop_back();
    p->refcount[(size_t)r] = 1;
    rows_host[i] = r;
  }
  p->rows_in_use += n;
  return PKV_OK;
}

pkv_status pkv_retain_row(pkv_pool* p, int32_t row) {
  if (!p) return PKV_ERR_INVALID;
  if (row < 0 || (size_t)row >= p->refcount.size() || p->refcount[(size_t)row] <= 0) return PKV_ERR_RANGE;
  p->refcount[(size_t)row] += 1;
  return PKV_OK;
}

pkv_status pkv_release_row(pkv_pool* p, int32_t row) {
  if (!p) return PKV_ERR_INVALID;
  if (row < 0 || (size_t)row >= p->refcount.size() || p->refcount[(size_t)row] <= 0) return PKV_ERR_RANGE;
  if (--p->refcount[(size_t)row] == 0) {
    p->free_rows.push_back(row);
    p->rows_in_use -= 1;
  }
  return PKV_OK;
}

int pkv_slab_runs(const int32_t* rows, int n, int slab_blocks, int32_t* run_start) {
  if (n <= 0) return 0;
  if (!rows || !run_start || slab_blocks < 1) return -1;
  int runs = 0;
  int32_t prev_slab = -1;
  for (int i = 0; i < n; ++i) {
    const int32_t s = rows[i] / slab_blocks;
    if (i == 0 || s != prev_slab) run_start[runs++] = i;
    prev_slab = s;
  }
  return runs;
}

pkv_status pkv_write_block(pkv_pool* p, int layer, int n, const int32_t* rows, const int32_t* slots,
                           const void* k, const void* v, void* stream) {
  if (!p || n < 0 || layer < 0 || layer >= p->cfg.n_layers) return PKV_ERR_INVALID;
  if (n == 0) return PKV_OK;
  if (!rows || !slots || !k || !v) return PKV_ERR_INVALID;
  if (((uintptr_t)k & 15u) != 0 || ((uintptr_t)v & 15u) != 0) return PKV_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  LayerView lv = layer_view(p, layer);
  PKV_CUDA(launch_write(lv, p->cfg.format, p->cfg.head_dim, p->cfg.group_size, n, rows, slots, (const uint16_t*)k,
                        (const uint16_t*)v, p->signs_dev, p->inv_sqrt_d, s),
           "write_block launch");
  p->last_stream = s;
  return PKV_OK;
}

pkv_status pkv_copy_on_write_block(pkv_pool* p, int n, const int32_t* src, const int32_t* dst, void* stream) {
  if (!p || n < 0) return PKV_ERR_INVALID;
  if (n == 0) return PKV_OK;
  if (!src || !dst) return PKV_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  int64_t block_bytes[4] = {0, 0, 0, 0};
  for (int k = 0; k < p->n_kinds; ++k) block_bytes[k] = p->row_bytes[k] * kBlockTokens * p->cfg.n_kv_heads;
  PKV_CUDA(launch_copy_blocks(p->table_dev, p->cfg.n_layers, p->n_kinds, block_bytes, p->cfg.slab_blocks,
                              (int64_t)p->groups.size() * p->cfg.slab_blocks, n, src, dst, p->err_dev, s),
           "copy_on_write_block launch");
  p->last_stream = s;
  return PKV_OK;
}

// Bytes of one block record: every layer, every stored tensor.
static size_t record_bytes(const pkv_pool* p, int64_t* block_bytes) {
  size_t per_layer = 0;
  for (int k = 0; k < 4; ++k) block_bytes[k] = 0;
  for (int k = 0; k < p->n_kinds; ++k) {
    block_bytes[k] = p->row_bytes[k] * kBlockTokens * p->cfg.n_kv_heads;
    per_layer += (size_t)block_bytes[k];
  }
  return per_layer * (size_t)p->cfg.n_layers;
}

pkv_status pkv_pool_get_config(const pkv_pool* p, pkv_pool_config* out) {
  if (!p || !out) return PKV_ERR_INVALID;
  *out = p->cfg;
  return PKV_OK;
}

pkv_status pkv_block_record_bytes(const pkv_pool* p, size_t* bytes) {
  if (!p || !bytes) return PKV_ERR_INVALID;
  int64_t bb[4];
  *bytes = record_bytes(p, bb);
  return PKV_OK;
}

static pkv_status serde_blocks(pkv_pool* p, int n, const int32_t* rows, uint8_t* buf, size_t buf_bytes, int to_pool,
                               cudaStream_t s) {
  if (n == 0) return PKV_OK;
  if (!rows || !buf || ((uintptr_t)buf & 15u) != 0) return PKV_ERR_INVALID;
  int64_t bb[4];
  const size_t rec = record_bytes(p, bb);
  if (buf_bytes / rec < (size_t)n) return PKV_ERR_RANGE;
  PKV_CUDA(launch_serde_blocks(p->table_dev, p->cfg.n_layers, p->n_kinds, bb, p->cfg.slab_blocks,
                               (int64_t)p->groups.size() * p->cfg.slab_blocks, n, rows, buf, (int64_t)rec, to_pool,
                               p->err_dev, s),
           to_pool ? "import_blocks launch" : "export_blocks launch");
  p->last_stream = s;
  return PKV_OK;
}

pkv_status pkv_export_blocks(pkv_pool* p, int n, const int32_t* rows_dev, void* out_dev, size_t out_bytes,
                             void* stream) {
  if (!p || n < 0) return PKV_ERR_INVALID;
  return serde_blocks(p, n, rows_dev, (uint8_t*)out_dev, out_bytes, 0, (cudaStream_t)stream);
}

pkv_status pkv_import_blocks(pkv_pool* p, const pkv_pool_config* identity, int n, const int32_t* rows_dev,
                             const void* in_dev, size_t in_bytes, void* stream) {
  if (!p || !identity || n < 0) return PKV_ERR_INVALID;
  // The records' storage identity (and layer count) must be this pool's, checked
  // before any device work.
  if (pkv_pool_check_identity(p, identity) != PKV_OK || identity->n_layers != p->cfg.n_layers) return PKV_ERR_FORMAT;
  return serde_blocks(p, n, rows_dev, (uint8_t*)const_cast<void*>(in_dev), in_bytes, 1, (cudaStream_t)stream);
}

pkv_status pkv_gather_visible(pkv_pool* p, int layer, const int32_t* bt_row, int ctx, void* k_out,
                              void* v_out, void* kmeta_out, void* vmeta_out, void* stream) {
  if (!p || layer < 0 || layer >= p->cfg.n_layers || ctx < 0) return PKV_ERR_INVALID;
  if (ctx == 0) return PKV_OK;  // nothing visible; output pointers may be NULL
  const bool packed = p->n_kinds == 4;
  if (packed != (kmeta_out != nullptr) || packed != (vmeta_out != nullptr)) return PKV_ERR_FORMAT;
  if (!bt_row || !k_out || !v_out) return PKV_ERR_INVALID;
  for (void* o : {k_out, v_out, kmeta_out, vmeta_out})
    if (((uintptr_t)o & 15u) != 0) return PKV_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* outs[4] = {(uint8_t*)k_out, (uint8_t*)v_out, (uint8_t*)kmeta_out, (uint8_t*)vmeta_out};
  PKV_CUDA(launch_gather(layer_view(p, layer), bt_row, ctx, outs, s), "gather_visible launch");
  p->last_stream = s;
  return PKV_OK;
}

static int decode_grid(const pkv_pool* p) { return p->decode_ctas > 0 ? p->decode_ctas : p->n_sm; }

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static size_t workspace_bytes(const pkv_pool* p, int B, int Hq) {
  const int D = p->cfg.head_dim;
  return align_up((size_t)B * sizeof(int32_t), 256) +
         (size_t)(decode_grid(p) + B) * (size_t)Hq * (size_t)(D + 4) * sizeof(float);
}

pkv_status pkv_decode_workspace_bytes(const pkv_pool* p, int B, int Hq, int max_ctx, size_t* bytes) {
  (void)max_ctx;
  if (!p || !bytes || B < 0 || Hq < 1) return PKV_ERR_INVALID;
  *bytes = workspace_bytes(p, B, Hq);
  return PKV_OK;
}

pkv_status pkv_decode_set_ctas(pkv_pool* p, int n_ctas) {
  if (!p || n_ctas < 0) return PKV_ERR_INVALID;
  p->decode_ctas = n_ctas;
  return PKV_OK;
}

static pkv_status decode_impl(pkv_pool* p, int layer, int B, int Hq, const void* q, const int32_t* bt,
                              int max_blocks, const int32_t* ctx, float scale, void* out, void* ws, size_t ws_bytes,
                              void* stream, int kv_reuse, int nq) {
  if (!p || layer < 0 || layer >= p->cfg.n_layers || B < 0 || Hq < 1 || max_blocks < 0)
    return PKV_ERR_INVALID;
  if (B == 0) return PKV_OK;
  const int hkv = p->cfg.n_kv_heads;
  if (Hq % hkv) return PKV_ERR_INVALID;
  const int G = Hq / hkv;  // with nq > 1: rows of the tile per kv head (nq x heads per kv head)
  if (!(G == 1 || G == 2 || G == 4 || G == 8 || (nq > 1 && G == 16))) return PKV_ERR_INVALID;
  if (!q || !bt || !ctx || !out || !ws) return PKV_ERR_INVALID;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID;
  if (ws_bytes < workspace_bytes(p, B, Hq)) return PKV_ERR_INVALID;
  if (((uintptr_t)ws & 255u) != 0 || ((uintptr_t)q & 15u) != 0 || ((uintptr_t)out & 15u) != 0)
    return PKV_ERR_INVALID;
  DecodePlan plan;
  if (!plan_decode(p->cfg.format, p->cfg.head_dim, G, hkv, B, p->cfg.group_size, &plan) ||
      plan.smem_bytes > p->smem_optin)
    return PKV_ERR_INVALID;
  DecodeArgs a;
  a.lv = layer_view(p, layer);
  a.fmt = p->cfg.format;
  a.D = p->cfg.head_dim;
  a.G = G;
  a.B = B;
  a.Hq = Hq;
  a.max_blocks = max_blocks;
  a.q = (const uint16_t*)q;
  a.bt = bt;
  a.ctx = ctx;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.inv_sqrt_d = (float)p->inv_sqrt_d;
  a.signs = p->signs_dev;
  a.out = (uint16_t*)out;
  a.counters = (int32_t*)ws;
  a.partials = (float*)((uint8_t*)ws + align_up((size_t)B * sizeof(int32_t), 256));
  a.grid = decode_grid(p);
  a.tokens_per_stage = plan.tokens_per_stage;
  a.n_stages = plan.n_stages;
  a.dim_split = plan.dim_split;
  a.group = p->cfg.group_size;
  a.kv_reuse = kv_reuse;
  a.nq = nq;
  // what a sequence start costs a CTA, in quarter units (the CTA split weighs it; the
  // values measured best on the bench workloads): bf16 only reads q's fragments; the
  // packed kernels rotate q at each start (worth more units where units are cheap, at
  // head_dim 64), and with 16 tile rows rotate 16 rows and write two row sets
  const int D = p->cfg.head_dim;
  a.seg_cost = p->cfg.format == PKV_FMT_BF16 ? 2 : (G > 8 ? 16 : (D <= 64 ? 8 : 4));
  a.smem_bytes = plan.smem_bytes;
  a.stream = (cudaStream_t)stream;
  cudaError_t e;
  switch (p->cfg.format) {
    case PKV_FMT_BF16: e = launch_decode_bf16(a); break;
    case PKV_FMT_K4V4: e = launch_decode_k4v4(a); break;
    case PKV_FMT_K8V4: e = launch_decode_k8v4(a); break;
    default: e = launch_decode_k8v8(a); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "paged_decode_attention launch");
  p->last_stream = (cudaStream_t)stream;
  return PKV_OK;
}

pkv_status pkv_paged_decode_attention(pkv_pool* p, int layer, int B, int Hq, const void* q,
                                      const int32_t* bt, int max_blocks, const int32_t* ctx, int max_ctx,
                                      float scale, void* out, void* ws, size_t ws_bytes, void* stream) {
  (void)max_ctx;
  return decode_impl(p, layer, B, Hq, q, bt, max_blocks, ctx, scale, out, ws, ws_bytes, stream, 0, 1);
}

// Chunked prefill: queries per virtual sequence.  The kernels serve nq queries of
// one sequence per tile when nq x (query heads per kv head) fits the tile's 16 rows
// (8 at head_dim 256) and nq divides the chunk: the bf16 kernel for any such power
// of two, the packed kernels for the tile's full 16 rows or 8 rows.
static int prefill_nq(const pkv_pool* p, int n_q, int Hq) {
  if (Hq % p->cfg.n_kv_heads) return 1;
  const int G = Hq / p->cfg.n_kv_heads;
  const int rows = p->cfg.head_dim <= 128 ? 16 : 8;
  if (p->cfg.format != PKV_FMT_BF16) {
    for (int r = rows; r >= 8; r >>= 1) {
      const int nq = r / G;
      if (nq > 1 && n_q % nq == 0) return nq;
    }
    return 1;
  }
  for (int nq = 16; nq > 1; nq >>= 1)
    if (nq * G <= rows && n_q % nq == 0) return nq;
  return 1;
}

// The expanded block table and context lengths, then the decode workspace of the
// B * n_q / nq virtual sequences (nq queries' heads each).
static void prefill_layout(const pkv_pool* p, int B, int n_q, int Hq, int max_blocks, size_t* bt_off, size_t* ctx_off,
                           size_t* dec_off, size_t* total) {
  const int nq = prefill_nq(p, n_q, Hq);
  const size_t nv = (size_t)B * (size_t)(n_q / nq);
  *bt_off = 0;
  *ctx_off = align_up(nv * (size_t)(max_blocks > 0 ? max_blocks : 1) * sizeof(int32_t), 256);
  *dec_off = *ctx_off + align_up(nv * sizeof(int32_t), 256);
  *total = *dec_off + workspace_bytes(p, (int)nv, Hq * nq);
}

pkv_status pkv_prefill_workspace_bytes(const pkv_pool* p, int B, int n_q, int Hq, int max_blocks, size_t* bytes) {
  if (!p || !bytes || B < 0 || n_q < 1 || Hq < 1 || max_blocks < 0 || (int64_t)B * n_q > 4096)
    return PKV_ERR_INVALID;
  size_t a, b, c;
  prefill_layout(p, B, n_q, Hq, max_blocks, &a, &b, &c, bytes);
  return PKV_OK;
}

pkv_status pkv_paged_prefill_attention(pkv_pool* p, int layer, int B, int n_q, int Hq, const void* q,
                                       const int32_t* bt, int max_blocks, const int32_t* ctx, int max_ctx,
                                       float scale, void* out, void* ws, size_t ws_bytes, void* stream) {
  (void)max_ctx;
  if (!p || layer < 0 || layer >= p->cfg.n_layers || B < 0 || n_q < 1 || Hq < 1 || max_blocks < 0 ||
      (int64_t)B * n_q > 4096)
    return PKV_ERR_INVALID;
  if (B == 0) return PKV_OK;
  if (Hq % p->cfg.n_kv_heads) return PKV_ERR_INVALID;
  const int G = Hq / p->cfg.n_kv_heads;
  if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PKV_ERR_INVALID;
  if (!q || !bt || !ctx || !out || !ws || !std::isfinite(scale)) return PKV_ERR_INVALID;
  if (((uintptr_t)ws & 255u) != 0 || ((uintptr_t)q & 15u) != 0 || ((uintptr_t)out & 15u) != 0)
    return PKV_ERR_INVALID;
  const int nq = prefill_nq(p, n_q, Hq);
  const int Bv = B * (n_q / nq);
  size_t bt_off, ctx_off, dec_off, total;
  prefill_layout(p, B, n_q, Hq, max_blocks, &bt_off, &ctx_off, &dec_off, &total);
  if (ws_bytes < total) return PKV_ERR_INVALID;
  DecodePlan plan;
  if (!plan_decode(p->cfg.format, p->cfg.head_dim, G * nq, p->cfg.n_kv_heads, Bv, p->cfg.group_size, &plan) ||
      plan.smem_bytes > p->smem_optin)
    return PKV_ERR_INVALID;
  // q [B, n_q, Hq, D] and out [B, n_q, Hq, D] are [Bv, nq * Hq, D]: virtual sequence v
  // holds queries nq * (v mod (n_q / nq)) .. + nq - 1 of its sequence.  The K/V blocks
  // of a sequence are read by all of its virtual sequences: normal L2 priority.  A
  // chunk of several queries that fits one tile (nq = n_q > 1) is its own virtual
  // sequence: the caller's block table and context lengths serve as they are (the
  // kernels treat a length below nq as a context error and the sequence as empty, as
  // the expansion does).
  const int32_t* bt_v = bt;
  const int32_t* ctx_v = ctx;
  if (nq != n_q || nq == 1) {
    int32_t* bt2 = (int32_t*)((uint8_t*)ws + bt_off);
    int32_t* ctx2 = (int32_t*)((uint8_t*)ws + ctx_off);
    PKV_CUDA(launch_expand_prefill(B, n_q, nq, max_blocks, bt, ctx, bt2, ctx2, p->err_dev, (cudaStream_t)stream),
             "prefill expansion launch");
    bt_v = bt2;
    ctx_v = ctx2;
  }
  return decode_impl(p, layer, Bv, Hq * nq, q, bt_v, max_blocks, ctx_v, scale, out, (uint8_t*)ws + dec_off,
                     ws_bytes - dec_off, stream, 1, nq);
}

pkv_status pkv_price_request(const pkv_pool* p, const pkv_request* r, pkv_price* out) {
  if (!p || !r || !out || r->new_blocks < 0 || r->B < 1 || r->Hq < 1 || r->n_q < 1 || r->max_blocks < 0)
    return PKV_ERR_INVALID;
  if (r->Hq % p->cfg.n_kv_heads) return PKV_ERR_INVALID;
  if (r->n_q > 1 && (int64_t)r->B * r->n_q > 4096) return PKV_ERR_INVALID;
  const int64_t free_rows = (int64_t)p->free_rows.size();
  const int64_t deficit = r->new_blocks > free_rows ? r->new_blocks - free_rows : 0;
  const int64_t slabs = (deficit + p->cfg.slab_blocks - 1) / p->cfg.slab_blocks;
  if ((int64_t)p->groups.size() + slabs > p->cfg.max_slabs) return PKV_ERR_RANGE;
  int64_t block_bytes = 0;  // one block of one layer, every stored tensor
  for (int k = 0; k < p->n_kinds; ++k) block_bytes += p->row_bytes[k] * kBlockTokens * p->cfg.n_kv_heads;
  memset(out, 0, sizeof *out);
  out->slabs_to_append = (int32_t)slabs;
  out->free_rows = free_rows;
  out->storage_bytes = (uint64_t)slabs * (uint64_t)p->group_bytes;
  out->page_bytes = (uint64_t)r->new_blocks * (uint64_t)block_bytes * (uint64_t)p->cfg.n_layers;
  out->fixed_bytes = (uint64_t)r->max_blocks * 4u + 4u + 2ull * (uint64_t)r->n_q * (uint64_t)r->Hq *
                                                          (uint64_t)p->cfg.head_dim * 2u;
  if (r->n_q == 1) {
    out->workspace_bytes = workspace_bytes(p, r->B, r->Hq);
  } else {
    size_t a, b, c, t;
    prefill_layout(p, r->B, r->n_q, r->Hq, r->max_blocks, &a, &b, &c, &t);
    out->workspace_bytes = t;
  }
  return PKV_OK;
}

pkv_status pkv_pool_stats(const pkv_pool* p, pkv_stats* out) {
  if (!p || !out) return PKV_ERR_INVALID;
  memset(out, 0, sizeof *out);
  out->n_slabs = (int32_t)p->groups.size();
  out->n_kinds = p->n_kinds;
  out->slab_append_events = p->append_events;
  out->rows_capacity = (int64_t)p->groups.size() * p->cfg.slab_blocks;
  out->rows_in_use = p->rows_in_use;
  out->bytes_reserved = (int64_t)p->groups.size() * p->layer_bytes * p->cfg.n_layers;  // slab data only
  for (int k = 0; k < 4; ++k) out->row_bytes[k] = p->row_bytes[k];
  return PKV_OK;
}

pkv_status pkv_slab_address(const pkv_pool* p, int layer, int kind, int slab, void** addr) {
  if (!p || !addr) return PKV_ERR_INVALID;
  if (layer < 0 || layer >= p->cfg.n_layers || kind < 0 || kind >= p->n_kinds || slab < 0 ||
      slab >= (int)p->groups.size())
    return PKV_ERR_RANGE;
  *addr = p->table_host[((size_t)slab * p->cfg.n_layers + layer) * p->n_kinds + kind];
  return PKV_OK;
}

pkv_status pkv_pool_check_identity(const pkv_pool* p, const pkv_pool_config* c) {
  if (!p || !c) return PKV_ERR_INVALID;
  const pkv_pool_config& a = p->cfg;
  bool same = a.format == c->format && a.head_dim == c->head_dim && a.n_kv_heads == c->n_kv_heads &&
              a.block_size == c->block_size && a.slab_blocks == c->slab_blocks;
  if (a.format != PKV_FMT_BF16)
    same = same && a.group_size == c->group_size && a.hadamard_seed == c->hadamard_seed;
  return same ? PKV_OK : PKV_ERR_FORMAT;
}

pkv_status pkv_pool_check_errors(pkv_pool* p, void* stream, int32_t* word_out) {
  if (!p) return PKV_ERR_INVALID;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t w = 0;
  PKV_CUDA(cudaMemcpyAsync(&w, p->err_dev, sizeof w, cudaMemcpyDeviceToHost, s), "read error word");
  PKV_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (word_out) *word_out = w;
  if (w) {
    PKV_CUDA(cudaMemsetAsync(p->err_dev, 0, sizeof w, s), "clear error word");
    PKV_CUDA(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    return PKV_ERR_DEVICE;
  }
  return PKV_OK;
}

}  // extern "C"
