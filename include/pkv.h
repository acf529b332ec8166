/*
 * pkv.h — C ABI of the GB300 paged-KV decode-attention library (libpkv.so).
 *
 * A pool stores the K/V cache of every layer in chunked slab storage: for each
 * layer and stored tensor, a vector of fixed-size slabs shaped
 *   [slab_blocks, block_size, n_kv_heads, row]
 * (row = head_dim bf16 values, or packed codes, or (scale, offset) pairs).  A
 * physical row (one block of block_size tokens) maps to slab = row / slab_blocks,
 * row_in_slab = row % slab_blocks.  Growth appends fresh zeroed slabs and never
 * copies or frees an existing one.
 *   [mlxcel issue #235, "chunked slab storage for the paged pool", Proposed
 *    solution: bullets 1-3]
 *
 * Stored formats: native bf16, or packed K4/V4, K8/V4, K8/V8 with token-local
 * affine groups of group_size values and an FP32 (scale, offset) pair per group;
 * K (and Q at attention time) is expressed in a fixed signed Hadamard basis.
 *   [mlx-swift-lm PR #142, "packed paged KV formats with bounded workspace
 *    admission", Summary]
 *
 * Conventions for every call
 *  - All pointers named *_dev are device pointers; *_host are host pointers.
 *    Device buffers passed in are owned by the caller and must stay valid until
 *    the work enqueued on `stream` has finished.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  Every call that touches device memory is asynchronous on that
 *    stream unless stated otherwise; none synchronises the device except
 *    pkv_pool_check_errors and pkv_pool_destroy.
 *  - Host-checkable errors (NULL pointers, sizes out of range, a layer index out
 *    of range, workspace too small, allocation failure) are returned
 *    synchronously, before any state changes or work is enqueued.
 *  - Device-detected range errors (a block-table row beyond the pool's rows, a
 *    context length beyond max_blocks*block_size, a slot beyond block_size) set
 *    the pool's device error word; the offending block/token is skipped (the
 *    result is then undefined but no memory outside the pool is touched).  Read
 *    and clear it with pkv_pool_check_errors.
 *  - A pool is not thread-safe; callers serialise calls on one pool.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_pool pkv_pool; /* opaque; owns slabs, pointer tables, row allocator */

typedef enum {
  PKV_FMT_BF16 = 0, /* native: K and V rows are head_dim bf16 values            */
  PKV_FMT_K4V4 = 1, /* K 4-bit codes (Hadamard basis), V 4-bit codes           */
  PKV_FMT_K8V4 = 2, /* K 8-bit codes (Hadamard basis), V 4-bit codes           */
  PKV_FMT_K8V8 = 3  /* K 8-bit codes (Hadamard basis), V 8-bit codes           */
} pkv_format;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = -1, /* bad argument (NULL, size, layer, alignment)          */
  PKV_ERR_OOM = -2,     /* the allocator returned NULL; the pool is unchanged    */
  PKV_ERR_CUDA = -3,    /* a CUDA runtime call failed (message: pkv_last_error)  */
  PKV_ERR_FORMAT = -4,  /* storage identity does not match the request           */
  PKV_ERR_RANGE = -5,   /* a host-visible index is out of range                  */
  PKV_ERR_DEVICE = -6   /* the device error word was set (pkv_pool_check_errors) */
} pkv_status;

/* Tensor kinds stored per layer. */
enum { PKV_KIND_K = 0, PKV_KIND_V = 1, PKV_KIND_KMETA = 2, PKV_KIND_VMETA = 3 };

typedef struct {
  int32_t n_layers;      /* >= 1                                                */
  int32_t n_kv_heads;    /* 1..8 (one decode consumer warp per kv head)         */
  int32_t head_dim;      /* 64, 128 or 256                                      */
  int32_t block_size;    /* tokens per block; must be 32                        */
  int32_t slab_blocks;   /* blocks per slab (POOL_SLAB_BLOCKS); 1..4096, 32 is the default */
  int32_t group_size;    /* values per affine group (ignored for bf16): 32, or 64 for K4/V4 with
                          * head_dim 128 or 256 (one FP32 scale/offset pair per 64 values: five
                          * bits per value, 3.2x against bf16)
                          *   [mlx-swift-lm #142, Summary: K4/V4 at five bits per value,
                          *    metadata included] */
  int32_t format;        /* pkv_format                                          */
  int32_t max_slabs;     /* capacity of the slab pointer table (>= 1)           */
  uint64_t hadamard_seed;/* signs s_i = -1 iff top bit of splitmix64(seed + i)  */
} pkv_pool_config;

/* Stream-ordered allocator used for slabs.  alloc returns NULL on failure.  With
 * a NULL allocator the pool uses cudaMallocAsync / cudaFreeAsync on the stream. */
typedef struct {
  void* (*alloc)(void* ctx, size_t bytes, void* stream);
  void (*release)(void* ctx, void* ptr, void* stream);
  void* ctx;
} pkv_allocator;

typedef struct {
  int32_t n_slabs;            /* slabs per (layer, tensor) currently held          */
  int32_t n_kinds;            /* 2 (bf16) or 4 (packed: K, V, K meta, V meta)      */
  int64_t slab_append_events; /* slabs appended since create (never a copy)        */
  int64_t rows_capacity;      /* n_slabs * slab_blocks                             */
  int64_t rows_in_use;        /* rows with a nonzero reference count               */
  int64_t bytes_reserved;     /* sum over every slab of every layer and tensor     */
  int64_t row_bytes[4];       /* bytes of one (token, head) row per tensor kind    */
} pkv_stats;

/* Create a pool with no slabs on the current device: per layer and stored tensor an
 * empty vector of slabs, the pointer table for up to max_slabs of them, the row
 * allocator and the device error word.  The allocator struct is copied.  *out
 * receives the pool (owned by the caller until pkv_pool_destroy).  Errors:
 * PKV_ERR_INVALID for an unsupported configuration (n_kv_heads outside 1..8,
 * head_dim not 64/128/256, block_size not 32, group_size not allowed for the
 * format), PKV_ERR_CUDA if the device cannot be used.  Synchronous.
 *   [mlxcel #235, Proposed solution, bullet 1: the single pool tensor of a layer
 *    becomes a vector of fixed-size slabs] */
pkv_status pkv_pool_create(const pkv_pool_config* cfg, const pkv_allocator* alloc, void* stream,
                           pkv_pool** out);

/* Wait for the device, then release every slab (through the pool's allocator) and
 * the pool itself.  NULL is ignored.  Slabs are freed only here, never while the
 * pool lives.
 *   [mlxcel #235, Proposed solution, bullet 2: growth never frees a slab] */
void pkv_pool_destroy(pkv_pool* pool);

/* Append n_slabs fresh zeroed slabs to every layer and tensor, in one step
 * (presize_for_span).  Existing slabs are neither copied nor freed; their base
 * addresses stay valid.  All-or-nothing: on PKV_ERR_OOM the pool is unchanged.
 *   [mlxcel #235, Proposed solution, bullet 2] */
pkv_status pkv_append_slab(pkv_pool* pool, int n_slabs, void* stream);

/* Take n rows from the free list (LIFO reuse of released rows, then rows of
 * appended slabs in ascending order), appending slabs when it is empty.  Each
 * returned row has reference count 1.  rows_host: n int32.
 *   [mlxcel #235, Behavioral invariants: block identities, reference counts and the
 *    reuse of freed rows remain row-level bookkeeping] */
pkv_status pkv_alloc_rows(pkv_pool* pool, int n, int32_t* rows_host, void* stream);

/* Reference counting of rows (host bookkeeping only).  retain requires a live
 * row; release returns a row to the free list when its count reaches 0.
 * PKV_ERR_RANGE for a row outside the pool or not live. */
pkv_status pkv_retain_row(pkv_pool* pool, int32_t row);
pkv_status pkv_release_row(pkv_pool* pool, int32_t row);

/* Maximal same-slab runs of a block-table row list, in logical order: writes the
 * starting index of each run to run_start_host (capacity n) and returns the number
 * of runs (0 for n <= 0, -1 for bad arguments).  Host only; no pool needed.
 *   [mlxcel #235, touch point 3, gather_visible] */
int pkv_slab_runs(const int32_t* rows_host, int n, int slab_blocks, int32_t* run_start_host);

/* write_block: token i of k/v goes to (rows_dev[i], slots_dev[i]) of `layer`.
 * k_bf16_dev, v_bf16_dev: [n_tokens, n_kv_heads, head_dim] bf16, row-major.
 * Packed formats quantise here, once: K is rotated into the Hadamard basis,
 * then every group of group_size values gets scale = (max-min)/(2^bits-1),
 * offset = min, code = round-half-even((x-min)/scale) (0 when scale is 0).
 *   [mlxcel #235, touch point 1; mlx-swift-lm #142, After flowchart: new K/V are
 *    quantised a single time, when written] */
pkv_status pkv_write_block(pkv_pool* pool, int layer, int n_tokens, const int32_t* rows_dev,
                           const int32_t* slots_dev, const void* k_bf16_dev, const void* v_bf16_dev,
                           void* stream);

/* copy_on_write_block: copy every byte of block src_rows_dev[i] to block
 * dst_rows_dev[i], for every layer and stored tensor.  Pairs must not overlap.
 *   [mlxcel #235, touch point 2] */
pkv_status pkv_copy_on_write_block(pkv_pool* pool, int n, const int32_t* src_rows_dev,
                                   const int32_t* dst_rows_dev, void* stream);

/* gather_visible: the visible context of one sequence (tokens [0, ctx_len)) as
 * dense arrays in logical order, equal to concatenating the maximal same-slab
 * runs of its block-table row.  bt_row_dev: ceil(ctx_len/block_size) rows.
 * Outputs (device): k_out, v_out [n_kv_heads, ctx_len, row_bytes(kind)];
 * kmeta_out, vmeta_out [n_kv_heads, ctx_len, head_dim/group_size, 2] float32,
 * which must be NULL for bf16 and non-NULL for packed (else PKV_ERR_FORMAT);
 * with ctx_len 0 nothing is written and every output may be NULL.
 *   [mlxcel #235, touch point 3] */
pkv_status pkv_gather_visible(pkv_pool* pool, int layer, const int32_t* bt_row_dev, int ctx_len,
                              void* k_out_dev, void* v_out_dev, void* kmeta_out_dev,
                              void* vmeta_out_dev, void* stream);

/* Workspace bytes needed by pkv_paged_decode_attention for batches of up to B
 * sequences with Hq query heads (max_ctx is the caller's bound on any context
 * length; it is accepted for interface stability and does not change the size).
 * The workspace holds the split-K partials and per-sequence arrival counters; it
 * must be zero-filled once before its first use (the kernel leaves it reusable).
 * Host only; PKV_ERR_INVALID for a NULL pool or bytes, B < 0 or Hq < 1.
 *   [mlx-swift-lm #142, Summary: the workspace a step is guaranteed is priced on
 *    its own, apart from storage] */
pkv_status pkv_decode_workspace_bytes(const pkv_pool* pool, int B, int Hq, int max_ctx,
                                      size_t* bytes);

/* Batched single-token decode attention with GQA (query head h reads KV head
 * h / (Hq / n_kv_heads)), no mask, over tokens [0, ctx_lens[b]) of each
 * sequence:  out[b,h] = softmax(scale * q[b,h] . K_b^T) V_b.
 * For packed formats q is rotated into K's Hadamard basis inside the kernel and
 * K/V are dequantised in registers (no dequantised history is materialised).
 *   q_bf16_dev:      [B, Hq, head_dim] bf16 (un-rotated)
 *   block_table_dev: [B, max_blocks] int32 rows
 *   ctx_lens_dev:    [B] int32; 0 gives a zero output row
 *   max_ctx:         host bound on ctx_lens (used only to size the launch)
 *   out_bf16_dev:    [B, Hq, head_dim] bf16
 *   workspace_dev:   ws_bytes >= pkv_decode_workspace_bytes(B, Hq), zeroed once
 * Deterministic: bitwise identical results for identical inputs on one device.
 * Limits: 1 <= B <= 4096 (the batch's unit prefix is staged in shared memory);
 * n_kv_heads <= 8 (one consumer warp per kv head, fixed at pool creation);
 * G = Hq / n_kv_heads in {1, 2, 4, 8}.
 * Range: q and K of any magnitude whose logits (scale * q.k) are finite in fp32
 * (|q| below 2^100), and V of magnitudes within about 2^-50..2^40, are handled at
 * the same accuracy as values near 1: the packed kernels keep their 16-bit tensor
 * operands in range with powers of two that are removed exactly in fp32 (the
 * rotated q per tile row, in fp16; the probabilities times the V scales with a fixed
 * 2^64, in bf16).  Slots of a block past a sequence's context are never read into
 * the result, whatever bytes they hold.
 * B = 0 returns PKV_OK with no device work.  PKV_ERR_INVALID, before any work,
 * when B > 4096, Hq is not n_kv_heads x G with G in {1, 2, 4, 8}, scale is not
 * finite, the workspace is smaller than pkv_decode_workspace_bytes or not 256-byte
 * aligned, or q / out are not 16-byte aligned.
 *   [mlxcel issue #2171, "one KV storage abstraction": Proposed Solution
 *    (KVCache::attend -> paged_batch_decode_attention) and Implementation Notes,
 *    edge cases (single token, no mask); mlx-swift-lm #142, Summary: packed pages
 *    are attended to directly, with no expanded copy of the history] */
pkv_status pkv_paged_decode_attention(pkv_pool* pool, int layer, int B, int Hq,
                                      const void* q_bf16_dev, const int32_t* block_table_dev,
                                      int max_blocks, const int32_t* ctx_lens_dev, int max_ctx,
                                      float scale, void* out_bf16_dev, void* workspace_dev,
                                      size_t ws_bytes, void* stream);

/* Size of the fixed device scratch array used by pkv_paged_decode_attention_noalloc. */
#define PKV_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* Decode attention without any device allocation by the caller or the library.
 * The source pages have no counterpart to this call.  It exists for callers that
 * cannot call cudaMalloc or borrow an allocator: for example a serving loop that
 * reserved all of its device memory at start-up and may not allocate during a
 * decode step, or a plugin whose host framework owns the device allocator.
 * Arguments and results are those of pkv_paged_decode_attention, minus the
 * workspace: the split-K partials and arrival counters live instead in a fixed
 * array of PKV_STATIC_SCRATCH_BYTES (8 MiB) compiled into the library, which every
 * GPU that loads the library holds until the process exits.
 *  - The first call on each device looks up that device's copy of the array
 *    (cudaGetSymbolAddress, with the device current); make that first call before
 *    any stream capture.
 *  - Each call clears the arrival counters on `stream` (a cudaMemsetAsync, not an
 *    allocation), then launches the same kernel as pkv_paged_decode_attention.
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents: calls whose GPU work overlaps (different streams, or different
 *    pools) race on it and give undefined results; serialise them.
 *  - PKV_ERR_RANGE, with a message from pkv_last_error, when (B, Hq, head_dim)
 *    need more scratch than the array holds (pkv_decode_workspace_bytes tells). */
pkv_status pkv_paged_decode_attention_noalloc(pkv_pool* pool, int layer, int B, int Hq,
                                              const void* q_bf16_dev, const int32_t* block_table_dev,
                                              int max_blocks, const int32_t* ctx_lens_dev, int max_ctx,
                                              float scale, void* out_bf16_dev, void* stream);

/* Number of CTAs a decode launch uses (0 = one per SM, the default).  Changing it
 * changes the split-K partition (results agree to rounding) and the workspace
 * size.  PKV_ERR_INVALID for n < 0.  Host only.  (A tuning and test knob; the
 * pages have no counterpart.) */
pkv_status pkv_decode_set_ctas(pkv_pool* pool, int n_ctas);

/* Pool statistics (host bookkeeping; no device access): slab count, the
 * slab-append counter (one per appended slab; no slab is ever copied), row
 * capacity and rows in use, and bytes_reserved as the sum over every slab of every
 * layer and tensor.  PKV_ERR_INVALID for NULL arguments.
 *   [mlxcel #235, Proposed solution, bullet 2 (the growth counter counts slab
 *    appends) and touch point 5 (reserved bytes summed over slabs)] */
pkv_status pkv_pool_stats(const pkv_pool* pool, pkv_stats* out);

/* Device base address of slab `slab` of (layer, kind); PKV_ERR_RANGE if absent.
 * Host only.
 *   [mlxcel #235, touch point 4: per-slab base pointers] */
pkv_status pkv_slab_address(const pkv_pool* pool, int layer, int kind, int slab, void** addr);

/* A request's price for admission into a step: the three costs that an admission
 * policy weighs separately.  Host only; nothing is allocated or changed.
 *   in  new_blocks:  blocks (rows) the request needs that it does not share with a
 *                    sequence already in the pool (e.g. ceil(tokens / 32) minus the
 *                    blocks of a shared prefix); >= 0
 *   in  B, Hq, n_q:  the step it joins: sequences (the request included), query
 *                    heads, queries per sequence (1 for decode, > 1 for a chunked
 *                    prefill of n_q tokens)
 *   in  max_blocks:  block-table width of that step
 *   out slabs_to_append: slabs pkv_alloc_rows(new_blocks) would append now (0
 *                    while the free list holds enough rows), the same count
 *                    pkv_append_slab(n) takes to presize for the span
 *   out free_rows:   rows on the free list now
 *   out storage_bytes: growing storage: the bytes the allocator is asked for by
 *                    those appends (every layer and tensor of each slab, plus the
 *                    slab's 128-byte tensor maps)
 *   out page_bytes:  page cost: the stored bytes of the request's new blocks, every
 *                    layer and tensor (pkv_block_record_bytes x new_blocks); this is
 *                    space inside the pool's capacity, not a further allocation
 *   out fixed_bytes: fixed per-request cost of a step: its block-table row
 *                    (max_blocks int32), context length (int32), and q and output
 *                    rows (n_q x Hq x head_dim bf16 each)
 *   out workspace_bytes: the step's guaranteed workspace for (B, Hq, n_q,
 *                    max_blocks): pkv_decode_workspace_bytes(B, Hq) when n_q == 1,
 *                    else pkv_prefill_workspace_bytes(B, n_q, Hq, max_blocks)
 * A request fits a device budget of free bytes F when storage_bytes + fixed_bytes
 * plus the growth of the step's workspace over what the caller already holds is at
 * most F.  Errors: PKV_ERR_INVALID for NULL pointers, negative or zero sizes, Hq
 * not a multiple of n_kv_heads or B * n_q > 4096 with n_q > 1; PKV_ERR_RANGE when
 * the slabs to append would exceed max_slabs (the pool can never hold the request).
 *   [mlx-swift-lm #142, Summary: admission prices the growth of storage, the page
 *    and fixed costs and the step's guaranteed workspace each on its own; After:
 *    admission = storage plus guaranteed workspace; mlxcel #235, Proposed
 *    solution, bullet 2: presize_for_span appends the slabs a span needs at once] */
typedef struct {
  int32_t new_blocks;
  int32_t B;
  int32_t Hq;
  int32_t n_q;
  int32_t max_blocks;
} pkv_request;

typedef struct {
  int32_t slabs_to_append;
  int64_t free_rows;
  uint64_t storage_bytes;
  uint64_t page_bytes;
  uint64_t fixed_bytes;
  uint64_t workspace_bytes;
} pkv_price;

pkv_status pkv_price_request(const pkv_pool* pool, const pkv_request* req, pkv_price* out);

/* Storage identity check: PKV_OK if cfg describes the same stored layout as the
 * pool (format, head_dim, n_kv_heads, block_size, slab_blocks, group_size and,
 * for packed formats, hadamard_seed), else PKV_ERR_FORMAT.  Used to reject an
 * incompatible storage identity before any allocation or copy.
 *   [mlx-swift-lm #142, Summary: a checkpoint of another storage identity is
 *    refused before anything is allocated] */
pkv_status pkv_pool_check_identity(const pkv_pool* pool, const pkv_pool_config* cfg);

/* Workspace bytes for pkv_paged_prefill_attention with B sequences, n_q new tokens
 * each, Hq query heads and block tables of max_blocks entries.  B * n_q <= 4096.
 * Synchronous, host only. */
pkv_status pkv_prefill_workspace_bytes(const pkv_pool* pool, int B, int n_q, int Hq, int max_blocks, size_t* bytes);

/* Causal chunked-prefill attention over the pool: sequence b holds ctx_lens[b]
 * tokens (its chunk of n_q new tokens already written with pkv_write_block, as the
 * last n_q), and query i of the chunk attends to tokens [0, ctx_lens[b] - n_q + i].
 * q_bf16: [B, n_q, Hq, head_dim] bf16, un-rotated (packed formats rotate q
 * internally); out_bf16: [B, n_q, Hq, head_dim]; block_table, ctx_lens and the GQA
 * mapping as for pkv_paged_decode_attention.  The workspace (caller-owned, 256-byte
 * aligned, pkv_prefill_workspace_bytes) holds, for each run of NQ consecutive
 * queries of a sequence, a view of the sequence (the same block-table row, the
 * last of those queries' causal length; when NQ = n_q > 1 the caller's block table
 * and lengths serve directly) and the split-K partials.  The attention kernels
 * serve the NQ queries in one tensor-core tile, each masked at its own causal
 * limit: up to 16 (query, head) rows per kv head at head_dim <= 128 and 8 at 256;
 * NQ is the largest such count dividing n_q (bf16), or the one filling 16 rows, else
 * 8 rows (packed formats), else 1.
 * A sequence with fewer than n_q tokens sets the device error word (bit 2) and its
 * rows are zero.
 * Errors as for pkv_paged_decode_attention; PKV_ERR_INVALID when B * n_q > 4096.
 * Asynchronous.
 *   [mlxcel #2171, Proposed Solution: attend = update the storage, then attention;
 *    mlx-swift-lm #142, Summary: packed pages are attended to directly] */
pkv_status pkv_paged_prefill_attention(pkv_pool* pool, int layer, int B, int n_q, int Hq, const void* q_bf16,
                                       const int32_t* block_table, int max_blocks, const int32_t* ctx_lens,
                                       int max_ctx, float scale, void* out_bf16, void* workspace, size_t ws_bytes,
                                       void* stream);

/* The pool's configuration (its storage identity plus n_layers and max_slabs), for
 * a checkpoint header.  Synchronous, host only.
 *   [mlx-swift-lm #142, After: a packed checkpoint carries its format identity] */
pkv_status pkv_pool_get_config(const pkv_pool* pool, pkv_pool_config* out);

/* Bytes of one block record: every stored byte of one block (row) of every layer,
 * layer-major, then tensor kind (K, V, K meta, V meta), each the block's
 * [block_size, n_kv_heads, row_bytes(kind)] bytes exactly as stored.  Equals
 * n_layers * block_size * n_kv_heads * sum over kinds of row_bytes(kind).
 * Synchronous, host only. */
pkv_status pkv_block_record_bytes(const pkv_pool* pool, size_t* bytes);

/* export_blocks: write the records of blocks rows_dev[0..n) to out_dev, one after
 * another in list order (n records; packed codes and FP32 metadata are copied
 * bit for bit, nothing is dequantised).  rows_dev: n int32 on the device; out_dev:
 * caller-owned device buffer, 16-byte aligned, at least n records long
 * (out_bytes).  Errors: PKV_ERR_INVALID for null or misaligned pointers,
 * PKV_ERR_RANGE when out_bytes is too small; a row outside the pool sets the
 * device error word (bit 1) and its record is left unwritten.  Asynchronous.
 *   [mlxcel #235, touch point 6: a block's content is read from the slab that holds
 *    its row, through the shared mapping helper; mlx-swift-lm #142, Summary: a full
 *    checkpoint keeps the packed bytes as they are] */
pkv_status pkv_export_blocks(pkv_pool* pool, int n, const int32_t* rows_dev, void* out_dev, size_t out_bytes,
                             void* stream);

/* import_blocks: the restore path.  Copy n records from in_dev (layout of
 * pkv_export_blocks) into blocks rows_dev[0..n) of this pool (live, distinct rows;
 * the caller allocates them).  `identity` is the configuration of the pool the
 * records came from: when its storage identity (pkv_pool_check_identity) or its
 * n_layers differs from this pool's, PKV_ERR_FORMAT is returned before any device
 * work, so an incompatible checkpoint is rejected before anything is written.
 * Other errors as for export.  Asynchronous.
 *   [mlxcel #235, touch point 6: restore path; mlx-swift-lm #142, Summary: a
 *    checkpoint of another storage identity is refused before anything is
 *    allocated; After: the packed checkpoint is exact and carries its format] */
pkv_status pkv_import_blocks(pkv_pool* pool, const pkv_pool_config* identity, int n, const int32_t* rows_dev,
                             const void* in_dev, size_t in_bytes, void* stream);

/* Synchronise `stream`, read and clear the device error word.  PKV_ERR_DEVICE if it
 * was set (bits: 1 row out of range, 2 context too long, 4 slot out of range,
 * 8 wait limit reached); *word_out (optional) receives the bits.  The kernels record
 * errors on the device instead of returning them, so that a decode step needs no
 * host synchronisation; the caller checks when it chooses.
 *   [mlxcel #2171, Implementation Notes: a decode step adds no host sync] */
pkv_status pkv_pool_check_errors(pkv_pool* pool, void* stream, int32_t* word_out);

/* Static description of a status code, and the last CUDA error message seen by
 * this thread (empty if none).  Never NULL; the strings belong to the library.
 * (C-ABI conveniences with no counterpart on the pages.) */
const char* pkv_status_string(pkv_status status);
const char* pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
