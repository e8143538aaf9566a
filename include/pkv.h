/*
 * pkv.h -- C ABI of libpkv: decode-phase attention over a paged KV cache on
 * GB300 (sm_103a).
 *
 * The operations follow the pages' statement of the problem:
 *   - "Inference part 1" (brunomaga), section "KV cache": each decode step
 *     computes q, k, v for the new token only, writes the new key and value
 *     into the cache in place (a static cache) and attends over every cached
 *     row; queries are not cached.  Several new tokens on top of a cache see
 *     the cached rows and the new rows up to themselves (the shifted causal
 *     mask of scaled_dot_product_attention_kv_cache).
 *   - same page, section "PagedAttention: memory management for the KV
 *     cache": the cache is split into fixed-size blocks allocated on demand;
 *     a per-sequence block table maps logical blocks to physical blocks
 *     anywhere in GPU memory, and the attention kernel reads through it.
 *     "KV cache, prefill va decode" (truongducdung), section 05, "Block
 *     table": 16 tokens per block in vLLM; a new block only when the last one
 *     is full.
 *   - "Inference part 1", section "Why attention matters": the attention
 *     equation softmax(Q K^T / sqrt(d_head)) V; section "Smaller KV caches:
 *     MQA, GQA and MLA": consecutive query heads share one KV head.
 *   - same page, section "FlashDecoding": the keys and values are split
 *     along the sequence, each chunk yields a partial output and its softmax
 *     statistics, and a final reduction rescales them as in the online
 *     softmax ("KV cache, prefill va decode", section 07, Flash-Decoding:
 *     the log-sum-exp of each chunk is kept and merged).
 *   - "Inference part 2" (brunomaga), section "Speculative decoding": the
 *     target scores the last accepted token and the K drafts (K + 1 queries)
 *     in one pass.
 *
 * Layouts (all row-major, C order; "elt" is the element type of `dtype`):
 *   k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim] elt
 *                      (one (block, kv-head) tile is contiguous)
 *   block_table      : [batch, max_blocks_per_seq] int32; entry n of row b is
 *                      the physical block holding rows n*block_size ..
 *                      (n+1)*block_size - 1 of sequence b.  Entries past the
 *                      sequence's last block are never read.
 *   context_lens     : [batch] int32, L_b = rows of sequence b INCLUDING the
 *                      new rows (the token just appended; for speculative
 *                      verification the K + 1 verified tokens).
 *   q, out (decode)  : [batch, num_heads, head_dim] elt
 *   q, out (verify)  : [batch, num_queries, num_heads, head_dim] elt
 *   Query head h reads KV head h / (num_heads / num_kv_heads).
 *   Query row j (0-based) of a sequence sees rows i <= L_b - num_queries + j.
 *   A query row that sees no row (e.g. L_b = 0) gets a zero output.
 *
 * Ownership and streams: the caller owns every buffer (device pointers,
 * including the workspace and the optional error word).  The library never
 * allocates, frees or synchronises in these calls; all work is enqueued on
 * `stream` (a cudaStream_t; NULL = the legacy default stream).
 *
 * Errors: argument errors are reported synchronously with nothing enqueued.
 * A failed launch returns PKV_ERR_CUDA.  Device-side precondition violations
 * (a slot or block id out of range, a context longer than max_context_len)
 * never fault: the offending row or block is skipped and, when `error_word`
 * (a device int32, caller-zeroed) is given, its first violation code
 * (PKV_DEVERR_*) is recorded there.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shapes */
  PKV_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, block_size, dtype */
  PKV_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime call or a launch failed */
  PKV_ERR_ALIGNMENT = 5,   /* a tensor pointer is not 16-byte aligned */
  PKV_ERR_HOST_MEMORY = 6  /* a host allocation failed (block manager) */
} pkv_status;

/* Element types.  PKV_FP8_E4M3 is a cache type only (one byte per element,
 * one float scale per cache tensor; see pkv_kv_append_fp8). */
typedef enum pkv_dtype { PKV_F32 = 0, PKV_BF16 = 1, PKV_F16 = 2, PKV_FP8_E4M3 = 3 } pkv_dtype;

/* Codes the kernels record in the optional device error word. */
enum {
  PKV_DEVERR_NONE = 0,
  PKV_DEVERR_SLOT = 1,        /* kv_append: slot >= num_blocks * block_size */
  PKV_DEVERR_BLOCK_ID = 2,    /* block_table entry outside [0, num_blocks) */
  PKV_DEVERR_CONTEXT_LEN = 3, /* context_lens[b] > max_context_len or > table */
  PKV_DEVERR_TIMEOUT = 4      /* a shared-memory copy did not arrive in time */
};

/* Kernel families. */
typedef enum pkv_kernel {
  PKV_KERNEL_AUTO = 0,
  PKV_KERNEL_SIMT = 1, /* CUDA-core dot products (any dtype; fp32 path) */
  PKV_KERNEL_MMA = 2,  /* tensor-core tiles (bf16 / fp16 q; 16-bit or FP8 cache);
                          up to 40 query rows per KV head in one CTA at head_dim
                          <= 128 (8 at 256), more cut into row chunks */
  PKV_KERNEL_TC = 3    /* tcgen05 tiles with TMEM accumulators: bf16 / fp16 caches,
                          head_dim 128, up to 64 query rows per CTA (more cut into
                          row chunks), fused append included; opt-in */
} pkv_kernel;

/* Optional launch controls (pass NULL for the planner's choice). */
typedef struct pkv_options {
  int kernel;       /* pkv_kernel */
  int split_blocks; /* 0: planner; > 0: KV blocks per split-K chunk */
  int stages;       /* 0: planner; mma.sync kernel: ring depth per block
                       lane, the tile's shallow or deep ring (at head_dim <= 128:
                       2 or 3 with one column group, 3 or 4 with two, 4 or 6
                       with three to five; 1 or 2 at 256; twice these for FP8
                       caches); tcgen05 kernel: the V ring's depth in 128-key
                       chunks, 1..3 (1..2 above 32 rows); other values are
                       refused */
  int rows_per_cta; /* 0: planner; cap on the query rows one CTA serves */
  int merge;        /* split-K merge: 0 planner, 1 by the sequence's last CTA,
                       2 by a separate kernel */
  int warp_tiles;   /* 0: planner; tensor-core kernel: 8-column query tiles
                       per warp (1..3 at head_dim <= 128, 1..4 at 64, 1 at 256) */
  int blocks_per_iter; /* 0: planner; tensor-core kernel: KV blocks one warp
                          takes per loop iteration (1 or 2; 2 with one tile) */
  int persistent;   /* tcgen05 kernel: 0 planner, 1 one CTA per resident slot
                       walks the work items, 2 one CTA per item */
  int split_waves;  /* split-K partition from the batch's real lengths, read
                       on the device (batch <= 32, split_blocks 0): k > 0
                       cuts the batch into at most k waves of resident CTAs
                       with splits of nearly equal length; -1: the host plan
                       (split length from max_context_len); 0: the default,
                       the host plan for the CUDA-core and mma.sync kernels
                       and the balanced partition for the tcgen05 kernel
                       (one CTA per SM, each taking an equal share of the
                       batch's blocks; see pkv_plan.stream_k) */
} pkv_options;

/* What one attention call launches (see pkv_attention_plan). */
typedef struct pkv_plan {
  int kernel;             /* PKV_KERNEL_SIMT, PKV_KERNEL_MMA or PKV_KERNEL_TC */
  int rows_per_cta;       /* query rows (queries x heads of one KV head) per CTA */
  int row_chunks;         /* CTAs that share one (sequence, KV head) */
  int split_blocks;       /* KV blocks per split */
  int num_splits;         /* splits of the longest sequence; 1 = no merge */
  int grid_x, grid_y, grid_z;
  int threads_per_cta;
  int stages;             /* shared-memory stages per warp (tcgen05: V ring depth) */
  int ctas_per_sm;        /* occupancy the planner assumed */
  size_t smem_bytes;      /* dynamic shared memory per CTA */
  size_t workspace_bytes; /* device workspace the call needs (0 = none) */
  int merge_kernel;       /* 1: a separate split-K merge launch follows;
                             0: no split, or the last CTA of each sequence merges */
  int warp_tiles;         /* tensor-core kernel: 8-column query tiles per warp */
  int blocks_per_iter;    /* tensor-core kernel: KV blocks per loop iteration */
  int split_target;       /* > 0: the partition is made on the device from the
                             real context lengths, into at most this many CTAs
                             (grid_x; split_blocks 0, num_splits an upper bound
                             per sequence); 0: the host partition above */
  int stream_k;           /* 1 (with split_target = grid_x > 0): the balanced
                             partition -- the (sequence, KV head) units of the
                             batch laid end to end as one list of blocks, and
                             CTA c of the grid_x taking the list's blocks
                             floor(c T / grid_x) .. floor((c + 1) T / grid_x) - 1
                             (T blocks in all), a split wherever its range meets
                             a unit; 0: otherwise */
} pkv_plan;

/* Human-readable name of a status code (static string). */
PKV_API const char *pkv_status_string(pkv_status status);

/* Library version string, e.g. "pkv 0.1.0 sm_103a". */
PKV_API const char *pkv_version(void);

/*
 * pkv_kv_append -- write the K/V rows of new tokens into their cache slots.
 * "Inference part 1", section "KV cache" (in-place write of a static cache);
 * "Inference part 2", GPTlite_StaticCache (k_cache[..., input_pos] = k);
 * "Efficient Inference" (obvix), the in-place slice write; in paged form a
 * slot s is row s % block_size of physical block s / block_size
 * ("KV cache, prefill va decode", section 05, "Block table").
 *
 *   k_new, v_new : [num_tokens, num_kv_heads, head_dim] elt, device
 *   k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim], device,
 *                  written in place
 *   slot_mapping : [num_tokens] int64, device; slot < 0 = padding, skipped.
 *                  Slots must be distinct within one call (else the row
 *                  written last is unspecified).
 * The copy is bit-exact.  head_dim * sizeof(elt) must be a multiple of 16 and
 * every pointer 16-byte aligned (slot_mapping 8-byte).
 */
PKV_API pkv_status pkv_kv_append(const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int64_t *slot_mapping,
                         int64_t num_tokens, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, pkv_dtype dtype,
                         int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_attention_plan -- the launch an attention call with these sizes makes
 * on the current device (kernel family, split-K partition, grid, workspace).
 * num_queries = 1 for decode.  Pure host computation plus device attribute
 * queries; enqueues nothing.
 */
PKV_API pkv_status pkv_attention_plan(int batch, int num_queries, int num_heads,
                              int num_kv_heads, int head_dim, int block_size,
                              int max_context_len, pkv_dtype dtype,
                              const pkv_options *options, pkv_plan *plan);

/*
 * pkv_attention_plan_for -- the same plan for a device with `num_sms` SMs
 * and `ctas_per_sm` resident CTAs of the chosen kernel (0 = estimate from
 * shared memory).  Needs no GPU.
 */
PKV_API pkv_status pkv_attention_plan_for(int batch, int num_queries, int num_heads,
                                  int num_kv_heads, int head_dim,
                                  int block_size, int max_context_len,
                                  pkv_dtype dtype, const pkv_options *options,
                                  int num_sms, int ctas_per_sm, pkv_plan *plan);

/*
 * pkv_attention_workspace_size -- device workspace bytes an attention call
 * with these sizes needs on the current device (the split-K partials: one
 * float32 output vector and one float32 log-sum-exp per query row and split;
 * when the last CTA of a sequence merges its splits, also one 32-bit arrival
 * counter per (sequence, KV head, row chunk), which every call zeroes on its
 * stream, by a small kernel enqueued just before the attention launch).
 * 0 when the plan does not split.  Nothing in the workspace needs to be
 * initialised by the caller.
 */
PKV_API pkv_status pkv_attention_workspace_size(int batch, int num_queries,
                                        int num_heads, int num_kv_heads,
                                        int head_dim, int block_size,
                                        int max_context_len, pkv_dtype dtype,
                                        const pkv_options *options,
                                        size_t *bytes);

/*
 * pkv_paged_decode_attention -- one query per sequence:
 *   out[b, h, :] = sum_i softmax_i(scale * <q[b,h], K_i>) V_i
 * over rows i < L_b of sequence b read through the block table, with the KV
 * head h / (num_heads / num_kv_heads) ("Inference part 1", sections "Why
 * attention matters", "PagedAttention", "Smaller KV caches"; the online
 * softmax of section "FlashAttention"; the split-K partition and merge of
 * section "FlashDecoding").
 *
 *   out, q        : [batch, num_heads, head_dim] elt, device
 *   block_table   : [batch, max_blocks_per_seq] int32, device
 *   context_lens  : [batch] int32, device, 0 <= L_b <= max_context_len
 *   max_context_len: host-side upper bound of context_lens (sizes the
 *                   split-K grid; no device read is made to find it)
 *   scale         : softmax scale; zero or negative selects 1/sqrt(head_dim),
 *                   the scale of standard attention; NaN or infinite is
 *                   PKV_ERR_INVALID_ARG
 *   workspace     : device buffer of pkv_attention_workspace_size() bytes
 *                   (may be NULL when that size is 0), 16-byte aligned; its
 *                   contents before the call do not matter
 *   options       : NULL or launch controls; error_word: NULL or device int32
 * Supported: head_dim in {64, 128, 256}, block_size 16, dtype F32/BF16/F16.
 */
PKV_API pkv_status pkv_paged_decode_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch,
    int num_heads, int num_kv_heads, int head_dim, int block_size,
    int64_t num_blocks, float scale, pkv_dtype dtype, void *workspace,
    size_t workspace_bytes, const pkv_options *options, int32_t *error_word,
    pkv_stream_t stream);

/*
 * pkv_spec_verify_attention -- num_queries = K + 1 queries per sequence (the
 * last accepted token and K drafts, "Inference part 2", section "Speculative
 * decoding"), causal among themselves: query j sees rows
 * i <= L_b - num_queries + j (the shifted mask tril(diagonal = Sk - Sq) of
 * "Inference part 1", section "KV cache").  The drafts' K/V rows must already
 * be in the cache (pkv_kv_append) and counted in context_lens.
 *
 *   out, q : [batch, num_queries, num_heads, head_dim] elt, device
 * Other arguments as for pkv_paged_decode_attention; num_queries = 1 is
 * exactly pkv_paged_decode_attention.
 */
PKV_API pkv_status pkv_spec_verify_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch,
    int num_queries, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, pkv_dtype dtype,
    void *workspace, size_t workspace_bytes, const pkv_options *options,
    int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_append_attention -- the cache write and the attention of one step in a
 * single launch: the num_queries new K/V rows of every sequence are written
 * at their positions L_b - num_queries .. L_b - 1 (through the block table)
 * and attended to, with the same results as pkv_kv_append followed by
 * pkv_spec_verify_attention (pkv_paged_decode_attention for num_queries = 1).
 * "Efficient Inference" (obvix) names this fusion (KV cache write +
 * attention); "Inference part 2", section "Kernel fusion and torch.compile":
 * a fused kernel saves a launch and a round trip through memory.
 *
 *   k_new, v_new : [batch, num_queries, num_kv_heads, head_dim] elt, device;
 *                  row (b, j) is sequence b's row L_b - num_queries + j
 *   k_cache, v_cache : written in place at those rows (the blocks must
 *                  already be in the block table)
 * Other arguments and layouts as for pkv_spec_verify_attention.  Rows at
 * negative positions (L_b < num_queries) are ignored.
 */
PKV_API pkv_status pkv_append_attention(
    void *out, const void *q, const void *k_new, const void *v_new, void *k_cache,
    void *v_cache, const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch, int num_queries,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, pkv_dtype dtype, void *workspace, size_t workspace_bytes,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_host_step_staging_size -- device bytes pkv_append_attention_host needs
 * for its staging buffer: room for the step's inputs (q, k_new, v_new,
 * block_table, context_lens), its output and the attention workspace, each
 * at a 256-byte boundary.  Enqueues nothing.  dtype F32/BF16/F16.
 */
PKV_API pkv_status pkv_host_step_staging_size(int batch, int num_queries, int num_heads,
                                              int num_kv_heads, int head_dim, int block_size,
                                              int max_blocks_per_seq, int max_context_len,
                                              pkv_dtype dtype, const pkv_options *options,
                                              size_t *bytes);

/*
 * pkv_append_attention_host -- one decode (or verify) step with the inputs
 * and the output in HOST memory: q_host, k_new_host, v_new_host,
 * block_table_host and context_lens_host (same layouts as for
 * pkv_append_attention) and out_host; pkv_append_attention runs on them
 * (the caches k_cache / v_cache are device memory, written in place).  A
 * buffer the GPU can address -- page-locked memory mapped into the device's
 * address space, as cudaHostAlloc / cudaHostRegister give it under unified
 * addressing; on GB300 the chip-to-chip link carries the accesses -- needs
 * no copy: the new rows, and q when the plan splits a sequence at most 4
 * ways, are read by the kernels in place, out_host is written in place, and
 * the block table, the lengths (read first by every CTA) and any other q
 * are pulled into `staging` by one gather kernel.  Any other
 * buffer takes one host-to-device copy into `staging` (the output: one copy
 * back).  All of it is enqueued on `stream`, and the call returns without
 * waiting: the caller synchronises the stream before it reads out_host or
 * rewrites the host inputs.
 *
 *   staging : device, 256-byte aligned, >= pkv_host_step_staging_size()
 *             bytes (PKV_ERR_WORKSPACE otherwise); owned by the caller and
 *             in use until the stream has passed this step
 * A copy that cannot be enqueued returns PKV_ERR_CUDA (the copies enqueued
 * before it stay enqueued).  Other errors as for pkv_append_attention.
 */
PKV_API pkv_status pkv_append_attention_host(
    void *out_host, const void *q_host, const void *k_new_host, const void *v_new_host,
    void *k_cache, void *v_cache, const int32_t *block_table_host, int max_blocks_per_seq,
    const int32_t *context_lens_host, int max_context_len, int batch, int num_queries,
    int num_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, pkv_dtype dtype, void *staging, size_t staging_bytes,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_tree_verify_attention -- verification of a candidate tree (Medusa):
 * "Inference part 2", section "Medusa": the candidates of a tree are
 * verified in one pass with tree attention, a mask that lets each candidate
 * attend only to its own ancestors.  The num_queries tree nodes of sequence
 * b occupy its last rows L_b - num_queries .. L_b - 1 (their K/V already
 * appended, node k at row L_b - num_queries + k); node j sees every earlier
 * (cached) row and tree row k exactly when bit k of
 * tree_mask[b * mask_batch_stride + j] is set (normally node j and its
 * ancestors).  The chain tree (bits 0..j) is pkv_spec_verify_attention.
 *
 *   tree_mask : device uint64 [batch, num_queries] (mask_batch_stride =
 *               num_queries) or [num_queries] shared by all sequences
 *               (mask_batch_stride = 0); 8-byte aligned
 *   num_queries <= 64.  Other arguments as for pkv_spec_verify_attention.
 */
PKV_API pkv_status pkv_tree_verify_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch,
    int num_queries, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, pkv_dtype dtype,
    const uint64_t *tree_mask, int64_t mask_batch_stride, void *workspace,
    size_t workspace_bytes, const pkv_options *options, int32_t *error_word,
    pkv_stream_t stream);

/*
 * FP8 E4M3 KV cache.  "Inference part 2" (brunomaga), section "KV cache
 * quantization": storing the cache in FP8 halves its size and the bytes read
 * at each decode step; section "Number formats": E4M3 is 1 sign / 4 exponent
 * / 3 mantissa bits, largest value 448.  Scheme (the pages leave it open):
 * one float scale per cache tensor, element value = code value * scale.
 *
 * pkv_kv_append_fp8 -- quantise and write the new rows: code = e4m3 nearest
 * to x / scale (IEEE float32 division, round to nearest even, saturating at
 * +-448).  k_new, v_new: [num_tokens, num_kv_heads, head_dim] of src_dtype
 * (F32/BF16/F16); caches: [num_blocks, num_kv_heads, block_size, head_dim]
 * bytes; other arguments as for pkv_kv_append.  head_dim % 16 == 0.
 */
PKV_API pkv_status pkv_kv_append_fp8(const void *k_new, const void *v_new, void *k_cache,
                                     void *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int num_kv_heads, int head_dim,
                                     int block_size, int64_t num_blocks, pkv_dtype src_dtype,
                                     float k_scale, float v_scale, int32_t *error_word,
                                     pkv_stream_t stream);

/*
 * pkv_paged_attention_fp8 -- decode (num_queries = 1) or causal verification
 * over FP8 E4M3 caches: the attention of pkv_spec_verify_attention with every
 * key element code * k_scale and every value element code * v_scale.  q and
 * out are of q_dtype (F32/BF16/F16), [batch, num_queries, num_heads,
 * head_dim]; head_dim 128 or 256.  Plans and workspace sizes: the plan and
 * workspace functions with dtype PKV_FP8_E4M3 (the plan is the one for
 * 16-bit q; the workspace size covers float32 q too).  Kernels: BF16/F16 q
 * run on the tensor-core kernel by default (codes widened exactly to f16, q
 * rescaled by a power of two per row into f16 range, f16 products with
 * float32 accumulation); F32 q, or PKV_KERNEL_SIMT, run the CUDA-core kernel
 * in float32.
 */
PKV_API pkv_status pkv_paged_attention_fp8(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch,
    int num_queries, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, pkv_dtype q_dtype,
    float k_scale, float v_scale, void *workspace, size_t workspace_bytes,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * Multi-head latent attention (MLA) decode.  "Inference part 1", section
 * "Smaller KV caches: MQA, GQA and MLA": each token's keys and values are
 * compressed into one latent vector c and only c is cached; with the key
 * and value up-projections absorbed into the query and output projections,
 * attention runs directly over the cached latents, which act as both keys
 * and values (multi-query attention with one large shared head).  A small
 * separate key part carries the rotary position ("KV cache, prefill va
 * decode", section 04: d_c = 512 latent and d_h^R = 64 rotary values per
 * token and layer).
 *
 * Cache: one tensor [num_blocks, block_size, latent_dim + rope_dim] elt,
 * row = [c ; k_rope], paged through the block table like the other caches.
 *   q   : [batch, num_heads, latent_dim + rope_dim] elt, device: the
 *         absorbed query [q_c ; q_r] of each head
 *   out : [batch, num_heads, latent_dim] elt, device: the latent output
 *         sum_i softmax_i(scale q_h . row_i) c_i (the caller applies the
 *         value up-projection and the output projection)
 * Supported: latent_dim 512, rope_dim 0 or 64, num_heads a multiple of 16,
 * block_size 16, dtype BF16 / F16 (PKV_ERR_UNSUPPORTED otherwise).  options:
 * only `stages` (3..5, 0 = 4) and `split_blocks` apply; the other fields
 * must be 0.  Other arguments, errors and the workspace (the split-K
 * partials, 256-byte aligned) as for pkv_paged_decode_attention; context
 * lengths above max_context_len are clamped and recorded, bad block ids
 * recorded and their rows ignored.
 */
/* The launch an MLA decode call with these sizes makes on the current device
 * (split-K partition, grid, ring depth, workspace); enqueues nothing. */
PKV_API pkv_status pkv_mla_plan(int batch, int num_heads, int latent_dim, int rope_dim,
                                int block_size, int max_context_len, pkv_dtype dtype,
                                const pkv_options *options, pkv_plan *plan);

PKV_API pkv_status pkv_mla_workspace_size(int batch, int num_heads, int latent_dim,
                                          int rope_dim, int block_size, int max_context_len,
                                          pkv_dtype dtype, const pkv_options *options,
                                          size_t *bytes);

PKV_API pkv_status pkv_mla_decode_attention(
    void *out, const void *q, const void *ckv_cache, const int32_t *block_table,
    int max_blocks_per_seq, const int32_t *context_lens, int max_context_len, int batch,
    int num_heads, int latent_dim, int rope_dim, int block_size, int64_t num_blocks,
    float scale, pkv_dtype dtype, void *workspace, size_t workspace_bytes,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_mla_append -- write new tokens' latent rows [c ; k_rope] into their
 * slots of the latent cache (the same slot rule and error behaviour as
 * pkv_kv_append, with one cache and no heads).
 *   ckv_new   : [num_tokens, width] elt, device
 *   ckv_cache : [num_blocks, block_size, width] elt, device, written in place
 * width * sizeof(elt) must be a multiple of 16 and pointers 16-byte aligned.
 */
PKV_API pkv_status pkv_mla_append(const void *ckv_new, void *ckv_cache,
                                  const int64_t *slot_mapping, int64_t num_tokens, int width,
                                  int block_size, int64_t num_blocks, pkv_dtype dtype,
                                  int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_paged_prefill_attention -- chunked prefill: each sequence brings a
 * chunk of new query rows whose K and V have already been appended
 * (pkv_kv_append), and every row attends to the cache up to itself
 * ("Inference part 1", sections "KV cache" and "Chunked prefill"; the
 * arithmetic of its section "FlashAttention").
 *   q, out       [total_q, num_heads, head_dim] of dtype (BF16 or F16),
 *                16-byte aligned; the rows of sequence b are
 *                query_start[b] .. query_start[b + 1] - 1 (q_len_b rows).
 *   query_start  device int32 [batch + 1], non-decreasing, query_start[0] >= 0,
 *                query_start[batch] <= total_q, each q_len_b <= max_query_len.
 *   context_lens device int32 [batch]: rows in sequence b's cache, the
 *                chunk's own rows included (L_b >= q_len_b).
 *   Row j of sequence b sees cache rows i <= L_b - q_len_b + j.
 *   scale: the softmax scale; zero or negative selects 1/sqrt(head_dim);
 *          NaN or infinite is PKV_ERR_INVALID_ARG.
 *   head_dim 64 or 128; block_size 16; num_heads / num_kv_heads must divide
 *   128.  No workspace: the work is split over query rows (256 per CTA),
 *   not over keys.  options: only `stages` is read: the K/V ring depth
 *   in chunks, which also picks the chunk (head_dim 128: 6 or 8 stages of
 *   64 keys, 3-5 of 128; head_dim 64: 12 or 16 of 64, 4, 6 or 8 of 128;
 *   0 = 8 or 12 stages of 64 keys); any other value is PKV_ERR_UNSUPPORTED.  Runs on the fifth-generation tensor cores (tcgen05), S and O in
 *   tensor memory, P rounded to dtype.
 * A sequence whose query_start / context_lens break these rules is skipped
 * (its rows are not written) and recorded as PKV_DEVERR_CONTEXT_LEN; an
 * out-of-range block id is recorded as PKV_DEVERR_BLOCK_ID and its keys are
 * ignored.  Argument errors return synchronously with nothing enqueued.
 */
PKV_API pkv_status pkv_paged_prefill_attention(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, const int32_t *query_start, int max_query_len,
    int batch, int total_q, int num_heads, int num_kv_heads, int head_dim,
    int block_size, int64_t num_blocks, float scale, pkv_dtype dtype,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * pkv_read_error_word -- copy the device error word to *host_code after all
 * work on `stream` (synchronises the stream; not for the hot path).
 */
PKV_API pkv_status pkv_read_error_word(const int32_t *error_word, int32_t *host_code,
                               pkv_stream_t stream);

/*
 * pkv_check_bounded_wait -- exercise the give-up path of the kernels' waits.
 * Every wait on an mbarrier in this library's kernels is bounded: past its
 * time limit it records PKV_DEVERR_TIMEOUT in the error word and the kernel
 * returns, so a lost completion never hangs the GPU.  This call launches one
 * thread that waits, through the same wait loop, on a barrier nothing ever
 * arrives on, for limit_us microseconds (1 .. 10^7); afterwards the error
 * word holds PKV_DEVERR_TIMEOUT (if it held 0) and *waited_ns (optional,
 * device memory) the time the wait took.  Asynchronous on `stream`.
 */
PKV_API pkv_status pkv_check_bounded_wait(int32_t *error_word, uint32_t limit_us,
                                          uint64_t *waited_ns, pkv_stream_t stream);

/*
 * pkv_paged_decode_attention_noalloc -- pkv_paged_decode_attention for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * of this call; it exists for callers such as a plugin inside a host
 * framework that owns every device allocation, or a latency-critical loop
 * that must not call cudaMalloc / cudaFree (they can synchronise the device
 * and fail under memory pressure), and so cannot provide the split-K
 * workspace.
 *
 * Same arguments and results as pkv_paged_decode_attention minus the
 * workspace: the split-K partials go to a scratch array of
 * PKV_NOALLOC_SCRATCH_BYTES that the library holds in device memory (a
 * file-scope __device__ array, present on every GPU that loads the library
 * until the process exits).  The call allocates nothing and calls no
 * allocating routine.
 *   - If the plan's partials need more than PKV_NOALLOC_SCRATCH_BYTES (see
 *     pkv_attention_workspace_size), it returns PKV_ERR_WORKSPACE with
 *     nothing enqueued; a larger split_blocks in `options` shrinks the need.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.  With lazy module loading (the CUDA default), that
 *     lookup may also be what loads the library's device code on the device
 *     and commits the array's memory, so it can fail under memory pressure
 *     (PKV_ERR_CUDA): make the first call at start-up.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero: every partial is written before
 *     it is read within a call, and the split-K arrival counters are zeroed
 *     by each call on its stream before its attention kernel counts in them.
 *     Calls whose work overlaps on the GPU (other streams, other threads)
 *     race on it: serialise them.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)
PKV_API pkv_status pkv_paged_decode_attention_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_table, int max_blocks_per_seq,
    const int32_t *context_lens, int max_context_len, int batch,
    int num_heads, int num_kv_heads, int head_dim, int block_size,
    int64_t num_blocks, float scale, pkv_dtype dtype,
    const pkv_options *options, int32_t *error_word, pkv_stream_t stream);

/*
 * ---- Block manager (host) and copy-on-write (device) ----------------------
 * "KV cache, prefill và decode" (blog.truongducdung.dev), section 05, "Block
 * table", "Chia sẻ block và copy-on-write" and "Prefix caching"; "Inference
 * part 1", section "Prefix caching"; "Efficient Inference", the paged
 * attention section.  The pages fix: fixed-size blocks, a new block only
 * when a sequence's last one is full; a reference count per physical block;
 * sequences forked from one prompt share its blocks and copy a shared block
 * before writing into it; a full block is identified by a hash of its tokens
 * chained with its parent block's hash, and a prompt's lookup walks its
 * blocks from the start to the first miss, reusing each hit (reference
 * count + 1); finished requests return their blocks to the free pool.
 * Readings of this library where the pages are silent:
 *   - free blocks are reused last-freed first;
 *   - a block is cached (registered under its hash) the moment it is full;
 *     a second full block with the same hash is not merged;
 *   - cached blocks that no sequence holds stay reusable until the pool runs
 *     dry, then the least recently used goes first (ties: lower id); a hit
 *     or a release is a use;
 *   - hash = 64-bit FNV-1a over (parent hash as 8 little-endian bytes, 0 for
 *     the first block) then the block's token ids as 4 little-endian bytes.
 * The manager is host memory only and not thread-safe: serialise calls on
 * one manager.  Block ids index the caches' first dimension.  A call that
 * returns PKV_ERR_HOST_MEMORY (the host ran out of memory part-way) may have
 * left the manager inconsistent: destroy it.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_blocks blocks of block_size tokens, all free; NULL on a
 * bad size or allocation failure.  Destroy frees it (NULL is a no-op). */
PKV_API pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size);
PKV_API void pkv_bm_destroy(pkv_block_manager *m);

/*
 * pkv_bm_add_sequence -- a new sequence `seq_id` holding the n tokens of a
 * prompt.  With use_prefix_cache, its leading full blocks whose hash chain is
 * cached are shared (*cached_tokens = their token count, a multiple of the
 * block size; the caller prefills only the rest).  slots[0 .. n - cached)
 * receive the cache slots (block * block_size + offset) of tokens
 * cached .. n - 1, in order: the slot_mapping of pkv_kv_append.
 * PKV_ERR_INVALID_ARG for a known seq_id; PKV_ERR_WORKSPACE when the pool
 * cannot hold the prompt (nothing changes).
 */
PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager *m, int64_t seq_id,
                                       const int32_t *tokens, int n, int use_prefix_cache,
                                       int *cached_tokens, int64_t *slots);

/*
 * pkv_bm_append -- append n tokens to a sequence (decode: n = 1; verify:
 * K + 1).  slots[0 .. n) receive their cache slots.  If the sequence's last
 * block is partly filled and shared, it is first replaced by a copy: one
 * (cow_src[0], cow_dst[0]) pair, *num_cow = 1, which the caller must copy
 * (pkv_copy_blocks) before writing the new rows; else *num_cow = 0.
 * PKV_ERR_WORKSPACE when the pool is short (nothing changes).
 */
PKV_API pkv_status pkv_bm_append(pkv_block_manager *m, int64_t seq_id, const int32_t *tokens,
                                 int n, int64_t *slots, int32_t *cow_src, int32_t *cow_dst,
                                 int *num_cow);

/* pkv_bm_fork -- sequence `child` shares all of `parent`'s blocks (parallel
 * sampling; every block's reference count + 1). */
PKV_API pkv_status pkv_bm_fork(pkv_block_manager *m, int64_t parent, int64_t child);

/* pkv_bm_free -- drop a sequence: its blocks' counts - 1; blocks reaching 0
 * return to the pool (cached ones stay reusable until evicted). */
PKV_API pkv_status pkv_bm_free(pkv_block_manager *m, int64_t seq_id);

/* pkv_bm_sequence -- a sequence's blocks (blocks[0 .. *num_blocks), NULL to
 * query the count) and token count. */
PKV_API pkv_status pkv_bm_sequence(const pkv_block_manager *m, int64_t seq_id, int32_t *blocks,
                                   int max_blocks, int *num_blocks, int *num_tokens);

/* pkv_bm_block_table -- the block_table [num_seqs, max_blocks_per_seq]
 * (unused entries -1) and context_lens [num_seqs] of the attention calls,
 * for the listed sequences. */
PKV_API pkv_status pkv_bm_block_table(const pkv_block_manager *m, const int64_t *seq_ids,
                                      int num_seqs, int32_t *table, int max_blocks_per_seq,
                                      int32_t *context_lens);

/* Counts: free (unreferenced, uncached) blocks, cached blocks, sequences. */
PKV_API pkv_status pkv_bm_stats(const pkv_block_manager *m, int64_t *free_blocks,
                                int64_t *cached_blocks, int64_t *num_sequences);

/* One block's reference count, whether it is cached, and its hash (valid
 * once the block has been full). */
PKV_API pkv_status pkv_bm_block_info(const pkv_block_manager *m, int32_t block, int32_t *ref,
                                     int32_t *cached, uint64_t *hash);

/* The block hash of the chain rule above, for n tokens after parent_hash. */
PKV_API uint64_t pkv_bm_hash(uint64_t parent_hash, const int32_t *tokens, int n);

/*
 * pkv_copy_blocks -- copy whole blocks src[i] -> dst[i] (i < num_pairs) in
 * both device caches [num_blocks, num_kv_heads, block_size, head_dim] of
 * dtype (any cache type): the copies of copy-on-write.  src / dst: device
 * int32 arrays; destinations distinct and not among the sources.
 * Out-of-range ids are skipped and recorded (PKV_DEVERR_BLOCK_ID).
 */
PKV_API pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src,
                                   const int32_t *dst, int num_pairs, int num_kv_heads,
                                   int head_dim, int block_size, int64_t num_blocks,
                                   pkv_dtype dtype, int32_t *error_word, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
