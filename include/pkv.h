/*
 * pkv.h -- C ABI of libpkv: the paged KV-cache decode hot path on one GPU
 * (NVIDIA GB300, sm_103a).
 *
 * The operations follow four web pages on paged KV caches (vLLM's
 * PagedAttention):
 *   [P1] "gpu_paged_kv_cache" (aicassindra.com)
 *   [P2] "PagedAttention internals: blocks, copy-on-write" (manishklach)
 *   [P3] "tm_paged_attention" (aicassindra.com)
 *   [P4] "KV Cache & PagedAttention" (lattice-ai-eng)
 *
 * Common conventions
 *   - Every pointer argument is a DEVICE pointer unless its comment says host.
 *   - The caller owns all memory.  The library allocates nothing, keeps no
 *     pointer after a call returns, never synchronises the device, and
 *     launches its kernels only on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Calls are asynchronous: a PKV_OK return means
 *     the arguments were valid and the kernels were launched.
 *   - A KV pool holds blocks of [block_size][num_kv_heads][head_dim]
 *     elements, head_dim innermost and contiguous [P1 "The write path"].  A
 *     "slot" is one row of num_kv_heads * head_dim elements; slot = block *
 *     block_size + offset [P1 "The write path"].  Consecutive blocks are
 *     block_stride elements apart:
 *       - block_stride = 0 (dense, block_size * num_kv_heads * head_dim):
 *         one K and one V tensor per layer [P1 "Sizing the pool"],
 *         [num_blocks][block_size][num_kv_heads][head_dim];
 *       - block_stride = num_layers * block_size * num_kv_heads * head_dim:
 *         one layer's view of a pool that keeps all layers of a block
 *         together, [num_blocks][num_layers][block_size][num_kv_heads]
 *         [head_dim] per K and per V as in the numpy sketch of [P4 section
 *         4]; the layer-l pool pointer is base + l * block_size *
 *         num_kv_heads * head_dim.
 *     Any other block_stride >= the dense one and a multiple of 8 elements
 *     works too.  Pool pointers are 16-byte aligned.
 *   - block_size is 8, 16, 32 or 64 tokens; 16 is the usual choice [P1
 *     "Fixed-size blocks"; P2 section 02].  FP8 pools and the balanced
 *     split take 16 only.
 *   - Elements are IEEE binary16 (PKV_F16) or bfloat16 (PKV_BF16).  Queries
 *     have the pools' type.
 *   - dev_status, when not NULL, is a device int32 into which kernels OR the
 *     PKV_DEV_ERR_* bits below when they meet an out-of-range index or a
 *     timed-out wait.  The offending element is skipped (nothing outside the
 *     caller's buffers is read or written).  The caller zeroes it and reads
 *     it after synchronising.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer */
  PKV_ERR_UNSUPPORTED = 2,   /* block_size not 8/16/32/64, head_dim not 64/128, group > 8 ... */
  PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than pkv_decode_workspace_bytes */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
  PKV_ERR_OUT_OF_BLOCKS = 5  /* block manager: not enough free blocks (pool exhausted) */
} pkv_status;

typedef enum pkv_dtype { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_ERR_SLOT 1u     /* write_cache: slot >= num_blocks * block_size or < -1 */
#define PKV_DEV_ERR_PAIR 2u     /* copy_blocks: src or dst outside [0, num_blocks) */
#define PKV_DEV_ERR_BLOCK 4u    /* decode: block-table entry outside [0, num_blocks) */
#define PKV_DEV_ERR_LENGTH 8u   /* decode: context length < 0 or > the table / max_context_len */
#define PKV_DEV_ERR_TIMEOUT 16u /* decode: a wait for a tile copy exceeded its time limit */
#define PKV_DEV_ERR_SMEM 32u    /* decode: shared memory not 1024-byte aligned; kernel did nothing */

/*
 * pkv_write_cache -- the write path [P1 "The write path: slot mapping and
 * scatter"]: for every token i in [0, num_tokens) with slot_mapping[i] >= 0,
 *     k_pool[slot / B][slot % B][:][:] = k_new[i][:][:]
 *     v_pool[slot / B][slot % B][:][:] = v_new[i][:][:]
 * as a bitwise copy.  slot_mapping[i] == -1 marks a padding token (no write;
 * the pages leave padding open, this is the library's convention).  Slots
 * must be distinct within a call.
 *   k_new, v_new : [num_tokens][num_kv_heads][head_dim]; consecutive tokens
 *                  are new_row_stride elements apart (0 = dense, i.e.
 *                  num_kv_heads*head_dim), so rows of a fused QKV projection
 *                  can be passed directly.  Rows must be 16-byte aligned.
 *   k_pool, v_pool, block_stride : pools as above (one layer).
 *   slot_mapping : int32[num_tokens].
 * num_tokens == 0 is a no-op.  Out-of-range slots set PKV_DEV_ERR_SLOT.
 * num_tokens may be a whole prompt (the bulk write of prefill, [P3
 * "End-to-end flow"]: a 300-token prompt fills 19 blocks).
 */
pkv_status pkv_write_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                           int64_t block_stride, const int32_t* slot_mapping, int num_tokens,
                           int64_t new_row_stride,
                           int num_kv_heads, int head_dim, int block_size, int num_blocks,
                           pkv_dtype kv_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_copy_blocks -- the copy-on-write block copy [P1 "Prefix sharing,
 * reference counts, and copy-on-write"; P2 section 03; P3 "The
 * architecture"]: for each pair i, block pairs[2i+1] := block pairs[2i] in
 * both pools, bitwise, device to device.  A block is num_layers consecutive
 * [block_size][num_kv_heads][head_dim] slices: 1 for per-layer pools; the
 * layer count for the all-layer layout, whose copy-on-write moves every
 * layer of the block at once (k_pool, v_pool: the K and V bases).
 *   pairs : int32[num_pairs][2] = (src, dst).  dsts must be distinct and no
 *           dst may also be a src in the same call (a copy-on-write target is
 *           always a freshly allocated block).
 * num_pairs == 0 is a no-op.  Out-of-range pairs set PKV_DEV_ERR_PAIR and are
 * skipped.
 */
pkv_status pkv_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int num_pairs,
                           int num_layers, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, pkv_dtype kv_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_swap_blocks -- swap out / swap in of block lists ["gpu_paged_kv_cache",
 * "Reclaiming memory: swap versus recompute": a preempted victim's blocks
 * are copied to pinned host memory, freed, and copied back on resume; P2
 * section 05]: for each pair i, block pairs[2i+1] of the destination pool
 * := block pairs[2i] of the source pool, for K and for V, block_bytes bytes
 * each.  Swap out: source = the device pool, destination = a pool in
 * pinned host memory; swap in: the reverse, to whatever free device blocks
 * the block manager picked (the caller repoints the tables).  One kernel
 * moves the whole list, reading or writing the host pool through its
 * device mapping (NVLink-C2C on GB300).
 *   dst_k, dst_v / src_k, src_v : block 0 of each pool, 16-byte aligned,
 *                  device memory, managed memory or pinned (page-locked or
 *                  registered) host memory; pageable host memory is
 *                  rejected (PKV_ERR_INVALID_ARG).
 *   *_block_stride : bytes between consecutive blocks of that pool, a
 *                  multiple of 16 and >= block_bytes.
 *   *_num_blocks : blocks in that pool (pair indices are checked against it).
 *   block_bytes  : bytes per block and per K / V, a multiple of 16: one
 *                  layer's block (16 * H_kv * D * elem), a whole all-layer
 *                  block (times num_layers), or an FP8 pool's codes or scales.
 *   pairs        : int32[num_pairs][2] = (source block, destination block),
 *                  device or pinned host memory; destination blocks distinct.
 * Out-of-range pairs set PKV_DEV_ERR_PAIR and are skipped.
 */
pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, int64_t dst_block_stride, int dst_num_blocks,
                           const void* src_k, const void* src_v, int64_t src_block_stride,
                           int src_num_blocks, int64_t block_bytes, const int32_t* pairs, int num_pairs,
                           int32_t* dev_status, void* stream);

/* partition_size value selecting the balanced split (see pkv_decode_attention). */
#define PKV_PARTITION_BALANCED (-1)

/*
 * Bytes of workspace pkv_decode_attention needs for split-K partial results
 * (0 when every sequence fits one partition).  Host function.  For fixed
 * partitions it makes no GPU call; for PKV_PARTITION_BALANCED the size
 * depends on the current device's SM count, which it queries (assuming 256
 * SMs when no device answers).  Returns 0 for invalid sizes.
 */
size_t pkv_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim, int max_context_len,
                                  int partition_size);

/*
 * pkv_decode_attention -- single-query (decode) grouped-query attention
 * through block tables [P1 "Inside the paged attention kernel"; P2 section
 * 02; P3 "End-to-end flow"].  For each sequence s and query head h, with
 * G = num_q_heads / num_kv_heads, g = h / G (contiguous groups: a KV head is
 * shared by G consecutive query heads [P2 section 02]) and L = context_lens[s]
 * (the history including the token written this step [P3]):
 *     k_t = k_pool[block_tables[s][t / 16]][t % 16][g],  v_t likewise,
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . k_t) v_t,  t in [0, L).
 * L == 0 gives a zero row.  Sequences longer than partition_size tokens
 * are split into partitions of partition_size tokens that are computed
 * independently and merged by a second reduce kernel (the split-K
 * restructuring of [P1 "Inside the paged attention kernel"]).
 *   out          : [num_seqs][num_q_heads][head_dim], out_dtype F32/F16/BF16.
 *   q            : [num_seqs][num_q_heads][head_dim], kv_dtype, 4-byte aligned.
 *   k_pool, v_pool, block_stride : pools as above (one layer).
 *   block_tables : int32[num_seqs][max_blocks_per_seq], row-major; entries at
 *                  and past ceil(L/16) are not used (those within the row
 *                  may be read).
 *   context_lens : int32[num_seqs].
 *   scale        : softmax scale (typically 1/sqrt(head_dim)).
 *   partition_size : tokens per split-K partition, a multiple of 16; 0 for
 *                  one partition per sequence; or PKV_PARTITION_BALANCED
 *                  (-1): the library splits the whole batch into equal
 *                  contiguous shares of (block, KV head) tiles, one per warp
 *                  of a persistent grid (one CTA per SM), so every warp
 *                  streams the same number of bytes whatever the length mix;
 *                  sequences are cut wherever shares end (needs
 *                  num_seqs <= 4096).
 *   max_context_len : host-side upper bound on every context_lens[s]; it
 *                  sizes the grid and the workspace (no device read is made
 *                  on the host).  Longer sequences set PKV_DEV_ERR_LENGTH and
 *                  are truncated.
 *   workspace    : device scratch of at least pkv_decode_workspace_bytes()
 *                  bytes, 16-byte aligned (may be NULL when that is 0).  Its
 *                  contents need no initialisation.  Calls that share a
 *                  workspace must not overlap on the GPU.
 * Supported: head_dim 64 or 128, block_size 8, 16, 32 or 64 (16 only for
 * PKV_PARTITION_BALANCED), 1 <= G <= 8.
 * The two kernels run back to back on `stream`; pkv_decode_partitions and
 * pkv_decode_reduce below expose them separately.
 */
pkv_status pkv_decode_attention(void* out, const void* q, const void* k_pool, const void* v_pool,
                                int64_t block_stride, const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                float scale, int partition_size, int max_context_len,
                                void* workspace, size_t workspace_bytes, pkv_dtype kv_dtype,
                                pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_decode_partitions -- the first of the two kernels of
 * pkv_decode_attention (same arguments and meaning).  Sequences that fit one
 * partition get their final output row; longer ones leave per-partition
 * (running max, running sum, unnormalised accumulator) in the workspace for
 * pkv_decode_reduce.
 */
pkv_status pkv_decode_partitions(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 int64_t block_stride, const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 float scale, int partition_size, int max_context_len,
                                 void* workspace, size_t workspace_bytes, pkv_dtype kv_dtype,
                                 pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_decode_reduce -- the second kernel: merges the partial softmax states of
 * every (sequence, query head) row that was split (the small merge step that
 * follows split-K in [P1 "Inside the paged attention kernel"]):  M = max_p m_p,
 *     out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
 * Arguments as in pkv_decode_attention; it must follow pkv_decode_partitions
 * with the same sizes, workspace and stream, on the same device.  A no-op
 * when no row is split (fixed partitions).
 */
pkv_status pkv_decode_reduce(void* out, const int32_t* context_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int partition_size, int max_context_len,
                             const void* workspace, size_t workspace_bytes, pkv_dtype out_dtype,
                             int32_t* dev_status, void* stream);

/*
 * pkv_decode_step -- one decode step in one call: the write path of the token
 * generated this step for every sequence, then decode attention over the
 * history including it ([P1 "The write path"; P3 "End-to-end flow"]).  For
 * every sequence s with slot_mapping[s] equal to the slot of position
 * L-1 = context_lens[s]-1 through its block table, the result equals
 * pkv_write_cache (one token per sequence, rows k_new[s], v_new[s]) followed
 * by pkv_decode_attention; the write is fused into the attention kernel:
 * the warp that reads the tile holding position L-1 stores the new rows to
 * the pools and uses them directly, so no separate write kernel runs.
 * slot_mapping[s] == -1 means sequence s adds no token this step.  Any other
 * slot (a token not at the end of its sequence, as in chunked prefill) sets
 * PKV_DEV_ERR_SLOT and is not written: use pkv_write_cache for those.
 *   k_new, v_new : [num_seqs][num_kv_heads][head_dim], consecutive sequences
 *                  new_row_stride elements apart (0 = dense), rows 16-byte
 *                  aligned.
 *   k_pool, v_pool, block_stride : pools (read and written).
 *   other arguments as in pkv_decode_attention.
 * pkv_decode_step_partitions is its first kernel alone (follow it with
 * pkv_decode_reduce, as for pkv_decode_partitions).
 */
pkv_status pkv_decode_step(void* out, const void* q, const void* k_new, const void* v_new,
                           int64_t new_row_stride, void* k_pool, void* v_pool, int64_t block_stride,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, const int32_t* slot_mapping, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, float scale, int partition_size, int max_context_len,
                           void* workspace, size_t workspace_bytes, pkv_dtype kv_dtype,
                           pkv_dtype out_dtype, int32_t* dev_status, void* stream);

pkv_status pkv_decode_step_partitions(void* out, const void* q, const void* k_new, const void* v_new,
                                      int64_t new_row_stride, void* k_pool, void* v_pool, int64_t block_stride,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, const int32_t* slot_mapping,
                                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, float scale, int partition_size,
                                      int max_context_len, void* workspace, size_t workspace_bytes,
                                      pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status,
                                      void* stream);

/*
 * pkv_decode_attention_static_workspace -- pkv_decode_attention for callers
 * that cannot allocate device memory when they run decode (for example
 * plugins whose host framework owns all device memory and forbids
 * cudaMalloc during execution, or loops that cannot take the device-wide
 * synchronisation an allocation may cause).  The caller passes the same
 * inputs and outputs as for pkv_decode_attention but no workspace; the
 * split-K partials go to a fixed device array inside the library.
 * The paged-attention pages have no counterpart of this entry point.
 *   - The array holds PKV_STATIC_WORKSPACE_BYTES bytes on every GPU where the
 *     library is loaded, until the process exits.  A call whose
 *     pkv_decode_workspace_bytes() exceeds it returns PKV_ERR_WORKSPACE and
 *     launches nothing.
 *   - A call made outside stream capture (with its device current) looks up
 *     the array's device address and keeps it for that device; a call inside
 *     stream capture uses the kept address.  So make the first call on a
 *     device before any stream capture (a captured first call returns
 *     PKV_ERR_CUDA).  After cudaDeviceReset the next uncaptured call looks
 *     the address up again.
 *   - Every call shares the array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls whose kernels overlap on
 *     the GPU race on it: order them (one stream, or explicit events).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define PKV_STATIC_WORKSPACE_BYTES (16u << 20)
pkv_status pkv_decode_attention_static_workspace(
    void* out, const void* q, const void* k_pool, const void* v_pool, int64_t block_stride,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int num_blocks, float scale, int partition_size, int max_context_len,
    pkv_dtype kv_dtype, pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * ---------------------------------------------------------------- FP8 pools
 *
 * Pools of 8-bit e4m3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; largest finite magnitude 448; codes 0x7F/0xFF are NaN; no infinity)
 * in the dense per-layer [num_blocks][block_size][num_kv_heads][head_dim]
 * layout, one byte per element, halving the bytes decode reads ([P4 section 5]: K, V
 * stored in FP8).  The 16-token block is the quantisation group and its
 * scales ride with it, through copy-on-write included [P2 section 06,
 * "Blocks as quantization groups"]:
 *   k_scale, v_scale : float32 [num_blocks][num_kv_heads], device, 4-byte
 *                      aligned; element value = decode(code) * scale of its
 *                      (block, KV head).
 * The library never chooses a scale: the caller sets a block's scales when
 * it allocates the block (e.g. from a calibrated per-layer amax) and the
 * write path quantises new rows with them.  Pool pointers 16-byte aligned.
 *
 * num_layers (1..4096) selects the all-layer layout, one allocation per
 * pool holding every layer's rows of a block together:
 *   codes  [num_blocks][num_layers][16][num_kv_heads][head_dim],
 *   scales [num_blocks][num_layers][num_kv_heads].
 * pkv_write_cache_fp8 and the decode entry points then take layer l's base
 * pointers (codes + l * 16 * num_kv_heads * head_dim bytes, scales +
 * l * num_kv_heads floats): block b of the layer starts num_layers times
 * further apart than in a one-layer pool.  pkv_copy_blocks_fp8 takes the
 * whole pools and copies a block's rows and scales of every layer.
 * num_layers = 1 is the per-layer layout above.  Out of range:
 * PKV_ERR_INVALID_ARG.
 */

/*
 * pkv_write_cache_fp8 -- the write path into FP8 pools: for every token i
 * with slot_mapping[i] >= 0 (b = slot / 16, o = slot % 16) and KV head g,
 *     k_pool[b][o][g][:] = e4m3(float32(k_new[i][g][:]) / k_scale[b][g])
 * (and V likewise), the division in IEEE float32, rounded to the nearest
 * code with ties to the even mantissa, magnitudes beyond 448 saturating to
 * +-448.  k_new, v_new hold new_dtype (PKV_F16 / PKV_BF16) values, rows
 * 16-byte aligned, new_row_stride as in pkv_write_cache.  head_dim must be a
 * multiple of 16.  Padding (-1) and error handling as pkv_write_cache.
 */
pkv_status pkv_write_cache_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                               const float* k_scale, const float* v_scale, const int32_t* slot_mapping,
                               int num_tokens, int64_t new_row_stride, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int num_layers, pkv_dtype new_dtype,
                               int32_t* dev_status, void* stream);

/*
 * pkv_copy_blocks_fp8 -- copy-on-write over FP8 pools: for each pair, block
 * dst := block src in both pools (bytes), and k_scale[dst][:] :=
 * k_scale[src][:], v_scale likewise (every layer's, with num_layers > 1).
 * Pair rules and errors as pkv_copy_blocks.
 */
pkv_status pkv_copy_blocks_fp8(void* k_pool, void* v_pool, float* k_scale, float* v_scale,
                               const int32_t* pairs, int num_pairs, int num_layers, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, int32_t* dev_status,
                               void* stream);

/*
 * pkv_decode_attention_fp8 -- pkv_decode_attention over FP8 pools:
 *     k_t = decode(k_pool[block_tables[s][t/16]][t%16][g]) * k_scale[that block][g],
 * v_t likewise, the rest as pkv_decode_attention (same workspace size from
 * pkv_decode_workspace_bytes, same split-K partials and reduce kernel).
 * q has q_dtype (PKV_F16 or PKV_BF16) and must be 16-byte aligned.
 * Supported: head_dim 128; fixed partitions (partition_size >= 0) or
 * PKV_PARTITION_BALANCED (the same equal tile shares per warp as for 16-bit
 * pools, num_seqs <= 4096).  Rows of tokens >= L in a sequence's last
 * block, NaN codes included, are never used.
 */
pkv_status pkv_decode_attention_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                    const float* k_scale, const float* v_scale,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int num_seqs, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                    int num_layers, float scale, int partition_size, int max_context_len,
                                    void* workspace, size_t workspace_bytes, pkv_dtype q_dtype,
                                    pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_decode_partitions_fp8 -- the first of the two kernels of
 * pkv_decode_attention_fp8 (same arguments); follow it with
 * pkv_decode_reduce exactly as pkv_decode_partitions.
 */
pkv_status pkv_decode_partitions_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                                     const float* k_scale, const float* v_scale,
                                     const int32_t* block_tables, int max_blocks_per_seq,
                                     const int32_t* context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                     int num_layers, float scale, int partition_size, int max_context_len,
                                     void* workspace, size_t workspace_bytes, pkv_dtype q_dtype,
                                     pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * pkv_decode_step_fp8 -- one decode step over FP8 pools in one call, as
 * pkv_decode_step: for every sequence s whose slot_mapping[s] is the slot of
 * position L-1 through its block table, the result equals
 * pkv_write_cache_fp8 (rows k_new[s], v_new[s], quantised with that
 * block's scales) followed by pkv_decode_attention_fp8.  The write is fused
 * into the partition kernel: the warp that reads the tile holding position
 * L-1 quantises the rows, stores the codes and uses them directly.
 * slot_mapping[s] == -1: no token; any other slot sets PKV_DEV_ERR_SLOT and
 * is not written.  k_new, v_new have q_dtype, [num_seqs][num_kv_heads][128],
 * rows 16-byte aligned, new_row_stride as in pkv_decode_step.
 * pkv_decode_step_partitions_fp8 is its first kernel alone (follow it with
 * pkv_decode_reduce).  Fixed partitions only: PKV_PARTITION_BALANCED returns
 * PKV_ERR_UNSUPPORTED (write with pkv_write_cache_fp8 and attend with
 * pkv_decode_attention_fp8 instead).
 */
pkv_status pkv_decode_step_fp8(void* out, const void* q, const void* k_new, const void* v_new,
                               int64_t new_row_stride, void* k_pool, void* v_pool, const float* k_scale,
                               const float* v_scale, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens,
                               const int32_t* slot_mapping, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int num_blocks,
                               int num_layers, float scale, int partition_size, int max_context_len, void* workspace,
                               size_t workspace_bytes, pkv_dtype q_dtype, pkv_dtype out_dtype,
                               int32_t* dev_status, void* stream);

pkv_status pkv_decode_step_partitions_fp8(void* out, const void* q, const void* k_new,
                                          const void* v_new, int64_t new_row_stride, void* k_pool,
                                          void* v_pool, const float* k_scale, const float* v_scale,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, const int32_t* slot_mapping,
                                          int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, int num_blocks, int num_layers,
                                          float scale, int partition_size, int max_context_len, void* workspace,
                                          size_t workspace_bytes, pkv_dtype q_dtype,
                                          pkv_dtype out_dtype, int32_t* dev_status, void* stream);

/*
 * ------------------------------------------------------------ block manager
 *
 * Host-side allocator of a pool's blocks (host functions, no GPU call): the
 * free list and reference counts of [P4 section 4]; prefix sharing by a
 * chained block hash [P1 "Prefix sharing, reference counts, and
 * copy-on-write"; P2 section 04]; copy-on-write of a shared tail block;
 * LRU eviction of cached blocks nobody references [P2 section 04]; a
 * watermark of blocks admissions may not take and swap bookkeeping [P1
 * "Reclaiming memory: swap versus recompute"].  It produces what the device
 * entry points consume: block-table rows, slot mappings and copy-on-write
 * pairs, for a whole batch at once with pkv_bm_decode_step; and the
 * operating signals of [P1 "Operating it"] with pkv_bm_get_stats.  Calls on
 * one manager are serialised by an internal lock.
 *
 * Functions returning int return a count (>= 0) on success or a negative
 * pkv_status: -PKV_ERR_INVALID_ARG (null manager, unknown or duplicate
 * sequence, null or short buffer, wrong state) or -PKV_ERR_OUT_OF_BLOCKS
 * (nothing was changed).
 *
 * Prefix cache: a full block (block_size tokens) is keyed by a hash of its
 * tokens chained onto the previous block's key, starting from the
 * request's extra_key (adapter identity, multimodal inputs: anything else
 * that changes the KV values), so a match means an identical history from
 * position 0.  A hit is also compared token for token.  Cached blocks with
 * no reference stay reusable until allocation needs them, least recently
 * used first; referenced blocks are never evicted.
 */
typedef struct pkv_bm pkv_bm;

/*
 * Blocks of a pool that fit kv_bytes of memory ("gpu_paged_kv_cache",
 * "Sizing the pool": the KV budget over the bytes of one block):
 *   floor(kv_bytes / (2 * num_layers * num_kv_heads * (block_size * head_dim
 *         * elem_bytes + (with_scales ? 4 : 0))))
 * -- K and V rows of every layer for block_size tokens, plus for FP8 pools
 * (elem_bytes 1, with_scales 1) a float K and V scale per layer and KV
 * head.  Pass num_layers = 1 for one layer's pool.  -1 on a non-positive
 * size.  Host function.
 */
int64_t pkv_pool_blocks(uint64_t kv_bytes, int num_layers, int block_size, int num_kv_heads, int head_dim,
                        int elem_bytes, int with_scales);

/* A manager of num_blocks blocks of block_size tokens; watermark_blocks are
 * kept back from admissions (add_sequence, swap_in).  NULL on bad sizes
 * (non-positive, a watermark above num_blocks, or num_blocks * block_size
 * slots beyond the int32 range). */
pkv_bm* pkv_bm_create(int num_blocks, int block_size, int watermark_blocks);
void pkv_bm_destroy(pkv_bm* bm);

/* Blocks that can be handed out (free + cached with no reference). */
int pkv_bm_available_blocks(pkv_bm* bm);
/* Blocks registered in the prefix cache (referenced or not). */
int pkv_bm_cached_blocks(pkv_bm* bm);
/* Reference count of a block. */
int pkv_bm_block_refcount(pkv_bm* bm, int block);

/*
 * Admits sequence seq_id with its prompt (host int32 tokens[num_tokens]):
 * the longest run of whole blocks from position 0 found in the prefix cache
 * is shared (refcount bump), the rest is allocated.  slots[num_tokens]
 * (host) receives each token's slot for pkv_write_cache (block * block_size
 * + offset), or -1 for a token already cached.  Returns the number of
 * cached prompt tokens (a multiple of block_size).
 */
int pkv_bm_add_sequence(pkv_bm* bm, int64_t seq_id, const int32_t* tokens, int num_tokens,
                        uint64_t extra_key, int32_t* slots);

/* child := a copy of parent sharing every block (parallel sampling, beams). */
int pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child);

/*
 * Appends one token (decode): *slot receives its slot; a fresh block is
 * taken when the tail is full; when the tail is shared (refcount > 1) it is
 * copied on write: a fresh block replaces it in the table and (*cow_src,
 * *cow_dst) is the pair for pkv_copy_blocks (else both -1).  A block that
 * becomes full is registered in the prefix cache.
 */
int pkv_bm_append(pkv_bm* bm, int64_t seq_id, int32_t token, int32_t* slot, int32_t* cow_src,
                  int32_t* cow_dst);

/*
 * One decode step's host bookkeeping for a batch, under one lock: appends
 * tokens[i] to sequence seq_ids[i] for i = 0 .. n-1 in order, exactly as n
 * calls of pkv_bm_append would, and writes the device step's inputs (host
 * arrays):
 *   slot_mapping[i]   the slot of the appended token;
 *   context_lens[i]   the sequence's length after the append;
 *   block_tables[i][max_blocks_per_seq]   its table row, padded with pad_value;
 *   cow_pairs[k][2]   (src, dst) of each copy-on-write, in batch order, for
 *                     pkv_copy_blocks; room for n pairs.
 * Returns the number of copy-on-write pairs.  All or nothing: unknown,
 * swapped-out or repeated sequences, or a table wider than
 * max_blocks_per_seq after the append, return -PKV_ERR_INVALID_ARG, and too
 * few blocks for the batch returns -PKV_ERR_OUT_OF_BLOCKS; either way
 * nothing changes.  A tail shared by several sequences of the batch is
 * copied by the first that appends; the last holder then owns it.
 */
int pkv_bm_decode_step(pkv_bm* bm, const int64_t* seq_ids, const int32_t* tokens, int n,
                       int32_t* slot_mapping, int32_t* context_lens, int32_t* block_tables,
                       int max_blocks_per_seq, int32_t pad_value, int32_t* cow_pairs);

/*
 * Operating signals of a manager ("gpu_paged_kv_cache", "Operating it": KV
 * utilisation, preemption rate, prefix hit ratio, blocks per sequence).
 * Gauges describe the state at the call; counters accumulate from creation.
 *   blocks_referenced / num_blocks           KV utilisation by blocks;
 *   slots_holding_tokens / (blocks_referenced * block_size)
 *                                            fill of the referenced blocks
 *                                            (1 - internal waste);
 *   prompt_tokens_cached / prompt_tokens     prefix hit ratio;
 *   swap_outs, refusals                      preemption pressure;
 *   table_entries / sequences_resident, max_blocks_per_sequence
 *                                            blocks per sequence.
 */
typedef struct pkv_bm_stats {
  int64_t num_blocks, block_size;
  int64_t blocks_free;                /* on the free list */
  int64_t blocks_cached_unreferenced; /* cached, no reference: reusable, evicted LRU first */
  int64_t blocks_referenced;          /* held by at least one resident sequence */
  int64_t blocks_cached;              /* in the prefix cache, referenced or not */
  int64_t slots_holding_tokens;       /* slots of referenced blocks holding a resident token */
  int64_t sequences_resident, sequences_swapped;
  int64_t table_entries;              /* sum of resident sequences' table lengths */
  int64_t max_blocks_per_sequence;
  /* counters */
  int64_t prompt_tokens;              /* admitted prompt tokens */
  int64_t prompt_tokens_cached;       /* of which found in the prefix cache */
  int64_t evictions;                  /* cached blocks taken back for new contents */
  int64_t cow_copies;                 /* copy-on-write pairs handed out */
  int64_t swap_outs;
  int64_t refusals;                   /* PKV_ERR_OUT_OF_BLOCKS returns */
} pkv_bm_stats;

/* Fills *out (host).  PKV_OK, or -PKV_ERR_INVALID_ARG for a NULL argument. */
int pkv_bm_get_stats(pkv_bm* bm, pkv_bm_stats* out);

/* Releases a sequence (its blocks' references). */
int pkv_bm_free_sequence(pkv_bm* bm, int64_t seq_id);

/* Tokens in a sequence; its block-table row into out[capacity] (returns the
 * number of blocks). */
int pkv_bm_seq_len(pkv_bm* bm, int64_t seq_id);
int pkv_bm_block_table(pkv_bm* bm, int64_t seq_id, int32_t* out, int capacity);
/* A sequence's token history (swapped out or not) into out[capacity];
 * returns its length. */
int pkv_bm_seq_tokens(pkv_bm* bm, int64_t seq_id, int32_t* out, int capacity);

/*
 * Swap: pkv_bm_swap_out lists the sequence's blocks in blocks[] (logical
 * order; move them to host memory with pkv_swap_blocks before they are
 * reused) and releases them; the sequence keeps its tokens.
 * pkv_bm_swap_in takes fresh blocks for it (blocks[i] receives logical
 * block i: move host block i there) and returns their number.
 */
int pkv_bm_swap_out(pkv_bm* bm, int64_t seq_id, int32_t* blocks, int capacity);
int pkv_bm_swap_in(pkv_bm* bm, int64_t seq_id, int32_t* blocks, int capacity);

/*
 * pkv_bm_swap_in with the prefix cache: the sequence's full blocks from
 * position 0 whose contents are still cached (by the admission rule, up to
 * the first miss) are shared again with a reference bump instead of being
 * copied back; the rest take fresh blocks.  blocks[i] receives logical
 * block i and from_host[i] is 1 when host block i must be moved there, 0
 * when the block already holds it.  Returns the number of blocks.  Swap-out
 * still moves every block: a shared block may be evicted before the
 * resume, and the host copy is then the only one.
 *
 * Preemption by recompute ("gpu_paged_kv_cache", "Reclaiming memory: swap
 * versus recompute") is the same pair of calls without the copies: skip the
 * move at pkv_bm_swap_out, and at the resume recompute (prefill) the K/V of
 * the tokens in the blocks whose from_host is 1 -- token t of logical block
 * i goes to slot blocks[i] * block_size + t % block_size -- from the history
 * pkv_bm_seq_tokens returns.  Cached prefix blocks need neither.
 */
int pkv_bm_swap_in_cached(pkv_bm* bm, int64_t seq_id, int32_t* blocks, int32_t* from_host,
                          int capacity);

/*
 * pkv_check_bounded_wait -- exercises the decode kernels' error path for a
 * tile copy that never lands, without any copy in flight, with the bounded
 * wait (%globaltimer) the decode kernels use but for timeout_ns instead of
 * their fixed 2 s.  A diagnostic: lets a test (or a deployment's health
 * check) see that a stuck copy turns into a status bit rather than a hung
 * kernel, and that the context stays usable.
 *   shared_ring = 0: one warp sets up the partition kernel's per-warp tile
 *     ring and waits on its first stage, which nothing arms; when the wait
 *     runs out it drains its (zero) outstanding copies, ORs
 *     PKV_DEV_ERR_TIMEOUT into *dev_status and returns.
 *   shared_ring = 1: four warps share stage barriers, as the warps of the
 *     FP8 head-group kernel share one ring; three pass a barrier completed by
 *     a plain arrival, one waits on a barrier nothing completes until its
 *     limit runs out, and the CTA-wide vote that follows sends all four out
 *     with PKV_DEV_ERR_TIMEOUT set.
 * timeout_ns in [0, 2e9]; dev_status is required (device int32).  The pages
 * have no counterpart of this call.
 */
pkv_status pkv_check_bounded_wait(int64_t timeout_ns, int shared_ring, int32_t* dev_status, void* stream);

/* Static string naming a status code.  Host function. */
const char* pkv_status_string(pkv_status status);

/*
 * The CUDA error behind the calling thread's most recent PKV_ERR_CUDA
 * return: a cudaError_t value, or minus the CUresult of a failed
 * cuTensorMapEncodeTiled; 0 when this thread has had none.  Thread-local,
 * so concurrent callers each see their own.  pkv_cuda_error_name() names a
 * value returned here.
 */
int pkv_last_cuda_error(void);
const char* pkv_cuda_error_name(int code);

/* Library version, major * 10000 + minor * 100 + patch.  Host function. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
