// Internal declarations shared by the host entry points and the kernel
// translation units of libpkv.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pkv {

constexpr int kBlockSize = 16;  // tokens per KV block: the default, and the only size of FP8 pools and the
                                // balanced split
constexpr int kTile = 16;       // tokens per shared-memory tile (the MMA's 16 rows); a block of B tokens
                                // is B/16 tiles (B >= 16) or half a tile (B = 8)

struct WriteCacheArgs {
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* slot_mapping;
  int32_t* dev_status;
  int64_t k_stride;   // elements between consecutive new tokens
  int64_t v_stride;
  int64_t num_slots;  // num_blocks * block_size
  int64_t block_stride;  // pool elements between consecutive blocks (>= block_size * row_elems)
  int num_tokens;
  int row_elems;      // num_kv_heads * head_dim
  int block_shift;    // log2(block_size)
};

// FP8 pools: e4m3 codes plus one float scale per (block, KV head) for K and
// for V.  New rows arrive as 16-bit values and are quantised with their
// block's scale.
struct WriteCacheFp8Args {
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint8_t* k_pool;
  uint8_t* v_pool;
  const float* k_scale;  // [num_blocks][num_kv_heads]
  const float* v_scale;
  const int32_t* slot_mapping;
  int32_t* dev_status;
  int64_t stride;        // elements between consecutive new tokens
  int64_t num_slots;
  int64_t block_stride;  // pool bytes between consecutive blocks
  int64_t scale_stride;  // scales (floats) between consecutive blocks' rows
  int num_tokens;
  int num_kv_heads;
  int head_dim;
  int new_bf16;          // new rows: 0 = f16, 1 = bf16
};

// Block lists moved between two pools, each in device memory or in pinned
// host memory reached through its device-mapped address (swap out / in).
struct SwapBlocksArgs {
  uint8_t* dst_k;
  uint8_t* dst_v;
  const uint8_t* src_k;
  const uint8_t* src_v;
  const int32_t* pairs;  // [num_pairs][2] = (src block, dst block)
  int32_t* dev_status;
  int64_t dst_stride;    // bytes between consecutive blocks
  int64_t src_stride;
  int64_t block_bytes;   // bytes moved per block (multiple of 16)
  int num_pairs;
  int dst_num_blocks;
  int src_num_blocks;
};

struct CopyBlocksArgs {
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* pairs;
  int32_t* dev_status;
  int64_t block_elems;  // 16-bit units per block: num_layers * block_size * num_kv_heads * head_dim
                        // (FP8 pools: half the block's bytes)
  int num_pairs;
  int num_blocks;
  // FP8 pools only (null otherwise): per-block scales copied with the block.
  float* k_scale;
  float* v_scale;
  int scales_per_block;  // num_kv_heads
};

struct DecodeArgs {
  void* out;
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_acc;     // partial records [..][D]: unnormalised partial outputs
  float2* ws_ml;     // partial records: (running max in log2 units, running sum)
  int2* ws_meta;     // balanced split: per (s, g) pair (first warp, 2 * pieces + its slot)
  int32_t* dev_status;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int max_blocks_per_seq;
  int num_blocks;
  int partition_size;  // tokens, multiple of 16
  int max_parts;
  int max_context_len;
  int block_shift;       // log2(tokens per block): 3, 4, 5 or 6
  int64_t block_stride;  // pool elements between consecutive blocks (the fused write's addressing)
  float scale_log2;    // scale * log2(e)
  int out_dtype;       // pkv_dtype
  int balanced_ctas;   // balanced split: persistent CTAs (one per SM); 0 otherwise
  int unit_warps;      // fixed partitions: warps per unit (1 or 2)
  int heads_per_box;   // KV heads per TMA box: 2 or 4 (head-group kernels), or 1
  long long timeout_ns;
  // Fused decode step only: the token generated this step, written to the
  // pools by the attention kernel itself (null when not fusing).
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t new_stride;           // elements between consecutive sequences' new rows
  const int32_t* slot_mapping;  // [S]: slot of position L-1, or -1
  uint16_t* k_pool_w;
  uint16_t* v_pool_w;
  // FP8 pools only: per-(block, KV head) scales, block b's row at b * scale_stride.
  const float* k_scale;
  const float* v_scale;
  int64_t scale_stride;
};

// Split-K workspace layout (regions 256-byte aligned).  Fixed partitions:
// records [S][H_q][max_parts].  Balanced split: per-pair metadata [S][<=H_q]
// then records [W warps][2 slots][<= 8 heads].
struct WorkspaceLayout {
  size_t acc_offset, ml_offset, meta_offset, total;
};
WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_parts);
WorkspaceLayout balanced_workspace_layout(int num_seqs, int num_q_heads, int head_dim, int64_t warps);

// SM count of the current device, cached per device; `fallback` when no
// device answers.
int current_sm_count(int fallback);
// Warps of `kernel` (launched with `threads` threads and `smem` bytes of
// dynamic shared memory) that the current device holds at once: SMs x
// resident CTAs x warps per CTA.  Cached per kernel, device and shape;
// safe to call from several host threads.
int resident_warp_slots(const void* kernel, int threads, size_t smem);
// Raises a kernel's dynamic shared memory limit to `bytes` on the current
// device (once per kernel, device and size).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// Upper bound on the layers an FP8 all-layer pool holds per block (keeps the
// per-block scale count, layers x H_kv, well inside an int).
constexpr int kMaxLayers = 4096;

// Balanced split geometry (pkv_decode_balanced.cu).
constexpr int kBalancedMaxSeqs = 4096;
int balanced_warps_per_cta(int head_dim, int num_seqs);
size_t balanced_smem_bytes(int head_dim, int num_seqs);

// Launches `kernel` with programmatic stream serialisation allowed: it may
// start while the previous grid on the stream finishes, and must execute
// griddepcontrol.wait before touching memory that grid could write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_write_cache(const WriteCacheArgs& a, cudaStream_t stream);
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);
// kv_bf16: 0 = f16, 1 = bf16.  Tensor maps describe the K and V pools.
// KV heads per TMA box of the 16-bit fixed-partition path (DecodeArgs::
// heads_per_box): 2 or 4, the head-group kernel (pkv_decode_hg.cu), for
// blocks of >= 16 tokens, an even KV head count and a batch whose sequences x
// KV heads fit one wave of the partition kernel's warp slots (where it gives
// every unit one warp); 4 when it divides the KV head count and the grid
// (sequences x KV heads x partitions) spans more than four waves; else 1, the
// partition kernel.
int partitions_heads_per_box(const DecodeArgs& a, int head_dim, int kv_bf16);
cudaError_t launch_decode_partitions_hg(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                        int head_dim, int kv_bf16, cudaStream_t stream);
cudaError_t launch_decode_partitions(const DecodeArgs& a, const CUtensorMap& tmap_k,
                                     const CUtensorMap& tmap_v, int head_dim, int kv_bf16,
                                     cudaStream_t stream);  // fuses the write when a.k_new is set
cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t stream);
// One warp waits on a tile barrier that no copy arms, for timeout_ns, and
// sets PKV_DEV_ERR_TIMEOUT in *status (pkv_check_bounded_wait).
cudaError_t launch_bounded_wait_check(int32_t* status, long long timeout_ns, cudaStream_t stream);
// The shared-ring form: four warps, a CTA-wide vote after the wait (pkv_checks.cu).
cudaError_t launch_bounded_wait_vote_check(int32_t* status, long long timeout_ns, cudaStream_t stream);
// FP8 pools (pkv_decode_fp8.cu): tensor maps describe the uint8 pools;
// q_bf16: 0 = f16 queries, 1 = bf16.
cudaError_t launch_decode_partitions_fp8(const DecodeArgs& a, const CUtensorMap& tmap_k,
                                         const CUtensorMap& tmap_v, int head_dim, int q_bf16,
                                         cudaStream_t stream);
// KV heads per TMA box of the FP8 decode kernels (DecodeArgs::heads_per_box):
// 4, the head-group partition kernel (four heads' tiles of a block per
// copy), for write-then-attend calls with fixed partitions and a head count
// divisible by 4; else 1 (one head's tile per copy: the partition kernel,
// used by the fused step, and the balanced split).
int fp8_heads_per_box(int num_kv_heads, bool fused, bool balanced);

// PKV_PARTITION_BALANCED over FP8 pools (head_dim 128, no fused write): one
// CTA of balanced_fp8_warps_per_cta() warps per SM (a.balanced_ctas CTAs).
cudaError_t launch_decode_balanced_fp8(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                       int head_dim, int q_bf16, cudaStream_t stream);
int balanced_fp8_warps_per_cta();
cudaError_t launch_write_cache_fp8(const WriteCacheFp8Args& a, cudaStream_t stream);
cudaError_t launch_swap_blocks(const SwapBlocksArgs& a, cudaStream_t stream);
cudaError_t launch_decode_balanced(const DecodeArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                   int head_dim, int kv_bf16, cudaStream_t stream);
cudaError_t launch_decode_reduce_balanced(const DecodeArgs& a, int head_dim, cudaStream_t stream);

}  // namespace pkv
