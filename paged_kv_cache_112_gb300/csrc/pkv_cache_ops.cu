// Write path and copy-on-write block copy.
//
//  * write_cache: each new token's K and V rows go to the pool row named by
//    its slot (block number times the block size plus the offset inside the
//    block).  Because head_dim is the innermost axis of a pool row, a row
//    moves as whole 16-byte vectors even though consecutive tokens land in
//    unrelated blocks ("gpu_paged_kv_cache", section "The write path: slot
//    mapping and scatter").
//  * copy_blocks: before a sequence appends into a block it shares, the
//    block's contents are duplicated into a block of its own, which the
//    sequence's table then points to ("gpu_paged_kv_cache", section "Prefix
//    sharing, reference counts, and copy-on-write"; "PagedAttention
//    internals", section 03).
//
// Both are pure byte movers: every thread moves one 16-byte vector, adjacent
// threads move adjacent vectors of the same row (coalesced 128-byte lines on
// both sides).  Grids are capped at a multiple of the SM count and
// grid-stride over the work.
#include "pkv_fp8.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__device__ __forceinline__ void flag(int32_t* status, unsigned bit) {
  if (status) atomicOr(reinterpret_cast<unsigned*>(status), bit);
}

__global__ void __launch_bounds__(256) write_cache_kernel(WriteCacheArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // inputs may come from the previous grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int vec_per_row = a.row_elems / 8;  // 16-byte vectors per K (or V) row
  const int64_t total = static_cast<int64_t>(a.num_tokens) * 2 * vec_per_row;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(idx % vec_per_row);
    const int64_t r = idx / vec_per_row;
    const int which = static_cast<int>(r & 1);  // 0 = K, 1 = V
    const int64_t tok = r >> 1;
    // The row load does not depend on the slot: issue both loads together.
    const uint16_t* src = which ? a.v_new + tok * a.v_stride : a.k_new + tok * a.k_stride;
    const uint4 val = __ldg(reinterpret_cast<const uint4*>(src) + v);
    const int64_t slot = a.slot_mapping[tok];
    if (slot < 0) {
      if (slot != -1 && v == 0 && which == 0) flag(a.dev_status, 1u);  // PKV_DEV_ERR_SLOT
      continue;
    }
    if (slot >= a.num_slots) {
      if (v == 0 && which == 0) flag(a.dev_status, 1u);
      continue;
    }
    uint16_t* dst = (which ? a.v_pool : a.k_pool) + (slot >> a.block_shift) * a.block_stride +
                    (slot & ((1 << a.block_shift) - 1)) * a.row_elems;
    reinterpret_cast<uint4*>(dst)[v] = val;
  }
}

__global__ void __launch_bounds__(256) copy_blocks_kernel(CopyBlocksArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t vec_per_block = a.block_elems / 8;
  const int64_t total = static_cast<int64_t>(a.num_pairs) * 2 * vec_per_block;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = idx % vec_per_block;
    const int64_t r = idx / vec_per_block;
    const int which = static_cast<int>(r & 1);
    const int64_t pair = r >> 1;
    const int src = a.pairs[2 * pair];
    const int dst = a.pairs[2 * pair + 1];
    if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
      if (v == 0 && which == 0) flag(a.dev_status, 2u);  // PKV_DEV_ERR_PAIR
      continue;
    }
    uint16_t* pool = which ? a.v_pool : a.k_pool;
    const uint4 val = reinterpret_cast<const uint4*>(pool + src * a.block_elems)[v];
    reinterpret_cast<uint4*>(pool + dst * a.block_elems)[v] = val;
  }
  // FP8 pools: the block's scales travel with it ("PagedAttention
  // internals", section 06).
  if (a.k_scale) {
    const int64_t n = static_cast<int64_t>(a.num_pairs) * 2 * a.scales_per_block;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int h = static_cast<int>(idx % a.scales_per_block);
      const int64_t r = idx / a.scales_per_block;
      const int64_t pair = r >> 1;
      const int src = a.pairs[2 * pair];
      const int dst = a.pairs[2 * pair + 1];
      if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) continue;  // flagged above
      float* sc = (r & 1) ? a.v_scale : a.k_scale;
      sc[static_cast<int64_t>(dst) * a.scales_per_block + h] = sc[static_cast<int64_t>(src) * a.scales_per_block + h];
    }
  }
}

// FP8 write path: each thread quantises 16 consecutive elements of one new
// row (one head's slice) with the scale of the destination block and KV
// head (fp8::quantize4) and stores the 16 codes as one vector.
__global__ void __launch_bounds__(256) write_cache_fp8_kernel(WriteCacheFp8Args a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int row = a.num_kv_heads * a.head_dim;
  const int vec_per_row = row / 16;
  const int64_t total = static_cast<int64_t>(a.num_tokens) * 2 * vec_per_row;
  const bool bf16 = a.new_bf16 != 0;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(idx % vec_per_row);
    const int64_t r = idx / vec_per_row;
    const int which = static_cast<int>(r & 1);
    const int64_t tok = r >> 1;
    const uint4* src = reinterpret_cast<const uint4*>((which ? a.v_new : a.k_new) + tok * a.stride) + 2 * v;
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    const int64_t slot = a.slot_mapping[tok];
    if (slot < 0 || slot >= a.num_slots) {
      if (slot != -1 && v == 0 && which == 0) flag(a.dev_status, 1u);  // PKV_DEV_ERR_SLOT
      continue;
    }
    const int g = (v * 16) / a.head_dim;
    const float sc = (which ? a.v_scale : a.k_scale)[(slot / kBlockSize) * a.scale_stride + g];
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = fp8::quantize4(w[2 * i], w[2 * i + 1], sc, bf16);
    uint8_t* dst = (which ? a.v_pool : a.k_pool) + (slot / kBlockSize) * a.block_stride + (slot % kBlockSize) * row;
    reinterpret_cast<uint4*>(dst)[v] = make_uint4(c[0], c[1], c[2], c[3]);
  }
}

// Swap out / in ("gpu_paged_kv_cache", "Reclaiming memory: swap versus
// recompute"; "PagedAttention internals", section 05): for each pair (s, d),
// block d of the destination pool := block s of the source pool, K and V.
// One side is pinned host memory, read or written directly by the kernel
// through its mapped address (on GB300 over NVLink-C2C), so a whole block
// list moves in one launch.  Each thread moves 16-byte vectors; adjacent
// threads move adjacent vectors of one block.
__global__ void __launch_bounds__(256) swap_blocks_kernel(SwapBlocksArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t vec_per_block = a.block_bytes / 16;
  const int64_t total = static_cast<int64_t>(a.num_pairs) * 2 * vec_per_block;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t v = idx % vec_per_block;
    const int64_t r = idx / vec_per_block;
    const int which = static_cast<int>(r & 1);
    const int64_t pair = r >> 1;
    const int src = a.pairs[2 * pair];
    const int dst = a.pairs[2 * pair + 1];
    if (src < 0 || src >= a.src_num_blocks || dst < 0 || dst >= a.dst_num_blocks) {
      if (v == 0 && which == 0) flag(a.dev_status, 2u);  // PKV_DEV_ERR_PAIR
      continue;
    }
    const uint8_t* from = (which ? a.src_v : a.src_k) + src * a.src_stride;
    uint8_t* to = (which ? a.dst_v : a.dst_k) + dst * a.dst_stride;
    reinterpret_cast<uint4*>(to)[v] = reinterpret_cast<const uint4*>(from)[v];
  }
}

int grid_for(int64_t work_items, int threads) {
  const int sms = current_sm_count(148);
  const int64_t want = (work_items + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * 16;  // 16 resident 256-thread CTAs per SM at most
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_write_cache(const WriteCacheArgs& a, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(a.num_tokens) * 2 * (a.row_elems / 8);
  if (work == 0) return cudaSuccess;
  return launch_pdl(write_cache_kernel, dim3(grid_for(work, 256)), dim3(256), 0, stream, a);
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(a.num_pairs) * 2 * (a.block_elems / 8);
  if (work == 0) return cudaSuccess;
  return launch_pdl(copy_blocks_kernel, dim3(grid_for(work, 256)), dim3(256), 0, stream, a);
}

cudaError_t launch_swap_blocks(const SwapBlocksArgs& a, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(a.num_pairs) * 2 * (a.block_bytes / 16);
  if (work == 0) return cudaSuccess;
  return launch_pdl(swap_blocks_kernel, dim3(grid_for(work, 256)), dim3(256), 0, stream, a);
}

cudaError_t launch_write_cache_fp8(const WriteCacheFp8Args& a, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(a.num_tokens) * 2 * (a.num_kv_heads * a.head_dim / 16);
  if (work == 0) return cudaSuccess;
  return launch_pdl(write_cache_fp8_kernel, dim3(grid_for(work, 256)), dim3(256), 0, stream, a);
}

}  // namespace pkv
