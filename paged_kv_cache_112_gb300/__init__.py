"""GB300-native paged KV-cache decode path.

The work is done by libpkv (include/pkv.h), hand-written CUDA for sm_103a:
  write_cache       -- scatter new tokens' K/V into the block pool by slot
  copy_blocks       -- copy-on-write block copies
  decode_attention  -- single-query grouped-query attention through block
                       tables, split-K partitions + reduce
  decode_step       -- the new token's write fused into decode attention
  *_fp8             -- the same over FP8 (e4m3) pools with per-block scales
  swap_blocks       -- block lists between device pools and pinned host pools
  BlockManager      -- the host allocator (refcounts, copy-on-write, chained-hash
                       prefix cache with LRU eviction, watermark, swap bookkeeping)
This package only marshals torch tensors into the C ABI.
"""
from ._binding import (BlockManager, OutOfBlocks, PKV_ERR_OUT_OF_BLOCKS, DEV_ERR_BLOCK, DEV_ERR_LENGTH, DEV_ERR_PAIR, DEV_ERR_SLOT, DEV_ERR_SMEM, DEV_ERR_TIMEOUT,
                       PKV_BF16,
                       PKV_ERR_CUDA, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_F16, PKV_F32,
                       PKV_OK, PARTITION_BALANCED, PkvError, check_bounded_wait, copy_blocks, copy_blocks_fp8, decode_attention,
                       decode_attention_fp8, decode_partitions, decode_partitions_fp8, decode_reduce, decode_step,
                       decode_step_fp8, decode_step_partitions, decode_step_partitions_fp8,
                       decode_workspace_bytes, library_path, load, pool_blocks, status_string, swap_blocks,
                       write_cache,
                       write_cache_fp8)

__all__ = [
    "load", "library_path", "status_string", "write_cache", "copy_blocks", "decode_attention",
    "decode_partitions", "decode_reduce", "decode_step", "decode_step_partitions", "decode_workspace_bytes",
    "write_cache_fp8", "copy_blocks_fp8", "decode_attention_fp8", "decode_partitions_fp8", "decode_step_fp8",
    "decode_step_partitions_fp8", "swap_blocks", "check_bounded_wait", "pool_blocks", "BlockManager", "OutOfBlocks", "PkvError",
    "PKV_ERR_OUT_OF_BLOCKS",
    "PKV_OK", "PKV_ERR_INVALID_ARG", "PKV_ERR_UNSUPPORTED", "PKV_ERR_WORKSPACE", "PKV_ERR_CUDA",
    "PKV_F32", "PKV_F16", "PKV_BF16", "PARTITION_BALANCED",
    "DEV_ERR_SLOT", "DEV_ERR_PAIR", "DEV_ERR_BLOCK", "DEV_ERR_LENGTH", "DEV_ERR_TIMEOUT", "DEV_ERR_SMEM",
]
