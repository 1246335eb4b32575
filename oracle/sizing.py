"""Closed forms for paged KV-cache sizing -- TEST INFRASTRUCTURE ONLY.

Stated from:
  * "gpu_paged_kv_cache" (aicassindra), "Sizing the pool": K and V of one
    token in one layer take 2 x kv_heads x head_dim x bytes; a token in all
    layers multiplies that by the layer count, a block by the block size;
    a memory budget holds budget // (bytes of a block) blocks.  "Fixed-size
    blocks ...": a table entry is 32 bits per block; a sequence leaves fewer
    than B tokens of its last block unused.
  * "PagedAttention internals" (manishklach), sections 01-05: the same
    per-token formula; expected internal waste (B - 1) / 2 tokens; table
    entries and gather-loop iterations = ceil(tokens / B).
  * "KV Cache & PagedAttention" (lattice-ai-eng), section 3.2 / flashcard:
    total cache = 2 * layers * kv_heads * head_dim * seq_len * batch * bytes.
"""
from __future__ import annotations


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return 2 * layers * kv_heads * head_dim * dtype_bytes


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int, seq_len: int, batch: int = 1,
                   dtype_bytes: int = 2) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, dtype_bytes) * seq_len * batch


def block_bytes(layers: int, kv_heads: int, head_dim: int, dtype_bytes: int, block_size: int) -> int:
    return kv_bytes_per_token(layers, kv_heads, head_dim, dtype_bytes) * block_size


def pool_blocks(kv_budget_bytes: int, bytes_per_block: int) -> int:
    return kv_budget_bytes // bytes_per_block


def blocks_for_tokens(tokens: int, block_size: int) -> int:
    """Table entries (= gather-loop iterations per head) for a sequence."""
    return -(-tokens // block_size)


def table_bytes(tokens: int, block_size: int, entry_bytes: int = 4) -> int:
    return blocks_for_tokens(tokens, block_size) * entry_bytes


def internal_waste_tokens(tokens: int, block_size: int) -> int:
    """Unused slots in the last partial block (at most block_size - 1)."""
    return blocks_for_tokens(tokens, block_size) * block_size - tokens


def expected_internal_waste(block_size: int) -> float:
    """Mean unused slots per sequence when lengths are uniform mod block_size."""
    return (block_size - 1) / 2


def shared_prefix_blocks(prefix_tokens: int, block_size: int) -> int:
    """Whole blocks a prefix can share (sharing is block-aligned from token 0)."""
    return prefix_tokens // block_size
