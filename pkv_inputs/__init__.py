"""Seeded synthetic workloads for paged decode attention.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.
It holds no arithmetic of the method itself (no attention, no gather, no copy):
it draws context lengths and values, and it runs a small host-side block
pool (block stack, reference counts, copy-on-write decision) to build block
tables, the slot mapping of the new tokens and the copy-on-write pairs -- the
bookkeeping a scheduler does on the host each step.

Sources (four web pages on paged KV caches):
  * "gpu_paged_kv_cache" (aicassindra), sections "Fixed-size blocks and the
    block-table indirection", "The write path: slot mapping and scatter" and
    "Prefix sharing, reference counts, and copy-on-write".
  * "PagedAttention internals" (manishklach), sections 02 "Block tables" and
    03 "Sharing via copy-on-write".
  * "tm_paged_attention" (aicassindra), section "End-to-end flow": a sequence's
    context length counts the token generated this step; a new block is
    taken when the last one has no free row left.
  * "KV Cache & PagedAttention" (lattice-ai-eng), section 4 "Minimal
    implementation": free list, refcount, fork by refcount bump.

Layouts (shared contract with the library):
  k_pool, v_pool : uint16 payload of f16/bf16, [num_blocks, block_size, H_kv, D]
  q              : uint16 payload, [S, H_q, D]
  k_new, v_new   : uint16 payload, [T, H_kv, D]
  block_tables   : int32 [S, max_blocks_per_seq]; entries past ceil(L/B) are -1
  context_lens   : int32 [S]  (includes the token written this step)
  slot_mapping   : int32 [T]
  copy_pairs     : int32 [P, 2]  (src, dst)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16

# 16-bit quiet-NaN payloads used to poison memory no sequence may read.
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0}

# Workload recipes.  Lengths are the post-append context length L_s.
# partition_size is the split-K partition the step runs with: config 4's
# definition fixes 512; for the others it is the best of a sweep on the
# bench's step (256 to 2048 tokens).  partition_size_fp8, where given, is the
# same choice for FP8 pools (another kernel, a sweep of its own).
CONFIGS = {
    1: dict(name="tiny: S=4 L={1,17,33,50} 4q/2kv D=64 f16 NB=64",
            dtype="f16", num_seqs=4, num_q_heads=4, num_kv_heads=2, head_dim=64,
            lens=("fixed", [1, 17, 33, 50]), num_blocks=64, partition_size=0),
    2: dict(name="8B-class GQA decode layer: S=64 32q/8kv D=128 bf16 L~U[128,2048]",
            dtype="bf16", num_seqs=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
            lens=("uniform", 128, 2048), pool_factor=1.25, partition_size=512, partition_size_fp8=384),
    3: dict(name="70B-class GQA decode layer: S=256 64q/8kv D=128 f16 L~lognormal(med 300, sigma 1, cap 4096)",
            dtype="f16", num_seqs=256, num_q_heads=64, num_kv_heads=8, head_dim=128,
            lens=("lognormal", 300.0, 1.0, 4096), pool_factor=1.25, partition_size=768,
            partition_size_fp8=448),
    4: dict(name="long-context split-K decode: S=8 32q/8kv D=128 bf16 L~U[32768,131072] partition 512",
            dtype="bf16", num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
            lens=("uniform", 32768, 131072), pool_factor=1.25, partition_size=512),
    5: dict(name="prefix sharing + copy-on-write: S=128 32q/4kv D=128 f16 2048 shared + U[0,512] private",
            dtype="f16", num_seqs=128, num_q_heads=32, num_kv_heads=4, head_dim=128,
            lens=("prefix", 2048, 0, 512), pool_factor=1.25, partition_size=768),
}


def fp8_partition_size(cfg: int) -> int:
    """The split-K partition of recipe `cfg` over FP8 pools."""
    spec = CONFIGS[cfg]
    return int(spec.get("partition_size_fp8", spec.get("partition_size", 0)))


def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to f16 or bf16 (round-to-nearest-even) and return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        if np.any((u & 0x7F800000) == 0x7F800000):
            raise ValueError("bf16 rounding helper takes finite values only")
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        return r.astype(np.uint16)
    raise ValueError(dtype)


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    """Widen f16/bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(dtype)


class BlockPool:
    """Host-side block pool: per-block reference counts in an int32 array and
    the unreferenced blocks on a stack (an int32 array and its fill level).

    The stack starts as a random permutation of the pool, so consecutive
    takes land on scattered physical blocks.  take() returns -1 when no block
    is left; callers turn that into their own error.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = num_blocks
        self.counts = np.zeros(num_blocks, dtype=np.int32)
        self._stack = rng.permutation(num_blocks).astype(np.int32)
        self._depth = num_blocks

    def take(self) -> int:
        """A block with one reference, or -1 when the pool is empty."""
        if self._depth == 0:
            return -1
        self._depth -= 1
        b = int(self._stack[self._depth])
        self.counts[b] = 1
        return b

    def ref(self, b: int) -> int:
        """One more reference to a held block; returns b."""
        assert self.counts[b] > 0, f"block {b} is not held"
        self.counts[b] += 1
        return b

    def unref(self, b: int) -> None:
        """Drops one reference; the block goes back on the stack at zero."""
        assert self.counts[b] > 0, f"block {b} is not held"
        self.counts[b] -= 1
        if self.counts[b] == 0:
            self._stack[self._depth] = b
            self._depth += 1

    def held(self) -> dict:
        """{block: references} of every held block."""
        idx = np.flatnonzero(self.counts)
        return {int(b): int(self.counts[b]) for b in idx}


def _take(pool: BlockPool) -> int:
    b = pool.take()
    if b < 0:
        raise RuntimeError(f"workload recipe needs more than the {pool.num_blocks} blocks of its pool")
    return b


@dataclass
class SeqState:
    table: list = field(default_factory=list)
    length: int = 0


def append_token(pool: BlockPool, seq: SeqState, block_size: int = BLOCK_SIZE):
    """Reserve the slot of one new token.

    A new block is taken when the last one has no free row; a last block
    held more than once is first swapped for a private copy, and its
    (source, destination) pair is returned.  Returns (slot, cow_pair_or_None).
    """
    pair = None
    if seq.length % block_size == 0:
        seq.table.append(_take(pool))
    else:
        tail = seq.table[-1]
        if pool.counts[tail] > 1:
            fresh = _take(pool)
            pair = (tail, fresh)
            pool.unref(tail)
            seq.table[-1] = fresh
    slot = seq.table[seq.length // block_size] * block_size + seq.length % block_size
    seq.length += 1
    return slot, pair


@dataclass
class Workload:
    cfg: int
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    partition_size: int
    context_lens: np.ndarray
    block_tables: np.ndarray
    slot_mapping: np.ndarray
    copy_pairs: np.ndarray
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    refcount: dict
    protected_blocks: np.ndarray  # blocks that must stay bit-unchanged by the step
    poisoned: bool
    live: np.ndarray  # bool [num_blocks, block_size]: slots holding a token cached before the step

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes_read(self) -> int:
        """K+V bytes a decode pass over this batch must read (16-bit elements)."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 2 * 2


def _draw_lens(spec, n, rng):
    kind = spec[0]
    if kind == "fixed":
        out = np.asarray(spec[1], dtype=np.int64)
        assert out.size == n
        return out
    if kind == "uniform":
        return rng.integers(spec[1], spec[2], size=n, endpoint=True)
    if kind == "lognormal":
        med, sigma, cap = spec[1], spec[2], spec[3]
        x = np.rint(np.exp(rng.normal(math.log(med), sigma, size=n)))
        return np.clip(x, 1, cap).astype(np.int64)
    raise ValueError(kind)


_TORCH_DTYPE = {}


def _fill_normal(shape, dtype, gen, chunk_rows=4096):
    """N(0,1) float32 draws (torch's seeded CPU generator) rounded to the 16-bit dtype."""
    import torch

    if not _TORCH_DTYPE:
        _TORCH_DTYPE.update(f16=torch.float16, bf16=torch.bfloat16)
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        vals = torch.randn((r1 - r0, flat.shape[1]), generator=gen, dtype=torch.float32)
        # torch's float32 -> f16/bf16 casts round to nearest even, as f32_to_bits does
        flat[r0:r1] = vals.to(_TORCH_DTYPE[dtype]).view(torch.int16).numpy().view(np.uint16)
    return out


def make_workload(cfg: int, *, poison: bool = False, seed: int | None = None, **overrides) -> Workload:
    """Build the seeded workload of recipe `cfg` (1..5).

    Seed defaults to the recipe number.  `overrides` may change num_seqs,
    lens, head counts, head_dim, dtype, num_blocks, pool_factor,
    partition_size or block_size (used by tests for small variants of a
    recipe; the recipes use 16-token blocks).
    With poison=True every pool slot that holds no live token (unused blocks,
    tail slots past a sequence's length, the slot the new token goes to) is
    filled with NaN.
    """
    spec = dict(CONFIGS[cfg])
    spec.update(overrides)
    rng = np.random.default_rng(cfg if seed is None else seed)
    B = int(spec.get("block_size", BLOCK_SIZE))
    S = spec["num_seqs"]
    Hq, Hkv, D = spec["num_q_heads"], spec["num_kv_heads"], spec["head_dim"]
    dtype = spec["dtype"]
    assert Hq % Hkv == 0

    lens_spec = spec["lens"]
    if lens_spec[0] == "prefix":
        prefix_len, lo, hi = lens_spec[1], lens_spec[2], lens_spec[3]
        suffix = rng.integers(lo, hi, size=S, endpoint=True)
        lens = prefix_len + suffix + 1
        # blocks: shared prefix + per-sequence private blocks + one fresh block per append/CoW
        needed = math.ceil(prefix_len / B) + int(sum(math.ceil(s / B) + 1 for s in suffix))
    else:
        prefix_len, suffix = 0, None
        lens = _draw_lens(lens_spec, S, rng)
        needed = int(sum(math.ceil(int(L) / B) for L in lens))
    lens = lens.astype(np.int64)
    if "num_blocks" in spec:
        NB = int(spec["num_blocks"])
    else:
        NB = int(math.ceil(spec.get("pool_factor", 1.25) * needed))
    assert NB >= needed, (NB, needed)

    bm = BlockPool(NB, rng)
    seqs = [SeqState() for _ in range(S)]
    slots, pairs = [], []
    protected = set()
    if prefix_len:
        assert prefix_len % B == 0, "shared prefix is whole blocks"
        prefix_blocks = [_take(bm) for _ in range(prefix_len // B)]
        protected.update(prefix_blocks)
        for i, sq in enumerate(seqs):
            sq.table = [bm.ref(b) if i else b for b in prefix_blocks]
            sq.length = prefix_len
            for _ in range(math.ceil(int(suffix[i]) / B)):
                sq.table.append(_take(bm))
            sq.length += int(suffix[i])
            if sq.length % B:
                # the partial tail block also belongs to a forked parent
                bm.ref(sq.table[-1])
                protected.add(sq.table[-1])
    else:
        for sq, L in zip(seqs, lens):
            hist = int(L) - 1
            for _ in range(math.ceil(hist / B)):
                sq.table.append(_take(bm))
            sq.length = hist
    # Slots holding a token cached before this step (history), from the
    # tables as they stand before the append (a CoW source is still live).
    live = np.zeros((NB, B), dtype=bool)
    for sq in seqs:
        full, rem = divmod(sq.length, B)
        live[sq.table[:full], :] = True
        if rem:
            live[sq.table[full], :rem] = True

    for sq in seqs:
        slot, pair = append_token(bm, sq, B)
        slots.append(slot)
        if pair is not None:
            pairs.append(pair)
    for sq, L in zip(seqs, lens):
        assert sq.length == int(L)

    max_blocks = max(1, max(math.ceil(int(L) / B) for L in lens))
    tables = np.full((S, max_blocks), -1, dtype=np.int32)
    for i, sq in enumerate(seqs):
        tables[i, : len(sq.table)] = sq.table

    import torch

    gen = torch.Generator().manual_seed(int(rng.integers(0, 2**62)))
    k_pool = _fill_normal((NB, B, Hkv, D), dtype, gen)
    v_pool = _fill_normal((NB, B, Hkv, D), dtype, gen)
    q = _fill_normal((S, Hq, D), dtype, gen)
    k_new = _fill_normal((S, Hkv, D), dtype, gen)
    v_new = _fill_normal((S, Hkv, D), dtype, gen)

    if poison:
        nan = NAN_BITS[dtype]
        k_pool[~live] = nan
        v_pool[~live] = nan

    scale = 1.0 / math.sqrt(D)
    return Workload(
        cfg=cfg, name=spec["name"], dtype=dtype, num_seqs=S, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, block_size=B, num_blocks=NB, scale=scale,
        partition_size=int(spec.get("partition_size", 0)),
        context_lens=lens.astype(np.int32), block_tables=tables,
        slot_mapping=np.asarray(slots, dtype=np.int32).reshape(-1),
        copy_pairs=np.asarray(pairs, dtype=np.int32).reshape(-1, 2),
        q=q, k_new=k_new, v_new=v_new, k_pool=k_pool, v_pool=v_pool,
        refcount=bm.held(), protected_blocks=np.asarray(sorted(protected), dtype=np.int32),
        poisoned=poison, live=live,
    )


# ------------------------------------------------------------------ FP8 pools
#
# FP8 (e4m3) pools for the quantised-cache variant: one byte per element in the
# same [num_blocks, block_size, H_kv, D] layout, plus one float32 scale per
# (block, KV head) for K and for V.  Codes are drawn directly (this module
# encodes nothing): sign uniform, magnitude code uniform over
# [FP8_MIN_MAG_CODE, 0x7E] (0.25 .. 448, log-uniform in value), so no draw is
# 0x7F/0xFF, the format's NaN.  Scales are 2^u with u ~ U[-7.5, -6.5] (so a
# block's largest magnitude 448 * scale lies in 2.5 .. 5, like a per-block
# absmax scale over N(0,1) data), or, with exact=True, integer powers of two
# (-8..-6) so that every dequantised value is exact in 16 bits.

FP8_NAN = 0x7F
FP8_MIN_MAG_CODE = 0x28


@dataclass
class Fp8Pools:
    k8: np.ndarray       # uint8 [NB, B, H_kv, D]
    v8: np.ndarray
    k_scale: np.ndarray  # float32 [NB, H_kv]
    v_scale: np.ndarray

    def kv_bytes_read(self, wl: "Workload") -> int:
        """Bytes a decode pass over `wl` reads from these pools: one byte per
        element plus the K and V scale of each (table entry, KV head)."""
        toks = int(wl.context_lens.astype(np.int64).sum())
        blocks = int(((wl.context_lens.astype(np.int64) + wl.block_size - 1) // wl.block_size).sum())
        return toks * wl.num_kv_heads * wl.head_dim * 2 + blocks * wl.num_kv_heads * 4 * 2


def draw_fp8_codes(shape, rng):
    """e4m3 codes: random sign, magnitude code uniform over [FP8_MIN_MAG_CODE, 0x7E]."""
    mag = rng.integers(FP8_MIN_MAG_CODE, 0x7E, size=shape, endpoint=True, dtype=np.uint8)
    mag |= rng.integers(0, 2, size=shape, dtype=np.uint8) << np.uint8(7)
    return mag


def make_fp8_pools(wl: Workload, *, seed: int | None = None, exact: bool = False,
                   poison: bool | None = None) -> Fp8Pools:
    """Seeded FP8 pools for workload `wl` (its tables, lengths, slot mapping
    and copy pairs; its 16-bit pools are not used).  With poison (default:
    wl.poisoned) every slot holding no live token reads as NaN codes, and the
    scales of blocks that neither a table (after the step) nor a copy source
    references, and of copy-on-write destinations (overwritten by the step's
    copy before any read), are NaN."""
    rng = np.random.default_rng((wl.cfg * 7919 + 17) if seed is None else seed)
    shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    k8 = draw_fp8_codes(shape, rng)
    v8 = draw_fp8_codes(shape, rng)
    sshape = (wl.num_blocks, wl.num_kv_heads)
    if exact:
        ks = np.ldexp(1.0, rng.integers(-8, -6, size=sshape, endpoint=True)).astype(np.float32)
        vs = np.ldexp(1.0, rng.integers(-8, -6, size=sshape, endpoint=True)).astype(np.float32)
    else:
        ks = np.exp2(rng.uniform(-7.5, -6.5, size=sshape)).astype(np.float32)
        vs = np.exp2(rng.uniform(-7.5, -6.5, size=sshape)).astype(np.float32)
    if wl.poisoned if poison is None else poison:
        k8[~wl.live] = FP8_NAN
        v8[~wl.live] = FP8_NAN
        used = np.zeros(wl.num_blocks, dtype=bool)
        t = wl.block_tables
        used[t[t >= 0]] = True
        if wl.copy_pairs.size:
            used[wl.copy_pairs[:, 0]] = True
        dead = ~used
        if wl.copy_pairs.size:
            dead[wl.copy_pairs[:, 1]] = True
        ks[dead] = np.nan
        vs[dead] = np.nan
    return Fp8Pools(k8=k8, v8=v8, k_scale=ks, v_scale=vs)


# ------------------------------------------------------------------ all-layer pools
#
# A model's layers share the block tables, lengths, slot mapping and
# copy-on-write pairs of a step; each layer has its own queries, new rows and
# pool contents.  "KV Cache & PagedAttention" section 4 keeps every layer of
# a block together: [2 (K, V)][num_blocks][num_layers][block_size][H_kv][D].


@dataclass
class LayerData:
    q: np.ndarray      # uint16 [L, S, H_q, D]
    k_new: np.ndarray  # uint16 [L, S, H_kv, D]
    v_new: np.ndarray
    pool: np.ndarray   # uint16 [2, NB, L, B, H_kv, D]


def make_layers(wl: Workload, num_layers: int, *, seed: int | None = None) -> LayerData:
    """Per-layer values for workload `wl` (its tables and bookkeeping are
    shared): layer 0 is wl's own arrays, the others are seeded N(0,1) draws
    rounded to wl.dtype, poisoned like wl (NaN in every slot no sequence
    owns)."""
    import torch

    gen = torch.Generator().manual_seed(wl.cfg * 1000003 + 11 if seed is None else seed)
    L, S, NB, B = num_layers, wl.num_seqs, wl.num_blocks, wl.block_size
    Hq, Hkv, D = wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    q = np.empty((L, S, Hq, D), dtype=np.uint16)
    k_new = np.empty((L, S, Hkv, D), dtype=np.uint16)
    v_new = np.empty_like(k_new)
    pool = np.empty((2, NB, L, B, Hkv, D), dtype=np.uint16)
    for layer in range(L):
        if layer == 0:
            q[0], k_new[0], v_new[0] = wl.q, wl.k_new, wl.v_new
            pool[0, :, 0], pool[1, :, 0] = wl.k_pool, wl.v_pool
            continue
        q[layer] = _fill_normal((S, Hq, D), wl.dtype, gen)
        k_new[layer] = _fill_normal((S, Hkv, D), wl.dtype, gen)
        v_new[layer] = _fill_normal((S, Hkv, D), wl.dtype, gen)
        for kv in range(2):
            blk = _fill_normal((NB, B, Hkv, D), wl.dtype, gen)
            if wl.poisoned:
                blk[~wl.live] = NAN_BITS[wl.dtype]
            pool[kv, :, layer] = blk
    return LayerData(q=q, k_new=k_new, v_new=v_new, pool=pool)
