"""Oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU statements of what the hot path computes.
Only the tests, the smoke check and the benchmark's CPU-baseline / reference
legs may import this package.  It shares no code with the CUDA library and
never imports it.

Contents
  write_cache      -- the slot-mapping scatter, a byte copy per token.
  copy_blocks      -- the copy-on-write block copy, a byte copy per pair.
  swap_blocks      -- block lists moved between two pools (device and host;
                      swap out / in), a byte copy per pair.
  decode_attention -- fp64 single-query grouped attention through block
                      tables (C++ in csrc/pkv_oracle.cpp, threaded over rows).
  brute            -- a pure-Python restatement used to pin the C++ one.
  sizing           -- the pages' closed forms for KV bytes, blocks and waste.
  e4m3_decode, e4m3_encode, write_cache_fp8, copy_blocks_fp8,
  decode_attention_fp8, apply_step_fp8
                   -- the same path over FP8 (e4m3) pools with one scale per
                      (physical block, KV head) for K and for V.

Sources (four web pages on paged KV caches):
  * "gpu_paged_kv_cache" (aicassindra), section "The write path: slot mapping
    and scatter": each new token's K and V go to linear slot
    block_index * B + offset of the pool.
  * same page, "Prefix sharing, reference counts, and copy-on-write", and
    "PagedAttention internals" (manishklach) section 03: copy-on-write copies
    the whole source block into a fresh block, device to device.
  * "PagedAttention internals" section 02 and "tm_paged_attention" (aicassindra)
    "The architecture" / "End-to-end flow": the table translation and the
    decode step attending over the full history (any block size: the block
    is the pools' second axis).
  * "gpu_paged_kv_cache", "Reclaiming memory: swap versus recompute", and
    "PagedAttention internals" section 05: a preempted sequence's blocks go
    to pinned host memory and come back to whatever blocks are free.
  * "PagedAttention internals" section 06, "Blocks as quantization groups":
    the 16-token block as the quantization group, its scales riding with the
    block, including across copy-on-write; and "KV Cache & PagedAttention"
    (lattice-ai-eng) sections 5 ("Quality") and 7: K, V stored in FP8 on
    Hopper/Blackwell.  Readings: one float scale per
    (block, KV head) for K and for V; a value is decode(code) * scale; the
    write path quantizes a new row with its block's scale as
    e4m3(float32(x) / float32(scale)), rounding to nearest-even and
    saturating to +-448 (the format has no infinities).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["write_cache", "copy_blocks", "swap_blocks", "decode_attention", "hardware_threads", "e4m3_decode",
           "e4m3_encode", "write_cache_fp8", "copy_blocks_fp8", "decode_attention_fp8", "apply_step_fp8"]

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        f = lib.pkv_oracle_decode_attention
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 6 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        f8 = lib.pkv_oracle_decode_attention_fp8
        f8.restype = ctypes.c_int
        f8.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 6 + [
            ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        lib.pkv_oracle_hardware_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def hardware_threads() -> int:
    return int(_lib().pkv_oracle_hardware_threads())


def write_cache(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                slot_mapping: np.ndarray) -> None:
    """In place: for each token i with slot >= 0, pool[slot // B][slot % B] = new[i] (K and V).

    Pools are [num_blocks, B, H_kv, D]; new rows are [T, H_kv, D].  A slot of
    -1 means "no write" (a padding token).  Pure byte copy.
    """
    B = k_pool.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        k_pool[slot // B, slot % B] = k_new[i]
        v_pool[slot // B, slot % B] = v_new[i]


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs: np.ndarray) -> None:
    """In place: for each (src, dst) pair, block dst := block src (K and V), byte for byte."""
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]


def swap_blocks(dst_k: np.ndarray, dst_v: np.ndarray, src_k: np.ndarray, src_v: np.ndarray,
                pairs: np.ndarray) -> None:
    """In place: for each (s, d) pair, dst block d := src block s (K and V), byte for byte.

    Swap out: src = the device pool, dst = a host pool ("gpu_paged_kv_cache",
    "Reclaiming memory: swap versus recompute": the victim's blocks are copied
    to pinned host memory and freed); swap in: the reverse, to whatever free
    device blocks the block manager picks ("PagedAttention internals" section
    05: copied back on resume).  Blocks are the arrays' first axis."""
    for s_idx, d_idx in np.asarray(pairs).reshape(-1, 2).tolist():
        dst_k[d_idx] = src_k[s_idx]
        dst_v[d_idx] = src_v[s_idx]


def decode_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_tables: np.ndarray,
                     context_lens: np.ndarray, scale: float, dtype: str, rows=None,
                     num_threads: int = 0) -> np.ndarray:
    """fp64 paged decode attention.

    q [S, H_q, D] and pools [NB, B, H_kv, D] hold f16 or bf16 bit patterns
    (uint16); dtype is "f16" or "bf16".  Returns float64 [S, H_q, D], or
    [n, D] for an explicit list of (s, h) rows.
    """
    lib = _lib()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
    v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, D = q.shape
    NB, B, Hkv, D2 = k_pool.shape
    assert D2 == D and v_pool.shape == k_pool.shape and bt.shape[0] == S and cl.shape == (S,)
    if rows is None:
        out = np.zeros((S, Hq, D), dtype=np.float64)
        rows_arr, n = None, S * Hq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n = rows_arr.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
    if n == 0:
        return out
    rc = lib.pkv_oracle_decode_attention(
        out.ctypes.data, q.ctypes.data, k_pool.ctypes.data, v_pool.ctypes.data, bt.ctypes.data,
        bt.shape[1], cl.ctypes.data, S, Hq, Hkv, D, B, NB, float(scale), 1 if dtype == "bf16" else 0,
        None if rows_arr is None else rows_arr.ctypes.data, n, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the input (code {rc}): table entry or length out of range")
    return out


def apply_step(wl, *, attention: bool = True, rows=None):
    """Runs one decode step of a pkv_inputs.Workload on copies of its pools:
    copy_blocks (copy-on-write), then write_cache, then (optionally) attention.
    Returns (k_pool, v_pool, out_or_None)."""
    k = wl.k_pool.copy()
    v = wl.v_pool.copy()
    copy_blocks(k, v, wl.copy_pairs)
    write_cache(k, v, wl.k_new, wl.v_new, wl.slot_mapping)
    out = None
    if attention:
        out = decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows)
    return k, v, out


# ------------------------------------------------------------------ FP8 pools


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes (uint8) -> float64, from the format's definition: sign bit,
    4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
    (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN; no infinities."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    v = np.where(e == 0, np.ldexp(m.astype(np.float64), -9), np.ldexp((8 + m).astype(np.float64), e - 10))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return sign * v


_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # codes 0x00..0x7E: 0 .. 448, ascending


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> e4m3 codes: round to the nearest representable value,
    ties to the even code (even mantissa), magnitudes above 448 saturate to
    448, NaN -> 0x7F (with the sign bit).  Nearest-value search over the
    format's finite values."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo, d_hi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick = np.where(d_hi < d_lo, hi, np.where(d_lo < d_hi, lo, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(np.isnan(x), 0x7F, pick) | sign
    return code.astype(np.uint8)


def _widen16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float32 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def write_cache_fp8(k8: np.ndarray, v8: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray, k_new: np.ndarray,
                    v_new: np.ndarray, slot_mapping: np.ndarray, dtype: str) -> None:
    """In place: for each token i with slot >= 0 (block b = slot // B, offset
    o = slot % B) and KV head g, pool[b][o][g] = e4m3(float32(new[i][g]) /
    scale[b][g]) for K and V.  new rows hold `dtype` (f16/bf16) patterns."""
    B = k8.shape[1]
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, o = divmod(slot, B)
        for pool, scales, new in ((k8, k_scale, k_new), (v8, v_scale, v_new)):
            x = _widen16(new[i], dtype)  # [H_kv, D]
            pool[b, o] = e4m3_encode(x / scales[b].astype(np.float32)[:, None])


def copy_blocks_fp8(k8: np.ndarray, v8: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray,
                    pairs: np.ndarray) -> None:
    """In place: for each (src, dst) pair, block dst := block src, codes and scales (K and V)."""
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k8[dst] = k8[src]
        v8[dst] = v8[src]
        k_scale[dst] = k_scale[src]
        v_scale[dst] = v_scale[src]


def decode_attention_fp8(q: np.ndarray, k8: np.ndarray, v8: np.ndarray, k_scale: np.ndarray, v_scale: np.ndarray,
                         block_tables: np.ndarray, context_lens: np.ndarray, scale: float, dtype: str, rows=None,
                         num_threads: int = 0) -> np.ndarray:
    """fp64 paged decode attention over FP8 pools: K = e4m3_decode(k8) *
    k_scale[block][g] (V likewise); q holds `dtype` patterns.  Returns as
    decode_attention does."""
    lib = _lib()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8)
    v8 = np.ascontiguousarray(v8, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, D = q.shape
    NB, B, Hkv, D2 = k8.shape
    assert D2 == D and v8.shape == k8.shape and ks.shape == (NB, Hkv) and vs.shape == (NB, Hkv)
    if rows is None:
        out = np.zeros((S, Hq, D), dtype=np.float64)
        rows_arr, n = None, S * Hq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n = rows_arr.shape[0]
        out = np.zeros((n, D), dtype=np.float64)
    if n == 0:
        return out
    rc = lib.pkv_oracle_decode_attention_fp8(
        out.ctypes.data, q.ctypes.data, k8.ctypes.data, v8.ctypes.data, ks.ctypes.data, vs.ctypes.data,
        bt.ctypes.data, bt.shape[1], cl.ctypes.data, S, Hq, Hkv, D, B, NB, float(scale), 1 if dtype == "bf16" else 0,
        None if rows_arr is None else rows_arr.ctypes.data, n, int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle rejected the input (code {rc}): table entry or length out of range")
    return out


def apply_step_fp8(wl, pools, *, attention: bool = True, rows=None):
    """One decode step of a workload over its FP8 pools (pkv_inputs.Fp8Pools),
    on copies: copy_blocks_fp8, write_cache_fp8, then (optionally) attention.
    Returns (k8, v8, k_scale, v_scale, out_or_None)."""
    k8, v8 = pools.k8.copy(), pools.v8.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    copy_blocks_fp8(k8, v8, ks, vs, wl.copy_pairs)
    write_cache_fp8(k8, v8, ks, vs, wl.k_new, wl.v_new, wl.slot_mapping, wl.dtype)
    out = None
    if attention:
        out = decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                   rows=rows)
    return k8, v8, ks, vs, out


if os.environ.get("PKV_ORACLE_EAGER_BUILD"):
    _lib()
