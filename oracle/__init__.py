"""Oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct CPU statements of what the hot path computes.
Only the tests, the smoke check and the benchmark's CPU-baseline / reference
legs may import this package.  It shares no code with the CUDA library and
never imports it.

Contents
  write_cache      -- the slot-mapping scatter, a byte copy per token.
  copy_blocks      -- the copy-on-write block copy, a byte copy per pair.
  decode_attention -- fp64 single-query grouped attention through block
                      tables (C++ in csrc/pkv_oracle.cpp, threaded over rows).
  brute            -- a pure-Python restatement used to pin the C++ one.
  sizing           -- the pages' closed forms for KV bytes, blocks and waste.

Sources (four web pages on paged KV caches):
  * "gpu_paged_kv_cache" (aicassindra), section "The write path: slot mapping
    and scatter": each new token's K and V go to linear slot
    block_index * B + offset of the pool.
  * same page, "Prefix sharing, reference counts, and copy-on-write", and
    "PagedAttention internals" (manishklach) section 03: copy-on-write copies
    the whole source block into a fresh block, device to device.
  * "PagedAttention internals" section 02 and "tm_paged_attention" (aicassindra)
    "The architecture" / "End-to-end flow": the table translation and the
    decode step attending over the full history.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["write_cache", "copy_blocks", "decode_attention", "hardware_threads"]

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


if os.environ.get("PKV_ORACLE_EAGER_BUILD"):
    _lib()
