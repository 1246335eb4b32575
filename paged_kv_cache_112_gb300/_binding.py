"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function takes torch tensors that already live on the GPU, checks
their dtype, shape, strides and that they are CUDA tensors, and forwards raw
pointers, sizes and the current CUDA stream to the C ABI.  The library
launches on the current CUDA device, so the tensors must live there (one
process per GPU; the device index is not checked per tensor).  All
computation happens in the library's kernels; there is no fallback path,
and the library must be built (see build.py) or calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA, PKV_ERR_OUT_OF_BLOCKS = range(6)
PKV_F32, PKV_F16, PKV_BF16 = 0, 1, 2
PARTITION_BALANCED = -1  # partition_size selecting the library's balanced split
DEV_ERR_SLOT, DEV_ERR_PAIR, DEV_ERR_BLOCK, DEV_ERR_LENGTH, DEV_ERR_TIMEOUT, DEV_ERR_SMEM = 1, 2, 4, 8, 16, 32

_DTYPES = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
_KV_DTYPES = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}

_c_void_p, _c_int, _c_int64, _c_size_t, _c_float = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                                    ctypes.c_size_t, ctypes.c_float)
_SIGS = {
    "pkv_write_cache": [_c_void_p] * 4 + [_c_int64, _c_void_p, _c_int, _c_int64] + [_c_int] * 5 + [_c_void_p] * 2,
    "pkv_copy_blocks": [_c_void_p] * 3 + [_c_int] * 7 + [_c_void_p, _c_void_p],
    "pkv_decode_workspace_bytes": [_c_int] * 5,
    "pkv_decode_attention": [_c_void_p] * 4 + [_c_int64, _c_void_p, _c_int, _c_void_p] + [_c_int] * 6 + [
        _c_float, _c_int, _c_int, _c_void_p, _c_size_t, _c_int, _c_int, _c_void_p, _c_void_p],
    "pkv_decode_reduce": [_c_void_p, _c_void_p] + [_c_int] * 6 + [_c_void_p, _c_size_t, _c_int, _c_void_p,
                                                                  _c_void_p],
    "pkv_status_string": [_c_int],
    "pkv_version": [],
}
_SIGS["pkv_decode_partitions"] = _SIGS["pkv_decode_attention"]
_SIGS["pkv_decode_step"] = ([_c_void_p] * 4 + [_c_int64] + [_c_void_p] * 2 + [_c_int64, _c_void_p, _c_int] +
                            [_c_void_p] * 2 + [_c_int] * 6 + [_c_float, _c_int, _c_int, _c_void_p, _c_size_t, _c_int,
                                                              _c_int, _c_void_p, _c_void_p])
_SIGS["pkv_decode_step_partitions"] = _SIGS["pkv_decode_step"]
_SIGS["pkv_write_cache_fp8"] = [_c_void_p] * 7 + [_c_int, _c_int64] + [_c_int] * 6 + [_c_void_p, _c_void_p]
_SIGS["pkv_copy_blocks_fp8"] = [_c_void_p] * 5 + [_c_int] * 6 + [_c_void_p, _c_void_p]
_SIGS["pkv_decode_attention_fp8"] = ([_c_void_p] * 7 + [_c_int, _c_void_p] + [_c_int] * 7 +
                                     [_c_float, _c_int, _c_int, _c_void_p, _c_size_t, _c_int, _c_int, _c_void_p,
                                      _c_void_p])
_SIGS["pkv_decode_partitions_fp8"] = _SIGS["pkv_decode_attention_fp8"]
_SIGS["pkv_swap_blocks"] = ([_c_void_p] * 2 + [_c_int64, _c_int] + [_c_void_p] * 2 + [_c_int64, _c_int, _c_int64,
                                                                                     _c_void_p, _c_int, _c_void_p,
                                                                                     _c_void_p])
_SIGS["pkv_decode_step_fp8"] = ([_c_void_p] * 4 + [_c_int64] + [_c_void_p] * 5 + [_c_int] + [_c_void_p] * 2 +
                                [_c_int] * 7 + [_c_float, _c_int, _c_int, _c_void_p, _c_size_t, _c_int, _c_int,
                                                _c_void_p, _c_void_p])
_SIGS["pkv_decode_step_partitions_fp8"] = _SIGS["pkv_decode_step_fp8"]
_SIGS["pkv_check_bounded_wait"] = [_c_int64, _c_int, _c_void_p, _c_void_p]
_SIGS["pkv_last_cuda_error"] = []
_SIGS["pkv_cuda_error_name"] = [_c_int]

class _BmStats(ctypes.Structure):
    """pkv_bm_stats (include/pkv.h): int64 fields in declaration order."""
    _fields_ = [(name, ctypes.c_int64) for name in (
        "num_blocks", "block_size", "blocks_free", "blocks_cached_unreferenced", "blocks_referenced",
        "blocks_cached", "slots_holding_tokens", "sequences_resident", "sequences_swapped", "table_entries",
        "max_blocks_per_sequence", "prompt_tokens", "prompt_tokens_cached", "evictions", "cow_copies",
        "swap_outs", "refusals")]


_BM_SIGS = {
    "pkv_pool_blocks": ([ctypes.c_uint64] + [ctypes.c_int] * 6, ctypes.c_int64),
    "pkv_bm_create": ([ctypes.c_int] * 3, ctypes.c_void_p),
    "pkv_bm_destroy": ([ctypes.c_void_p], None),
    "pkv_bm_available_blocks": ([ctypes.c_void_p], ctypes.c_int),
    "pkv_bm_cached_blocks": ([ctypes.c_void_p], ctypes.c_int),
    "pkv_bm_block_refcount": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "pkv_bm_add_sequence": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                             ctypes.c_void_p], ctypes.c_int),
    "pkv_bm_fork": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64], ctypes.c_int),
    "pkv_bm_append": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32] + [ctypes.POINTER(ctypes.c_int32)] * 3,
                      ctypes.c_int),
    "pkv_bm_decode_step": ([ctypes.c_void_p] * 3 + [ctypes.c_int] + [ctypes.c_void_p] * 3 +
                           [ctypes.c_int, ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "pkv_bm_get_stats": ([ctypes.c_void_p, ctypes.POINTER(_BmStats)], ctypes.c_int),
    "pkv_bm_free_sequence": ([ctypes.c_void_p, ctypes.c_int64], ctypes.c_int),
    "pkv_bm_seq_len": ([ctypes.c_void_p, ctypes.c_int64], ctypes.c_int),
    "pkv_bm_block_table": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "pkv_bm_seq_tokens": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "pkv_bm_swap_out": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "pkv_bm_swap_in": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "pkv_bm_swap_in_cached": ([ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int],
                              ctypes.c_int),
}

_LIB = None


class PkvError(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Loads libpkv.so (building it first if asked).  Raises when it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB):
        raise PkvError(f"libpkv is not built ({_build.LIB} missing); run "
                       "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_build.LIB)
    for name, argtypes in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = ctypes.c_size_t if name == "pkv_decode_workspace_bytes" else (
            ctypes.c_char_p if name in ("pkv_status_string", "pkv_cuda_error_name") else ctypes.c_int)
    for name, (argtypes, restype) in _BM_SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = restype
    _LIB = lib
    return lib


def status_string(code: int) -> str:
    return load().pkv_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != PKV_OK:
        detail = ""
        if code == PKV_ERR_CUDA:
            lib = load()
            err = int(lib.pkv_last_cuda_error())
            detail = f" ({lib.pkv_cuda_error_name(err).decode()}, code {err})"
        raise PkvError(f"{what}: {status_string(code)}{detail}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t):
    return None if t is None else int(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise PkvError("tensors must be contiguous CUDA tensors")


def _pool_stride(k_pool, v_pool) -> int:
    """Block stride (elements) of a pool given as [NB, 16, H_kv, D] with dense
    blocks: a per-layer tensor, or one layer's view of an all-layer pool
    (e.g. pool[0, :, layer] of a [2, NB, layers, 16, H_kv, D] tensor)."""
    for t in (k_pool, v_pool):
        if not t.is_cuda or t.dim() != 4:
            raise PkvError("pools must be CUDA tensors [NB, 16, H_kv, D]")
        NB, B, Hkv, D = t.shape
        if t.stride(3) != 1 or t.stride(2) != D or t.stride(1) != Hkv * D or t.stride(0) < B * Hkv * D:
            raise PkvError("pool blocks must be dense [16, H_kv, D] slices")
    if k_pool.stride(0) != v_pool.stride(0) or k_pool.shape != v_pool.shape:
        raise PkvError("k_pool and v_pool must share shape and block stride")
    return int(k_pool.stride(0))


def check_bounded_wait(timeout_ns: int, status, *, shared_ring=False, stream=None):
    """pkv_check_bounded_wait: a wait on a tile barrier nothing completes runs
    out after timeout_ns and ORs DEV_ERR_TIMEOUT into `status` (a CUDA int32
    tensor); shared_ring: in a CTA whose warps share stages and leave by a
    CTA-wide vote."""
    _need_cuda(status)
    if status is None or status.dtype != torch.int32:
        raise PkvError("status must be a CUDA int32 tensor")
    _check(load().pkv_check_bounded_wait(int(timeout_ns), int(bool(shared_ring)), _ptr(status), _stream(stream)),
           "pkv_check_bounded_wait")


def _kv_dtype(t) -> int:
    if t.dtype not in _KV_DTYPES:
        raise PkvError(f"KV dtype must be float16 or bfloat16, got {t.dtype}")
    return _KV_DTYPES[t.dtype]


def write_cache(k_new, v_new, k_pool, v_pool, slot_mapping, *, status=None, stream=None):
    """pkv_write_cache: k_new/v_new [T, H_kv, D] (rows may be strided), pools [NB, 16, H_kv, D]
    (per-layer tensors or layer views of an all-layer pool)."""
    bstride = _pool_stride(k_pool, v_pool)
    _need_cuda(slot_mapping, status)
    NB, B, Hkv, D = k_pool.shape
    T = k_new.shape[0]
    for t in (k_new, v_new):
        if not t.is_cuda or t.dim() != 3 or t.shape[1:] != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise PkvError("k_new/v_new must be CUDA [T, H_kv, D] with dense rows")
    if k_new.stride(0) != v_new.stride(0):
        raise PkvError("k_new and v_new must share a row stride")
    _check(load().pkv_write_cache(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), bstride, _ptr(slot_mapping),
                                  T, int(k_new.stride(0)), Hkv, D, B, NB, _kv_dtype(k_pool), _ptr(status),
                                  _stream(stream)), "pkv_write_cache")


def copy_blocks(k_pool, v_pool, pairs, *, status=None, stream=None):
    """pkv_copy_blocks: pairs int32 [P, 2] (src, dst).  Pools are contiguous per-layer
    [NB, 16, H_kv, D] tensors, or the K and V halves [NB, layers, 16, H_kv, D] of an
    all-layer pool, whose blocks are copied with every layer."""
    _need_cuda(k_pool, v_pool, pairs, status)
    if k_pool.shape != v_pool.shape or k_pool.dim() not in (4, 5):
        raise PkvError("pools must be [NB, 16, H_kv, D] or [NB, layers, 16, H_kv, D], K and V alike")
    layers = 1 if k_pool.dim() == 4 else int(k_pool.shape[1])
    NB, B, Hkv, D = k_pool.shape[0], k_pool.shape[-3], k_pool.shape[-2], k_pool.shape[-1]
    _check(load().pkv_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(pairs), int(pairs.shape[0]), layers, Hkv, D, B,
                                  NB, _kv_dtype(k_pool), _ptr(status), _stream(stream)), "pkv_copy_blocks")


def decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, partition_size) -> int:
    return int(load().pkv_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len, partition_size))


def _decode_args(out, q, k_pool, v_pool, block_tables, context_lens, scale, partition_size, max_context_len,
                 workspace, status, stream):
    bstride = _pool_stride(k_pool, v_pool)
    _need_cuda(out, q, block_tables, context_lens, workspace, status)
    S, Hq, D = q.shape
    NB, B, Hkv, D2 = k_pool.shape
    if D2 != D or v_pool.shape != k_pool.shape or q.dtype != k_pool.dtype or v_pool.dtype != k_pool.dtype:
        raise PkvError("q, k_pool, v_pool shapes/dtypes disagree")
    if out.shape != q.shape or out.dtype not in _DTYPES:
        raise PkvError("out must be [S, H_q, D] float32/float16/bfloat16")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError("block_tables and context_lens must be int32")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), bstride, _ptr(block_tables), int(block_tables.shape[1]),
            _ptr(context_lens), S, Hq, Hkv, D, B, NB, float(scale), int(partition_size), int(max_context_len),
            _ptr(workspace), ws_bytes, _kv_dtype(k_pool), _DTYPES[out.dtype], _ptr(status), _stream(stream))


def decode_attention(out, q, k_pool, v_pool, block_tables, context_lens, scale, *, partition_size=0,
                     max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_attention (partition kernel + reduce kernel)."""
    _check(load().pkv_decode_attention(*_decode_args(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                                                     partition_size, max_context_len, workspace, status, stream)),
           "pkv_decode_attention")


def decode_partitions(out, q, k_pool, v_pool, block_tables, context_lens, scale, *, partition_size=0,
                      max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_partitions: the first kernel of decode_attention alone."""
    _check(load().pkv_decode_partitions(*_decode_args(out, q, k_pool, v_pool, block_tables, context_lens, scale,
                                                      partition_size, max_context_len, workspace, status,
                                                      stream)), "pkv_decode_partitions")


def decode_reduce(out, context_lens, *, num_q_heads, num_kv_heads, head_dim, partition_size, max_context_len,
                  workspace=None, status=None, stream=None):
    """pkv_decode_reduce: the second kernel of decode_attention alone."""
    _need_cuda(out, context_lens, workspace, status)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().pkv_decode_reduce(_ptr(out), _ptr(context_lens), int(context_lens.shape[0]), num_q_heads,
                                    num_kv_heads, head_dim, int(partition_size), int(max_context_len),
                                    _ptr(workspace), ws_bytes, _DTYPES[out.dtype], _ptr(status), _stream(stream)),
           "pkv_decode_reduce")


def _step_args(out, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens, slot_mapping, scale,
               partition_size, max_context_len, workspace, status, stream):
    base = _decode_args(out, q, k_pool, v_pool, block_tables, context_lens, scale, partition_size,
                        max_context_len, workspace, status, stream)
    _need_cuda(slot_mapping)
    NB, B, Hkv, D = k_pool.shape
    for t in (k_new, v_new):
        if not t.is_cuda or t.dim() != 3 or t.shape != (q.shape[0], Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise PkvError("k_new/v_new must be CUDA [S, H_kv, D] with dense rows")
    if k_new.stride(0) != v_new.stride(0) or k_new.dtype != k_pool.dtype or v_new.dtype != k_pool.dtype:
        raise PkvError("k_new and v_new must share a row stride and the pools' dtype")
    if slot_mapping.dtype != torch.int32 or slot_mapping.shape != (q.shape[0],):
        raise PkvError("slot_mapping must be int32 [S]")
    (o, qp, kp, vp, bs, bt, maxb, cl, S, Hq, Hkv_, D_, B_, NB_, sc, ps, mcl, ws, wsb, kvd, od, st, strm) = base
    return (o, qp, _ptr(k_new), _ptr(v_new), int(k_new.stride(0)), kp, vp, bs, bt, maxb, cl, _ptr(slot_mapping), S,
            Hq, Hkv_, D_, B_, NB_, sc, ps, mcl, ws, wsb, kvd, od, st, strm)


def decode_step(out, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens, slot_mapping, scale, *,
                partition_size=0, max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_step: write of the new token fused into decode attention, then the reduce."""
    _check(load().pkv_decode_step(*_step_args(out, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens,
                                              slot_mapping, scale, partition_size, max_context_len, workspace,
                                              status, stream)), "pkv_decode_step")


def decode_step_partitions(out, q, k_new, v_new, k_pool, v_pool, block_tables, context_lens, slot_mapping, scale, *,
                           partition_size=0, max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_step_partitions: the first kernel of decode_step alone."""
    _check(load().pkv_decode_step_partitions(*_step_args(out, q, k_new, v_new, k_pool, v_pool, block_tables,
                                                         context_lens, slot_mapping, scale, partition_size,
                                                         max_context_len, workspace, status, stream)),
           "pkv_decode_step_partitions")


# ------------------------------------------------------------------ FP8 pools
# Pools are uint8 [NB, 16, H_kv, D] tensors of e4m3 codes; scales float32
# [NB, H_kv] (one per block and KV head, for K and for V).  Either per-layer
# tensors, or one layer's views of all-layer pools [NB, layers, 16, H_kv, D]
# and scales [NB, layers, H_kv] (pool[:, layer], scale[:, layer]).


def _fp8_pools(k_pool, v_pool, k_scale, v_scale):
    """(NB, 16, H_kv, D, layers) of FP8 pools given as per-layer tensors or
    layer views of all-layer pools; the layer count comes from the strides."""
    for t in (k_pool, v_pool, k_scale, v_scale):
        if not t.is_cuda or t.dim() not in (2, 4):
            raise PkvError("FP8 pools must be CUDA [NB, 16, H_kv, D] and scales CUDA [NB, H_kv]")
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8 or v_pool.shape != k_pool.shape or \
            k_pool.dim() != 4:
        raise PkvError("FP8 pools must be uint8 tensors of one shape [NB, 16, H_kv, D]")
    NB, B, Hkv, D = k_pool.shape
    block = B * Hkv * D
    for t in (k_pool, v_pool):
        if t.stride(3) != 1 or t.stride(2) != D or t.stride(1) != Hkv * D or t.stride(0) % block or \
                t.stride(0) < block:
            raise PkvError("FP8 pool blocks must be dense [16, H_kv, D] slices, layers x 16 rows apart")
    layers = int(k_pool.stride(0)) // block
    for sc in (k_scale, v_scale):
        if sc.dtype != torch.float32 or tuple(sc.shape) != (NB, Hkv) or sc.stride(1) != 1 or \
                sc.stride(0) != layers * Hkv:
            raise PkvError("scales must be float32 [NB, H_kv] with the pools' layer count")
    if v_pool.stride(0) != k_pool.stride(0):
        raise PkvError("k_pool and v_pool must share a block stride")
    return NB, B, Hkv, D, layers


def write_cache_fp8(k_new, v_new, k_pool, v_pool, k_scale, v_scale, slot_mapping, *, status=None, stream=None):
    """pkv_write_cache_fp8: k_new/v_new f16/bf16 [T, H_kv, D] quantised into the FP8 pools."""
    NB, B, Hkv, D, layers = _fp8_pools(k_pool, v_pool, k_scale, v_scale)
    _need_cuda(slot_mapping, status)
    T = k_new.shape[0]
    for t in (k_new, v_new):
        if not t.is_cuda or t.dim() != 3 or t.shape[1:] != (Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise PkvError("k_new/v_new must be CUDA [T, H_kv, D] with dense rows")
    if k_new.stride(0) != v_new.stride(0) or k_new.dtype != v_new.dtype:
        raise PkvError("k_new and v_new must share a row stride and a dtype")
    _check(load().pkv_write_cache_fp8(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(slot_mapping), T, int(k_new.stride(0)), Hkv, D, B, NB,
                                      layers, _kv_dtype(k_new), _ptr(status), _stream(stream)), "pkv_write_cache_fp8")


def copy_blocks_fp8(k_pool, v_pool, k_scale, v_scale, pairs, *, status=None, stream=None):
    """pkv_copy_blocks_fp8: pairs int32 [P, 2] (src, dst); codes and scales move together.  Pools
    and scales are contiguous per-layer tensors ([NB, 16, H_kv, D], [NB, H_kv]) or whole
    all-layer ones ([NB, layers, 16, H_kv, D], [NB, layers, H_kv]), copied with every layer."""
    _need_cuda(k_pool, v_pool, k_scale, v_scale, pairs, status)
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8 or v_pool.shape != k_pool.shape or \
            k_pool.dim() not in (4, 5):
        raise PkvError("FP8 pools must be uint8 [NB, 16, H_kv, D] or [NB, layers, 16, H_kv, D], K and V alike")
    layers = 1 if k_pool.dim() == 4 else int(k_pool.shape[1])
    NB, B, Hkv, D = k_pool.shape[0], k_pool.shape[-3], k_pool.shape[-2], k_pool.shape[-1]
    want = (NB, Hkv) if k_pool.dim() == 4 else (NB, layers, Hkv)
    for sc in (k_scale, v_scale):
        if sc.dtype != torch.float32 or tuple(sc.shape) != want:
            raise PkvError(f"scales must be float32 {list(want)}")
    _check(load().pkv_copy_blocks_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(pairs),
                                      int(pairs.shape[0]), layers, Hkv, D, B, NB, _ptr(status), _stream(stream)),
           "pkv_copy_blocks_fp8")


def _decode_fp8_args(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale, partition_size,
                     max_context_len, workspace, status, stream):
    NB, B, Hkv, D, layers = _fp8_pools(k_pool, v_pool, k_scale, v_scale)
    _need_cuda(out, q, block_tables, context_lens, workspace, status)
    S, Hq, Dq = q.shape
    if Dq != D or out.shape != q.shape or out.dtype not in _DTYPES:
        raise PkvError("q and out must be [S, H_q, D] with the pools' D")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise PkvError("block_tables and context_lens must be int32")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return (_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
            int(block_tables.shape[1]), _ptr(context_lens), S, Hq, Hkv, D, B, NB, layers, float(scale),
            int(partition_size),
            int(max_context_len), _ptr(workspace), ws_bytes, _kv_dtype(q), _DTYPES[out.dtype], _ptr(status),
            _stream(stream))


def decode_attention_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale, *,
                         partition_size=0, max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_attention_fp8 (partition kernel + reduce kernel); q f16/bf16 [S, H_q, D]."""
    _check(load().pkv_decode_attention_fp8(*_decode_fp8_args(out, q, k_pool, v_pool, k_scale, v_scale, block_tables,
                                                             context_lens, scale, partition_size, max_context_len,
                                                             workspace, status, stream)),
           "pkv_decode_attention_fp8")


def decode_partitions_fp8(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale, *,
                          partition_size=0, max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_partitions_fp8: the first kernel of decode_attention_fp8 alone (follow with decode_reduce)."""
    _check(load().pkv_decode_partitions_fp8(*_decode_fp8_args(out, q, k_pool, v_pool, k_scale, v_scale,
                                                              block_tables, context_lens, scale, partition_size,
                                                              max_context_len, workspace, status, stream)),
           "pkv_decode_partitions_fp8")


def _step_fp8_args(out, q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, slot_mapping,
                   scale, partition_size, max_context_len, workspace, status, stream):
    base = _decode_fp8_args(out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale,
                            partition_size, max_context_len, workspace, status, stream)
    _need_cuda(slot_mapping)
    NB, B, Hkv, D = k_pool.shape
    for t in (k_new, v_new):
        if not t.is_cuda or t.dim() != 3 or t.shape != (q.shape[0], Hkv, D) or t.stride(2) != 1 or t.stride(1) != D:
            raise PkvError("k_new/v_new must be CUDA [S, H_kv, D] with dense rows")
    if k_new.stride(0) != v_new.stride(0) or k_new.dtype != q.dtype or v_new.dtype != q.dtype:
        raise PkvError("k_new and v_new must share a row stride and the queries' dtype")
    if slot_mapping.dtype != torch.int32 or slot_mapping.shape != (q.shape[0],):
        raise PkvError("slot_mapping must be int32 [S]")
    (o, qp, kp, vp, ksp, vsp, bt, maxb, cl, S, Hq, Hkv_, D_, B_, NB_, L, sc, ps, mcl, ws, wsb, qd, od, st, strm) = base
    return (o, qp, _ptr(k_new), _ptr(v_new), int(k_new.stride(0)), kp, vp, ksp, vsp, bt, maxb, cl, _ptr(slot_mapping),
            S, Hq, Hkv_, D_, B_, NB_, L, sc, ps, mcl, ws, wsb, qd, od, st, strm)


def decode_step_fp8(out, q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, slot_mapping,
                    scale, *, partition_size=0, max_context_len, workspace=None, status=None, stream=None):
    """pkv_decode_step_fp8: the quantising write of the new token fused into FP8 decode attention, then the reduce."""
    _check(load().pkv_decode_step_fp8(*_step_fp8_args(out, q, k_new, v_new, k_pool, v_pool, k_scale, v_scale,
                                                      block_tables, context_lens, slot_mapping, scale, partition_size,
                                                      max_context_len, workspace, status, stream)),
           "pkv_decode_step_fp8")


def decode_step_partitions_fp8(out, q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens,
                               slot_mapping, scale, *, partition_size=0, max_context_len, workspace=None, status=None,
                               stream=None):
    """pkv_decode_step_partitions_fp8: the first kernel of decode_step_fp8 alone."""
    _check(load().pkv_decode_step_partitions_fp8(*_step_fp8_args(out, q, k_new, v_new, k_pool, v_pool, k_scale,
                                                                 v_scale, block_tables, context_lens, slot_mapping,
                                                                 scale, partition_size, max_context_len, workspace,
                                                                 status, stream)),
           "pkv_decode_step_partitions_fp8")


# ------------------------------------------------------------------ swap


def _block_layout(t):
    """(bytes between blocks, bytes per block) of a pool whose blocks are dense slices along dim 0."""
    esz = t.element_size()
    inner = 1
    expect = 1
    for d in range(t.dim() - 1, 0, -1):
        if t.stride(d) != expect:
            raise PkvError("pool blocks must be dense slices along the first axis")
        expect *= t.shape[d]
        inner *= t.shape[d]
    if t.stride(0) < inner:
        raise PkvError("pool blocks overlap")
    return int(t.stride(0)) * esz, inner * esz


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, *, status=None, stream=None):
    """pkv_swap_blocks: for each (s, d) in pairs, dst block d := src block s (K and V).

    Pools are tensors whose first axis is the block ([NB, 16, H_kv, D] per layer,
    [NB, layers, 16, H_kv, D] all layers, FP8 codes, or [NB, H_kv] scales), each on
    the GPU or in pinned host memory (tensor.pin_memory()); pairs int32 [P, 2]."""
    for t in (dst_k, dst_v, src_k, src_v, pairs):
        if not (t.is_cuda or t.is_pinned()):
            raise PkvError("swap operands must be CUDA tensors or pinned host tensors")
    if pairs.dtype != torch.int32 or not pairs.is_contiguous():
        raise PkvError("pairs must be a contiguous int32 [P, 2] tensor")
    d_stride, d_bytes = _block_layout(dst_k)
    s_stride, s_bytes = _block_layout(src_k)
    if _block_layout(dst_v) != (d_stride, d_bytes) or _block_layout(src_v) != (s_stride, s_bytes):
        raise PkvError("K and V pools must share their block layout")
    if d_bytes != s_bytes or dst_k.shape[0] != dst_v.shape[0] or src_k.shape[0] != src_v.shape[0]:
        raise PkvError("source and destination blocks must have the same size")
    _need_cuda(status)
    _check(load().pkv_swap_blocks(_ptr(dst_k), _ptr(dst_v), d_stride, int(dst_k.shape[0]), _ptr(src_k), _ptr(src_v),
                                  s_stride, int(src_k.shape[0]), d_bytes, _ptr(pairs), int(pairs.shape[0]),
                                  _ptr(status), _stream(stream)), "pkv_swap_blocks")


# ------------------------------------------------------------------ block manager


class OutOfBlocks(PkvError):
    """The block manager has not enough free blocks (nothing was changed)."""


def pool_blocks(kv_bytes: int, num_layers: int, block_size: int, num_kv_heads: int, head_dim: int,
                elem_bytes: int = 2, with_scales: bool = False) -> int:
    """pkv_pool_blocks: how many blocks fit kv_bytes (all layers of a block, K and V; FP8 scales optional)."""
    n = load().pkv_pool_blocks(int(kv_bytes), int(num_layers), int(block_size), int(num_kv_heads), int(head_dim),
                               int(elem_bytes), int(bool(with_scales)))
    if n < 0:
        raise PkvError("pool_blocks: sizes must be positive")
    return int(n)


class BlockManager:
    """The host block manager of libpkv (pkv_bm_*): free list, reference
    counts, chained-hash prefix cache with LRU eviction, copy-on-write,
    watermark and swap bookkeeping.  Produces block-table rows, slot
    mappings and copy-on-write pairs for the device entry points."""

    def __init__(self, num_blocks: int, block_size: int = 16, watermark_blocks: int = 0):
        import numpy as np

        self._np = np
        self._lib = load()
        self._h = self._lib.pkv_bm_create(int(num_blocks), int(block_size), int(watermark_blocks))
        if not self._h:
            raise PkvError("pkv_bm_create: invalid sizes")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _rc(self, rc: int, what: str) -> int:
        if rc >= 0:
            return rc
        if -rc == PKV_ERR_OUT_OF_BLOCKS:
            raise OutOfBlocks(what)
        raise PkvError(f"{what}: {status_string(-rc)}")

    @property
    def available_blocks(self) -> int:
        return self._lib.pkv_bm_available_blocks(self._h)

    @property
    def cached_blocks(self) -> int:
        return self._lib.pkv_bm_cached_blocks(self._h)

    def refcount(self, block: int) -> int:
        return self._rc(self._lib.pkv_bm_block_refcount(self._h, int(block)), "refcount")

    def add_sequence(self, seq_id: int, tokens, extra_key: int = 0):
        """Admits a prompt; returns (cached_tokens, slots int32[n]; -1 for cached tokens)."""
        np = self._np
        t = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        slots = np.empty(t.size, dtype=np.int32)
        rc = self._lib.pkv_bm_add_sequence(self._h, int(seq_id), t.ctypes.data, int(t.size),
                                           int(extra_key) & 0xFFFFFFFFFFFFFFFF, slots.ctypes.data)
        return self._rc(rc, "add_sequence"), slots

    def fork(self, parent: int, child: int) -> None:
        self._rc(self._lib.pkv_bm_fork(self._h, int(parent), int(child)), "fork")

    def append(self, seq_id: int, token: int):
        """Appends one token; returns (slot, (cow_src, cow_dst) or None)."""
        slot, src, dst = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        self._rc(self._lib.pkv_bm_append(self._h, int(seq_id), int(token), ctypes.byref(slot), ctypes.byref(src),
                                         ctypes.byref(dst)), "append")
        return slot.value, ((src.value, dst.value) if src.value >= 0 else None)

    def decode_step(self, seq_ids, tokens, max_blocks_per_seq: int, pad_value: int = -1):
        """pkv_bm_decode_step: appends tokens[i] to seq_ids[i] for the whole batch at once and returns
        the device step's host inputs (slot_mapping int32[n], context_lens int32[n],
        block_tables int32[n, max_blocks_per_seq], cow_pairs int32[P, 2]).  All or nothing."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64).reshape(-1)
        toks = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        if ids.size != toks.size:
            raise PkvError("decode_step: one token per sequence")
        n, w = ids.size, int(max_blocks_per_seq)
        slots = np.empty(n, dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        tables = np.empty((n, w), dtype=np.int32)
        pairs = np.empty((max(n, 1), 2), dtype=np.int32)
        rc = self._lib.pkv_bm_decode_step(self._h, ids.ctypes.data, toks.ctypes.data, n, slots.ctypes.data,
                                          lens.ctypes.data, tables.ctypes.data, w, int(pad_value),
                                          pairs.ctypes.data)
        p = self._rc(rc, "decode_step")
        return slots, lens, tables, pairs[:p].copy()

    def stats(self) -> dict:
        """pkv_bm_get_stats as a dict (gauges at the call, counters since creation)."""
        st = _BmStats()
        self._rc(self._lib.pkv_bm_get_stats(self._h, ctypes.byref(st)), "get_stats")
        return {name: int(getattr(st, name)) for name, _ in _BmStats._fields_}

    def free(self, seq_id: int) -> None:
        self._rc(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)), "free_sequence")

    def seq_len(self, seq_id: int) -> int:
        return self._rc(self._lib.pkv_bm_seq_len(self._h, int(seq_id)), "seq_len")

    def _blocks(self, fn, seq_id, what):
        np = self._np
        cap = self.num_blocks
        out = np.empty(cap, dtype=np.int32)
        n = self._rc(fn(self._h, int(seq_id), out.ctypes.data, cap), what)
        return out[:n].copy()

    def tokens(self, seq_id: int):
        """pkv_bm_seq_tokens: the sequence's token history (int32)."""
        np = self._np
        n = self.seq_len(seq_id)
        out = np.empty(max(n, 1), dtype=np.int32)
        m = self._rc(self._lib.pkv_bm_seq_tokens(self._h, int(seq_id), out.ctypes.data, n), "seq_tokens")
        return out[:m].copy()

    def block_table(self, seq_id: int):
        return self._blocks(self._lib.pkv_bm_block_table, seq_id, "block_table")

    def swap_out(self, seq_id: int):
        """Releases the sequence's blocks; returns them (logical order) for the device-to-host copy."""
        return self._blocks(self._lib.pkv_bm_swap_out, seq_id, "swap_out")

    def swap_in(self, seq_id: int):
        """Takes fresh blocks for a swapped-out sequence; returns them (logical order)."""
        return self._blocks(self._lib.pkv_bm_swap_in, seq_id, "swap_in")

    def swap_in_cached(self, seq_id: int):
        """swap_in reusing still-cached prefix blocks: returns (blocks, from_host) int32 arrays in
        logical order; from_host[i] == 1 where host block i must be moved to blocks[i]."""
        np = self._np
        cap = self.num_blocks
        blocks = np.empty(cap, dtype=np.int32)
        from_host = np.empty(cap, dtype=np.int32)
        n = self._rc(self._lib.pkv_bm_swap_in_cached(self._h, int(seq_id), blocks.ctypes.data,
                                                     from_host.ctypes.data, cap), "swap_in_cached")
        return blocks[:n].copy(), from_host[:n].copy()
