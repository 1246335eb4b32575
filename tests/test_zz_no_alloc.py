"""The scratch-free decode entry point, called through the C ABI.

pkv_decode_attention_static_workspace serves callers that cannot allocate
device memory when they run decode (framework plugins whose host owns all
device memory, loops that cannot take an allocation's synchronisation, C
callers without an allocator): the split-K partials live in a fixed array
inside the library instead of a caller workspace.  This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import DeviceStep

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


@pytest.fixture(scope="module")
def entry():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = pkv.load(build_if_missing=True)
    fn = lib.pkv_decode_attention_static_workspace
    fn.restype = ctypes.c_int
    fn.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p] +
                   [ctypes.c_int] * 6 +
                   [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                    ctypes.c_void_p])
    return fn


def _call(fn, ds, out):
    kv = pkv.PKV_BF16 if ds.k_pool.dtype == torch.bfloat16 else pkv.PKV_F16
    NB, B, Hkv, D = ds.k_pool.shape
    S, Hq, _ = ds.q.shape
    return fn(out.data_ptr(), ds.q.data_ptr(), ds.k_pool.data_ptr(), ds.v_pool.data_ptr(), 0,
              ds.block_tables.data_ptr(), ds.block_tables.shape[1], ds.context_lens.data_ptr(), S, Hq, Hkv, D, B,
              NB, ds.wl.scale, ds.partition_size, ds.max_context_len, kv, pkv.PKV_F32, ds.status.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("first,second", [((2, 64), (5, 128)), ((3, 256), (2, 32))])
def test_static_workspace_matches_workspace_entry_point(entry, first, second):
    """Two calls in a row (different workloads, split-K partials in the
    shared array) each agree with pkv_decode_attention."""
    for cfg, ps in (first, second):
        kw = dict(num_seqs=12) if cfg != 5 else dict(num_seqs=12, lens=("prefix", 256, 0, 300))
        wl = P.make_workload(cfg, poison=True, partition_size=ps, **kw)
        ds = DeviceStep(wl)
        assert 0 < pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.max_context_len,
                                              ps) <= STATIC_BYTES
        ds.copy()
        ds.write()
        ds.attend()
        out = torch.full_like(ds.out, float("nan"))
        assert _call(entry, ds, out) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert int(ds.status.item()) == 0
        assert torch.isfinite(out).all()
        # the same kernels on the same inputs: only where the partials live differs
        assert torch.equal(out, ds.out)


def test_static_workspace_rejects_oversized_calls(entry):
    wl = P.make_workload(2, num_seqs=4)
    ds = DeviceStep(wl)
    ds.partition_size = 16
    ds.max_context_len = 1 << 20  # needs far more than the fixed array
    need = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, ds.max_context_len, 16)
    assert need > STATIC_BYTES
    assert _call(entry, ds, ds.out) == pkv.PKV_ERR_WORKSPACE
