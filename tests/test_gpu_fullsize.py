"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (its partition size, fp32 output, one write token per sequence, the
recipe's copy-on-write pairs).  Pools are compared bit for bit in full and
every (sequence, query head) output row is compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStep, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


@pytest.mark.parametrize("cfg,ps", [(2, None), (3, None), (4, None), (5, None),
                                    (2, pkv.PARTITION_BALANCED), (3, pkv.PARTITION_BALANCED),
                                    (5, pkv.PARTITION_BALANCED)])
def test_full_size_step(cfg, ps):
    wl = P.make_workload(cfg, poison=True)
    ds = DeviceStep(wl, partition_size=ps)  # None: the recipe's partition size; fp32 output
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    k_ref, v_ref = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(k_ref, v_ref, wl.copy_pairs)
    oracle.write_cache(k_ref, v_ref, wl.k_new, wl.v_new, wl.slot_mapping)
    assert np.array_equal(to_bits(ds.k_pool), k_ref)
    assert np.array_equal(to_bits(ds.v_pool), v_ref)
    ref = oracle.decode_attention(wl.q, k_ref, v_ref, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL, err
    # every row is finite (NaN poison in unowned slots never leaks)
    assert np.all(np.isfinite(out))
