"""Bad indices become status bits, never faults: the kernels range-check
every table entry, slot, copy pair and length, skip the bad element and OR a
PKV_DEV_ERR_* bit into the caller's status word.  Everything else is still
computed correctly."""
import time

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


@pytest.mark.parametrize("ps", [0, 64, pkv.PARTITION_BALANCED])
def test_out_of_range_table_entry(ps):
    wl = P.make_workload(2, num_seqs=6)
    k, v, ref = oracle.apply_step(wl)
    bt = wl.block_tables.copy()
    bt[2, 1] = wl.num_blocks + 7  # past the pool
    ds = DeviceStep(wl, partition_size=ps)
    ds.block_tables = torch.from_numpy(bt).cuda()
    out = ds.step().cpu().numpy()
    assert ds.status_bits() & pkv.DEV_ERR_BLOCK
    others = [s for s in range(wl.num_seqs) if s != 2]
    assert float(np.max(np.abs(out[others] - ref[others]))) <= ATOL
    assert np.all(np.isfinite(out[2]))


def test_out_of_range_slot_and_negative_slot():
    wl = P.make_workload(1)
    sm = wl.slot_mapping.copy()
    sm[0] = wl.num_blocks * 16  # one past the last slot
    sm[3] = -5                  # negative and not the padding marker
    ds = DeviceStep(wl)
    ds.slot_mapping = torch.from_numpy(sm).cuda()
    ds.write()
    assert ds.status_bits() & pkv.DEV_ERR_SLOT
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.write_cache(k, v, wl.k_new[1:3], wl.v_new[1:3], wl.slot_mapping[1:3])
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)


def test_out_of_range_copy_pair():
    wl = P.make_workload(5, num_seqs=16, lens=("prefix", 64, 0, 70))
    pairs = wl.copy_pairs.copy()
    assert len(pairs) >= 2
    pairs[0, 1] = wl.num_blocks  # dst past the pool
    ds = DeviceStep(wl)
    ds.pairs = torch.from_numpy(pairs).cuda()
    ds.copy()
    assert ds.status_bits() & pkv.DEV_ERR_PAIR
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(k, v, pairs[1:])
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)


@pytest.mark.parametrize("ps", [0, 64, pkv.PARTITION_BALANCED])
def test_length_beyond_bound_is_clamped_and_flagged(ps):
    wl = P.make_workload(2, num_seqs=5)
    k, v, _ = oracle.apply_step(wl, attention=False)
    ds = DeviceStep(wl, partition_size=ps)
    cl = wl.context_lens.copy()
    cl[1] = ds.max_context_len + 100  # beyond the host bound the grid was sized for
    ds.context_lens = torch.from_numpy(cl).cuda()
    out = ds.step().cpu().numpy()
    assert ds.status_bits() & pkv.DEV_ERR_LENGTH
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    others = [s for s in range(wl.num_seqs) if s != 1]
    assert float(np.max(np.abs(out[others] - ref[others]))) <= ATOL
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("shared_ring", [False, True])
@pytest.mark.parametrize("limit_ms", [2, 20])
def test_timed_out_wait_sets_the_status_bit_and_the_context_stays_usable(limit_ms, shared_ring):
    """A tile wait that nothing completes ends after its limit with
    PKV_DEV_ERR_TIMEOUT (the decode kernels' bounded wait and drain, run with
    a short limit and no copy in flight; with shared_ring, one warp of four
    times out and the CTA-wide vote of the shared-ring kernels sends all four
    out); the same context then runs a normal decode step that matches the
    oracle."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    pkv.check_bounded_wait(limit_ms * 1_000_000, status, shared_ring=shared_ring)
    e1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert int(status.item()) == pkv.DEV_ERR_TIMEOUT
    waited_ms = e0.elapsed_time(e1)
    assert 0.5 * limit_ms <= waited_ms < limit_ms + 500, waited_ms
    assert wall < 5.0
    wl = P.make_workload(2, num_seqs=5, poison=True)
    _, _, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl, partition_size=64)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    assert float(np.max(np.abs(out - ref))) <= ATOL


def test_bounded_wait_check_rejects_bad_arguments():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.check_bounded_wait(-1, status)
    with pytest.raises(pkv.PkvError):
        pkv.check_bounded_wait(3_000_000_000, status)
    assert pkv.load().pkv_check_bounded_wait(1000, 0, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert pkv.load().pkv_check_bounded_wait(1000, 3, None, None) == pkv.PKV_ERR_INVALID_ARG
