"""Split-K decode on the batch shapes whose partition bookkeeping is easy
to get wrong: every length a multiple of the partition (no partial
partition), every sequence shorter than one partition, empty sequences
among split ones, one long sequence split many ways, a large batch of
short ones, partitions of 1024 and 2048 tokens, fewer units than SMs, and a
shared prefix with copy-on-write.  Each is checked against the oracle
through the fused step, both 16-bit types and head_dim 64 on a subset;
repeated calls agree bit for bit, and one workspace sized for the largest
call serves smaller calls in any order."""
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


CASES = {
    # every length a multiple of the partition: full units only
    "full_only": dict(cfg=2, num_seqs=12, lens=("fixed", [64, 128, 192, 64, 256, 64, 128, 320, 64, 64, 192, 128]),
                      ps=64),
    # every sequence shorter than one partition: partial units only (single-partition outputs)
    "partial_only": dict(cfg=3, num_seqs=40, lens=("uniform", 1, 63), ps=64),
    # empty sequences among split ones (lengths 0 set after the build, their slots -1)
    "with_empty": dict(cfg=2, num_seqs=9, lens=("fixed", [1, 300, 1, 17, 1, 1, 512, 33, 1]), ps=32,
                       empty=[0, 2, 5, 8]),
    # one long sequence split many ways
    "one_sequence": dict(cfg=4, num_seqs=1, lens=("fixed", [5000]), ps=128),
    # a large batch of short sequences
    "large_batch": dict(cfg=3, num_seqs=1025, lens=("uniform", 1, 100), ps=32),
    # large partitions
    "partition_1024": dict(cfg=2, num_seqs=10, lens=("uniform", 900, 2600), ps=1024),
    "partition_2048": dict(cfg=2, num_seqs=10, lens=("uniform", 900, 2600), ps=2048),
    # fewer units than SMs
    "few_units": dict(cfg=1, num_seqs=4, lens=("fixed", [1, 17, 33, 50]), ps=16),
    # prefix sharing with copy-on-write, split
    "prefix": dict(cfg=5, num_seqs=16, lens=("prefix", 256, 0, 100), ps=64),
}


def _workload(name, **kw):
    c = dict(CASES[name])
    cfg = c.pop("cfg")
    ps = c.pop("ps")
    empty = c.pop("empty", [])
    c.update(kw)
    wl = P.make_workload(cfg, poison=True, partition_size=ps, **c)
    for s in empty:  # an empty sequence: no history, no token written this step
        wl.context_lens[s] = 0
        wl.slot_mapping[s] = -1
    return wl


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_edge_case_matches_oracle(name):
    wl = _workload(name)
    k, v, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl)
    out = ds.fused_step().cpu().numpy()
    assert ds.status_bits() == 0
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)
    assert float(np.max(np.abs(out - ref))) <= ATOL
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("name", ["partial_only", "with_empty", "one_sequence"])
def test_split_edge_case_both_dtypes_and_head_dim_64(name, dtype):
    wl = _workload(name, dtype=dtype, head_dim=64)
    _, _, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    assert float(np.max(np.abs(out - ref))) <= ATOL


def test_repeated_calls_agree_bit_for_bit():
    wl = P.make_workload(3, num_seqs=200, poison=True, partition_size=128)
    ds = DeviceStep(wl)
    ds.copy()
    ds.write()
    outs = []
    for _ in range(5):
        ds.attend()
        outs.append(ds.out.clone())
    torch.cuda.synchronize()
    assert ds.status_bits() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int32), outs[0].view(torch.int32))
    _, _, ref = oracle.apply_step(wl)
    assert float(np.max(np.abs(outs[0].cpu().numpy() - ref))) <= ATOL


def test_calls_of_different_sizes_share_one_workspace():
    """A workspace sized for the largest call serves smaller ones in any
    order (a call's records depend only on its own sizes)."""
    big = P.make_workload(2, num_seqs=48, poison=True, partition_size=64)
    small = P.make_workload(3, num_seqs=10, poison=True, partition_size=32)
    dbig, dsmall = DeviceStep(big), DeviceStep(small)
    shared = max((dbig.workspace, dsmall.workspace), key=lambda w: w.numel())
    dbig.workspace = dsmall.workspace = shared
    for ds, wl in ((dbig, big), (dsmall, small), (dbig, big), (dsmall, small)):
        out = ds.step().cpu().numpy()
        assert ds.status_bits() == 0
        _, _, ref = oracle.apply_step(wl)
        assert float(np.max(np.abs(out - ref))) <= ATOL
