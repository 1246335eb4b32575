"""The SM-streaming partition kernel: one persistent CTA per SM takes
(sequence, KV head, partition) units from a longest-first queue held in the
workspace's control words.  Its results are checked against the oracle on
the batch shapes its plan has to get right (no partial partitions, only
partial ones, empty sequences, one sequence, the largest batch it plans for,
more CTAs than units, the grid kernel just past its limit), the control
words must read zero after every call, and repeated calls must agree bit
for bit (the queue hands units to different CTAs each time, but every unit
is computed the same way)."""
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
    # the largest batch the kernel plans for
    "max_batch": dict(cfg=3, num_seqs=1024, lens=("uniform", 1, 100), ps=32),
    # one more sequence: the grid kernel
    "grid_fallback": dict(cfg=3, num_seqs=1025, lens=("uniform", 1, 100), ps=32),
    # fewer units than CTAs
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
def test_stream_kernel_matches_oracle(name):
    wl = _workload(name)
    k, v, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl)
    out = ds.fused_step().cpu().numpy()
    assert ds.status_bits() == 0
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)
    assert float(np.max(np.abs(out - ref))) <= ATOL
    assert np.all(np.isfinite(out))
    # the queue's control words are back at zero for the next call
    assert ds.workspace is None or int(ds.workspace[:8].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("name", ["partial_only", "with_empty", "one_sequence"])
def test_stream_kernel_both_dtypes_and_head_dim_64(name, dtype):
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
    assert int(ds.workspace[:8].view(torch.int32).abs().sum()) == 0


def test_calls_of_different_sizes_share_one_workspace():
    """The control words sit at the start of every layout, so a workspace
    sized for the largest call serves smaller ones in any order."""
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
