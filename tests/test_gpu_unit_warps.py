"""The partition kernel serves a unit (sequence, KV head, partition) with one
warp, or with two warps that split its blocks and merge their softmax states
through shared memory.  The host picks two when the sequences alone
(H_kv x S, a unit each at least) overfill one wave of warp slots, else one.
These cases take each path on a GB300 (152 SMs x 6 CTAs x 2 warps = 1824
warp slots) with short sequences the oracle finishes quickly, including a
one-warp batch whose partition-indexed grid is mostly empty and one whose
units exceed a wave; on another GPU the paths may differ but every result
must still match."""
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
    # 256 x 8 = 2048 sequence-heads > 1824 slots: two warps per unit.
    "two_warps": dict(cfg=3, num_seqs=256, lens=("uniform", 1, 90), ps=32, max_len=None),
    # 64 x 8 = 512 sequence-heads: one warp; a bound of 16 partitions per sequence
    # while the lengths need at most 2 leaves most of the grid empty.
    "one_warp_sparse": dict(cfg=2, num_seqs=64, lens=("uniform", 1, 30), ps=16, max_len=256),
    # same shape, lengths near the bound: 64 x 8 x ~15 units, several waves of one-warp units.
    "one_warp_waves": dict(cfg=2, num_seqs=64, lens=("uniform", 224, 255), ps=16, max_len=256),
}


def _workload(case, dtype=None):
    c = CASES[case]
    kw = dict(num_seqs=c["num_seqs"], lens=c["lens"], partition_size=c["ps"])
    if dtype:
        kw["dtype"] = dtype
    return P.make_workload(c["cfg"], **kw), c["max_len"]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_unit_warps_match_oracle(case, dtype):
    wl, max_len = _workload(case, dtype)
    k, v, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl)
    if max_len:
        ds.max_context_len = max_len
        nbytes = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, max_len, ds.partition_size)
        ds.workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    assert float(np.max(np.abs(out - ref))) <= ATOL
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)


@pytest.mark.parametrize("case", sorted(CASES))
def test_unit_warps_fused_step_equals_write_then_attend(case):
    wl, max_len = _workload(case)
    a, b = DeviceStep(wl), DeviceStep(wl)
    for ds in (a, b):
        if max_len:
            ds.max_context_len = max_len
            nbytes = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, max_len, ds.partition_size)
            ds.workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    out_a = a.step().clone()
    out_b = b.fused_step().clone()
    assert a.status_bits() == 0 and b.status_bits() == 0
    assert torch.equal(out_a.view(torch.int32), out_b.view(torch.int32))
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(a.v_pool.view(torch.int16), b.v_pool.view(torch.int16))
