"""The balanced split over FP8 pools (partition_size = PARTITION_BALANCED
through decode_attention_fp8) against the FP8 oracle, every row, on shapes
that take each path of its work split: fewer tiles than warps (every pair
cut into one-tile pieces), many short pairs per warp (odd last tiles that
go through a softmax step alone), long pairs crossing several 32-tile
chunks, a shared prefix, and empty sequences among split ones; then the
benchmark's 8B- and 70B-class layers at full size on sampled rows.

Also the accumulator's unit change at large V scales, for fixed partitions
and the balanced split: V scales multiplied by 2^11 (exact in f32) must
multiply the output by exactly 2^11.  The first unit change of a pair then
spans more than 126 binades, the case the kernels' unit_change covers."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStepFp8

pytestmark = pytest.mark.gpu

BAL = pkv.PARTITION_BALANCED


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


CASES = {
    # ~960 tiles for 1824 warps: every warp holds one tile, every pair is cut
    "few_tiles": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300)),
    # 64 query heads (group 8), 1-3 tiles per pair: several pairs per warp
    "many_short_pairs": dict(cfg=3, num_seqs=512, lens=("uniform", 1, 40)),
    # ~1500 tiles per pair, ~27 per warp: shares start mid-chunk and cross chunks
    "long_pairs": dict(cfg=4, num_seqs=4, lens=("uniform", 20000, 30000)),
    # shared prefix and copy-on-write of partial tail blocks
    "prefix": dict(cfg=5, num_seqs=8, lens=("prefix", 64, 0, 40)),
    # empty sequences (length 0, no token written) among split ones
    "with_empty": dict(cfg=2, num_seqs=9, lens=("fixed", [1, 300, 1, 17, 1, 1, 512, 33, 1]), empty=[0, 2, 5, 8]),
}


def _case(name, dtype=None):
    c = dict(CASES[name])
    cfg = c.pop("cfg")
    empty = c.pop("empty", [])
    if dtype:
        c["dtype"] = dtype
    wl = P.make_workload(cfg, poison=True, **c)
    for s in empty:  # an empty sequence: no history, no token written this step
        wl.context_lens[s] = 0
        wl.slot_mapping[s] = -1
    return wl, P.make_fp8_pools(wl)


def _ref_pools(wl, pools):
    k8, v8 = pools.k8.copy(), pools.v8.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    oracle.copy_blocks_fp8(k8, v8, ks, vs, wl.copy_pairs)
    oracle.write_cache_fp8(k8, v8, ks, vs, wl.k_new, wl.v_new, wl.slot_mapping, wl.dtype)
    return k8, v8, ks, vs


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_balanced_matches_oracle(name, dtype):
    wl, pools = _case(name, dtype)
    ds = DeviceStepFp8(wl, pools, partition_size=BAL)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    k8, v8, ks, vs = _ref_pools(wl, pools)
    assert np.array_equal(ds.k8.cpu().numpy(), k8) and np.array_equal(ds.v8.cpu().numpy(), v8)
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL, err
    for s in np.nonzero(wl.context_lens == 0)[0]:
        assert not np.any(out[s])


def test_fp8_balanced_repeats_bit_for_bit():
    """Same inputs, same bits: the split depends on the lengths and the SM
    count only."""
    wl, pools = _case("long_pairs")
    ds = DeviceStepFp8(wl, pools, partition_size=BAL)
    ds.copy()
    ds.write()
    outs = []
    for _ in range(3):
        ds.attend()
        torch.cuda.synchronize()
        outs.append(ds.out.clone())
    assert ds.status_bits() == 0
    assert all(torch.equal(o.view(torch.int32), outs[0].view(torch.int32)) for o in outs[1:])


def test_fp8_balanced_bad_table_entry_is_flagged():
    wl, pools = _case("few_tiles", "f16")
    ds = DeviceStepFp8(wl, pools, partition_size=BAL)
    ds.copy()
    ds.write()
    bt = wl.block_tables.copy()
    s_bad = int(np.argmax(wl.context_lens))
    bt[s_bad, 0] = wl.num_blocks + 3
    ds.block_tables.copy_(torch.from_numpy(bt))
    ds.attend()
    assert ds.status_bits() & pkv.DEV_ERR_BLOCK
    out = ds.out.cpu().numpy()
    k8, v8, ks, vs = _ref_pools(wl, pools)
    rows = [(s, h) for s in range(wl.num_seqs) if s != s_bad for h in range(wl.num_q_heads)]
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                      rows=rows)
    got = np.stack([out[s, h] for s, h in rows])
    assert float(np.max(np.abs(got - ref))) <= ATOL


@pytest.mark.parametrize("cfg", [2, 3])
def test_fp8_balanced_full_size(cfg):
    wl = P.make_workload(cfg, poison=True)
    pools = P.make_fp8_pools(wl)
    ds = DeviceStepFp8(wl, pools, partition_size=BAL)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    k8, v8, ks, vs = _ref_pools(wl, pools)
    rng = np.random.default_rng(cfg)
    S, Hq = wl.num_seqs, wl.num_q_heads
    rows = {(int(s), int(h)) for s, h in zip(rng.integers(0, S, 64), rng.integers(0, Hq, 64))}
    for s in (int(np.argmin(wl.context_lens)), int(np.argmax(wl.context_lens))):
        rows.update({(s, 0), (s, Hq - 1)})
    rows = sorted(rows)
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                      rows=rows)
    got = np.stack([out[s, h] for s, h in rows])
    assert float(np.max(np.abs(got.astype(np.float64) - ref))) <= ATOL
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("ps", [64, BAL])
def test_fp8_large_v_scales_scale_the_output_exactly(ps):
    """Copy-on-write and attention only (no write, so both pools hold the
    same codes), over unpoisoned pools."""
    c = dict(CASES["long_pairs" if ps == BAL else "few_tiles"])
    wl = P.make_workload(c.pop("cfg"), poison=False, dtype="f16", **c)
    pools = P.make_fp8_pools(wl, poison=False)
    big = dataclasses.replace(pools, v_scale=pools.v_scale * np.float32(2048.0))
    outs = []
    for pl in (pools, big):
        ds = DeviceStepFp8(wl, pl, partition_size=ps)
        ds.copy()
        ds.attend()
        assert ds.status_bits() == 0
        outs.append(ds.out.clone())
    assert torch.all(torch.isfinite(outs[1]))
    assert torch.equal(outs[1], outs[0] * 2048.0)
    k8, v8 = big.k8.copy(), big.v8.copy()
    ks, vs = big.k_scale.copy(), big.v_scale.copy()
    oracle.copy_blocks_fp8(k8, v8, ks, vs, wl.copy_pairs)
    rows = [(s, h) for s in range(min(wl.num_seqs, 4)) for h in range(0, wl.num_q_heads, 5)]
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                      rows=rows)
    got = np.stack([outs[1].cpu().numpy()[s, h] for s, h in rows])
    assert float(np.max(np.abs(got.astype(np.float64) - ref))) <= ATOL * 2048
