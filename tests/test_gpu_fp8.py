"""FP8 (e4m3) pools with per-(block, KV head) scales on the GPU, checked
against the FP8 oracle: the write path and the copy-on-write copy bit for
bit (codes and scales), decode attention within ATOL, at sizes the oracle
finishes in seconds (several partitions, ragged tails, one and two warps per
unit, both reduce kernels, the head-group grid and the one-head-per-copy
kernel) and at the benchmark's full sizes, every row.  Pools are poisoned:
NaN codes in every slot no sequence owns and NaN scales on blocks nothing
references."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStepFp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def _ref_pools(wl, pools):
    k8, v8 = pools.k8.copy(), pools.v8.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    oracle.copy_blocks_fp8(k8, v8, ks, vs, wl.copy_pairs)
    oracle.write_cache_fp8(k8, v8, ks, vs, wl.k_new, wl.v_new, wl.slot_mapping, wl.dtype)
    return k8, v8, ks, vs


def _check_pools(ds, ref):
    k8, v8, ks, vs = ref
    assert np.array_equal(ds.k8.cpu().numpy(), k8)
    assert np.array_equal(ds.v8.cpu().numpy(), v8)
    assert np.array_equal(ds.k_scale.cpu().numpy(), ks, equal_nan=True)
    assert np.array_equal(ds.v_scale.cpu().numpy(), vs, equal_nan=True)


SMALL = {
    # several partitions and ragged tails, one warp per unit
    "c2_ps16": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), ps=16),
    "c2_ps64": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), ps=64),
    "c2_single": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), ps=0),
    # 256 x 8 sequence-heads overfill the warp slots: two warps per unit
    "c3_two_warps": dict(cfg=3, num_seqs=256, lens=("uniform", 1, 90), ps=32),
    # shared prefix, copy-on-write of partial tail blocks
    "c5_prefix": dict(cfg=5, num_seqs=8, lens=("prefix", 64, 0, 40), ps=32),
    # more than 16 partitions per row: the long-row reduce kernel
    "c4_long": dict(cfg=4, num_seqs=2, lens=("uniform", 3000, 5000), ps=128),
    # KV head counts not divisible by 4: write-then-attend runs the one-head-per-copy partition kernel
    "hkv2": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), ps=64, num_q_heads=8, num_kv_heads=2),
    "hkv6_two_warps": dict(cfg=3, num_seqs=400, lens=("uniform", 1, 90), ps=32, num_q_heads=24, num_kv_heads=6),
}


def _small(case, dtype=None):
    c = dict(SMALL[case])
    kw = dict(num_seqs=c["num_seqs"], lens=c["lens"], partition_size=c["ps"])
    kw.update({k: c[k] for k in ("num_q_heads", "num_kv_heads") if k in c})
    if dtype:
        kw["dtype"] = dtype
    wl = P.make_workload(c["cfg"], poison=True, **kw)
    return wl, P.make_fp8_pools(wl)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("case", sorted(SMALL))
def test_fp8_step_matches_oracle(case, dtype):
    wl, pools = _small(case, dtype)
    ds = DeviceStepFp8(wl, pools)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    ref_pools = _ref_pools(wl, pools)
    _check_pools(ds, ref_pools)
    k8, v8, ks, vs = ref_pools
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL, err


def _fused_unit_warps(wl):
    """Warps per unit of the fused step's partition kernel: 2 when the
    sequences x KV heads overfill its warp slots (six 2-warp CTAs per SM)."""
    slots = 12 * torch.cuda.get_device_properties(0).multi_processor_count
    return 2 if wl.num_seqs * wl.num_kv_heads > slots else 1


@pytest.mark.parametrize("case", sorted(SMALL))
def test_fp8_fused_step_equals_write_then_attend(case):
    """The write fused into the partition kernel stores the same codes and
    gives the same output as the write kernel followed by attention: bit for
    bit where both sum a unit's tiles in the same order (one warp per unit;
    the head-group grid of write-then-attend keeps that order), else to
    float32 rounding (two warps per unit merge two halves)."""
    for dtype in (["f16", "bf16"] if case == "c2_ps16" else [None]):
        wl, pools = _small(case, dtype)
        a, b = DeviceStepFp8(wl, pools), DeviceStepFp8(wl, pools)
        out_a = a.step().clone()
        out_b = b.fused_step().clone()
        assert a.status_bits() == 0 and b.status_bits() == 0
        if _fused_unit_warps(wl) == 1 or wl.num_kv_heads % 4 != 0:
            assert torch.equal(out_a.view(torch.int32), out_b.view(torch.int32))
        else:
            assert float((out_a - out_b).abs().max()) <= 1e-5
        assert torch.equal(a.k8, b.k8) and torch.equal(a.v8, b.v8)
        assert torch.equal(a.k_scale.view(torch.int32), b.k_scale.view(torch.int32))


def test_fp8_fused_step_slot_checks():
    """slot -1: no write, no flag; a slot that is not position L-1 through
    the table: PKV_DEV_ERR_SLOT and no write; everything else as the oracle."""
    wl, pools = _small("c2_ps64", "f16")
    sm = wl.slot_mapping.copy()
    s_skip, s_bad = 0, 1
    sm[s_skip] = -1
    sm[s_bad] = sm[s_bad] ^ 1 if wl.context_lens[s_bad] > 1 else sm[s_bad] + 1  # another slot of the pool
    wl.slot_mapping = sm
    ds = DeviceStepFp8(wl, pools)
    ds.fused_step()
    assert ds.status_bits() == pkv.DEV_ERR_SLOT
    k8 = ds.k8.cpu().numpy()
    for s in (s_skip, s_bad):
        b, o = divmod(int(sm[s]) if sm[s] >= 0 else 0, 16)
        if sm[s] >= 0:
            assert np.array_equal(k8[b, o], pools.k8[b, o])  # untouched
    # the other sequences' rows were written as the oracle writes them
    keep = [s for s in range(wl.num_seqs) if s not in (s_skip, s_bad)]
    ks = pools.k_scale.copy()
    for s in keep:
        b, o = divmod(int(sm[s]), 16)
        x = P.bits_to_f32(wl.k_new[s], wl.dtype)
        want = oracle.e4m3_encode(x / ks[b][:, None])
        assert np.array_equal(k8[b, o], want)


def test_fp8_write_saturates_and_rounds_like_the_oracle():
    """New rows scaled up so that many quotients pass 448: saturated codes
    and round-to-nearest-even agree with the oracle bit for bit."""
    wl, pools = _small("c2_ps16", "bf16")
    big = P.bits_to_f32(wl.k_new, "bf16") * 40.0
    wl.k_new = P.f32_to_bits(big, "bf16")
    ds = DeviceStepFp8(wl, pools)
    ds.copy()
    ds.write()
    assert ds.status_bits() == 0
    _check_pools(ds, _ref_pools(wl, pools))
    k8 = ds.k8.cpu().numpy()
    written = np.stack([k8[s // 16, s % 16] for s in wl.slot_mapping.tolist()])
    assert np.mean((written & 0x7F) == 0x7E) > 0.05


def test_fp8_bf16_queries_beyond_f16_range():
    """bf16 queries of magnitude ~1e6 (beyond f16) with the softmax scale
    reduced to match: the kernel's power-of-two prescale keeps them exact."""
    wl, pools = _small("c2_ps64", "bf16")
    wl.q = P.f32_to_bits(P.bits_to_f32(wl.q, "bf16") * np.float32(2.0 ** 20), "bf16")
    assert np.max(np.abs(P.bits_to_f32(wl.q, "bf16"))) > 65504
    wl.scale = wl.scale * 2.0 ** -20
    ds = DeviceStepFp8(wl, pools)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    k8, v8, ks, vs = _ref_pools(wl, pools)
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert float(np.max(np.abs(out - ref))) <= ATOL


def test_fp8_empty_and_one_token_sequences():
    """L = 0 gives a zero row; L = 1 gives the dequantised v_0."""
    wl, pools = _small("c2_ps16", "f16")
    ds = DeviceStepFp8(wl, pools)
    ds.copy()
    ds.write()
    cl = wl.context_lens.copy()
    cl[0], cl[1] = 0, 1
    ds.context_lens.copy_(torch.from_numpy(cl))
    ds.attend()
    out = ds.out.cpu().numpy()
    assert ds.status_bits() == 0
    k8, v8, ks, vs = _ref_pools(wl, pools)
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, cl, wl.scale, wl.dtype)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert float(np.max(np.abs(out - ref))) <= ATOL


def test_fp8_bad_table_entry_is_flagged():
    wl, pools = _small("c2_ps64", "f16")
    ds = DeviceStepFp8(wl, pools)
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
    keep = [s for s in range(wl.num_seqs) if s != s_bad]
    rows = [(s, h) for s in keep for h in range(wl.num_q_heads)]
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                      rows=rows)
    got = np.stack([out[s, h] for s, h in rows])
    assert float(np.max(np.abs(got - ref))) <= ATOL


@pytest.mark.parametrize("cfg", [2, 3, 4, 5])
def test_fp8_full_size_step(cfg):
    """The benchmark's workloads at the partition sizes the FP8 bench runs
    (fp32 output), every row against the oracle."""
    wl = P.make_workload(cfg, poison=True)
    pools = P.make_fp8_pools(wl)
    ds = DeviceStepFp8(wl, pools, partition_size=P.fp8_partition_size(cfg))
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    ref_pools = _ref_pools(wl, pools)
    _check_pools(ds, ref_pools)
    k8, v8, ks, vs = ref_pools
    ref = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    err = float(np.max(np.abs(out.astype(np.float64) - ref)))
    assert err <= ATOL, err
    assert np.all(np.isfinite(out))
