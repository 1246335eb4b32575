"""GPU parity: the library's kernels against the fp64 oracle on the same seeded
inputs.  Writes and copies are bit-exact; attention is within 2e-3 max-abs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStep, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def _max_err(got, ref):
    return float(np.max(np.abs(got.astype(np.float64) - ref))) if ref.size else 0.0


def test_config1_step():
    wl = P.make_workload(1, poison=True)
    ds = DeviceStep(wl)
    out = ds.step().cpu().numpy()
    k_ref, v_ref, ref = oracle.apply_step(wl)
    assert np.array_equal(to_bits(ds.k_pool), k_ref)
    assert np.array_equal(to_bits(ds.v_pool), v_ref)
    assert np.all(np.isfinite(out))
    assert _max_err(out, ref) <= ATOL
    assert ds.status_bits() == 0


SHAPES = [  # (H_q, H_kv, D): group sizes 1, 2, 3, 4, 8
    (4, 4, 64), (4, 2, 64), (6, 2, 128), (8, 2, 128), (16, 2, 128), (24, 3, 64),
]
LENS = [0, 1, 15, 16, 17, 33, 100, 257, 600]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
@pytest.mark.parametrize("ps", [0, 16, 48, 512, pkv.PARTITION_BALANCED])
def test_decode_sweep(dtype, shape, ps):
    Hq, Hkv, D = shape
    lens = [L for L in LENS] + [1]
    wl = P.make_workload(2, num_seqs=len(lens), lens=("fixed", [max(L, 1) for L in lens]), num_q_heads=Hq,
                         num_kv_heads=Hkv, head_dim=D, dtype=dtype, partition_size=ps, poison=True,
                         seed=100 + Hq + D + ps)
    wl.context_lens[0] = 0  # an empty sequence gives a zero row
    ds = DeviceStep(wl)
    out = ds.step().cpu().numpy()
    k_ref, v_ref, _ = oracle.apply_step(wl, attention=False)
    ref = oracle.decode_attention(wl.q, k_ref, v_ref, wl.block_tables, wl.context_lens, wl.scale, dtype)
    assert np.array_equal(to_bits(ds.k_pool), k_ref)
    assert np.all(out[0] == 0)
    err = _max_err(out, ref)
    assert err <= ATOL, err
    assert ds.status_bits() == 0


def test_copy_blocks_bit_exact():
    wl = P.make_workload(5, num_seqs=24, lens=("prefix", 64, 0, 70), poison=True)
    assert wl.copy_pairs.shape[0] > 0
    ds = DeviceStep(wl)
    ds.copy()
    torch.cuda.synchronize()
    k = wl.k_pool.copy()
    v = wl.v_pool.copy()
    oracle.copy_blocks(k, v, wl.copy_pairs)
    assert np.array_equal(to_bits(ds.k_pool), k)
    assert np.array_equal(to_bits(ds.v_pool), v)
    assert ds.status_bits() == 0


def test_write_cache_padding_and_strided_rows():
    wl = P.make_workload(1)
    ds = DeviceStep(wl)
    sm = wl.slot_mapping.copy()
    sm[2] = -1
    ds.slot_mapping = torch.from_numpy(sm).cuda()
    # new rows taken from a wider fused buffer: [T, 3 * H_kv, D], K and V slices
    T, Hkv, D = wl.k_new.shape
    fused = torch.zeros(T, 3 * Hkv, D, dtype=ds.k_new.dtype, device="cuda")
    fused[:, Hkv:2 * Hkv] = ds.k_new
    fused[:, 2 * Hkv:] = ds.v_new
    ds.k_new, ds.v_new = fused[:, Hkv:2 * Hkv], fused[:, 2 * Hkv:]
    ds.write()
    torch.cuda.synchronize()
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.write_cache(k, v, wl.k_new, wl.v_new, sm)
    assert np.array_equal(to_bits(ds.k_pool), k)
    assert np.array_equal(to_bits(ds.v_pool), v)


@pytest.mark.parametrize("ps", [64, pkv.PARTITION_BALANCED])
def test_split_kernels_equal_fused_call_and_are_deterministic(ps):
    wl = P.make_workload(2, num_seqs=6, poison=True)
    ds = DeviceStep(wl, partition_size=ps)
    ds.copy()
    ds.write()
    ds.attend()
    a = ds.out.clone()
    ds.attend()
    b = ds.out.clone()
    out2 = torch.empty_like(ds.out)
    pkv.decode_partitions(out2, ds.q, ds.k_pool, ds.v_pool, ds.block_tables, ds.context_lens, wl.scale,
                          partition_size=ps, max_context_len=ds.max_context_len, workspace=ds.workspace)
    pkv.decode_reduce(out2, ds.context_lens, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                      head_dim=wl.head_dim, partition_size=ps, max_context_len=ds.max_context_len,
                      workspace=ds.workspace)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(a, out2)


@pytest.mark.parametrize("odt", [torch.float16, torch.bfloat16])
def test_16bit_output_is_rounded_fp32_output(odt):
    wl = P.make_workload(3, num_seqs=16, poison=True)
    ds = DeviceStep(wl, partition_size=128)
    ds.step()
    o16 = torch.empty(ds.out.shape, dtype=odt, device="cuda")
    ds.attend(out=o16)
    torch.cuda.synchronize()
    assert torch.equal(o16, ds.out.to(odt))


def test_partition_size_does_not_change_much():
    wl = P.make_workload(2, num_seqs=8, poison=True)
    outs = []
    for ps in (0, 16, 64, 512, pkv.PARTITION_BALANCED):
        ds = DeviceStep(wl, partition_size=ps)
        outs.append(ds.step().cpu().numpy())
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 1e-4


@pytest.mark.parametrize("num_seqs,lens", [(1, ("fixed", [5000])), (300, ("uniform", 1, 40)),
                                           (40, ("fixed", [16] * 40))])
def test_balanced_split_shapes(num_seqs, lens):
    """Balanced split on one long sequence (many warps on one pair), many tiny
    sequences (a warp crossing many pairs) and block-aligned lengths."""
    wl = P.make_workload(2, num_seqs=num_seqs, lens=lens, poison=True, partition_size=pkv.PARTITION_BALANCED,
                         seed=7 + num_seqs)
    ds = DeviceStep(wl)
    out = ds.step().cpu().numpy()
    k_ref, v_ref, ref = oracle.apply_step(wl)
    assert _max_err(out, ref) <= ATOL
    assert ds.status_bits() == 0
