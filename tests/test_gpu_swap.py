"""Swap out / swap in of block lists between the device pool and a pool in
pinned host memory ("gpu_paged_kv_cache", "Reclaiming memory: swap versus
recompute"; "PagedAttention internals", section 05), checked against the
oracle byte for byte; a swapped-in sequence, its table repointed to other
blocks, attends bit-identically on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStep, DeviceStepFp8, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def _victims(wl, n):
    """The blocks of the n longest sequences (what a preemption would swap out)."""
    order = np.argsort(-wl.context_lens)[:n]
    blocks = []
    for s in order:
        blocks += wl.block_tables[s, : -(-int(wl.context_lens[s]) // 16)].tolist()
    return order, np.asarray(blocks, dtype=np.int32)


def _free_blocks(wl, n, rng):
    used = set(wl.block_tables[wl.block_tables >= 0].tolist()) | set(wl.copy_pairs.reshape(-1).tolist())
    free = np.array([b for b in range(wl.num_blocks) if b not in used], dtype=np.int32)
    return rng.permutation(free)[:n]


def test_swap_out_and_in_to_other_blocks():
    wl = P.make_workload(2, poison=True, num_seqs=16, lens=("uniform", 100, 600), partition_size=128,
                         pool_factor=2.0)
    ds = DeviceStep(wl)
    before = ds.step().clone()
    order, victims = _victims(wl, 3)
    n = victims.size
    hk = torch.zeros((n,) + tuple(ds.k_pool.shape[1:]), dtype=ds.k_pool.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = torch.from_numpy(np.stack([victims, np.arange(n, dtype=np.int32)], 1)).cuda()
    pkv.swap_blocks(hk, hv, ds.k_pool, ds.v_pool, out_pairs, status=ds.status)
    torch.cuda.synchronize()
    k_dev, v_dev = to_bits(ds.k_pool), to_bits(ds.v_pool)
    ref_hk, ref_hv = np.zeros((n,) + k_dev.shape[1:], np.uint16), np.zeros((n,) + v_dev.shape[1:], np.uint16)
    oracle.swap_blocks(ref_hk, ref_hv, k_dev, v_dev, out_pairs.cpu().numpy())
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), ref_hk)
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), ref_hv)
    # the victims' blocks are freed and reused: poison them
    nan = torch.tensor(P.NAN_BITS[wl.dtype], dtype=torch.int16).view(ds.k_pool.dtype)
    vict = torch.from_numpy(victims).cuda().long()
    ds.k_pool[vict] = nan
    ds.v_pool[vict] = nan
    # resume: swap in to other free blocks (pairs in pinned host memory), repoint the tables
    target = _free_blocks(wl, n, np.random.default_rng(3))
    in_pairs = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), target], 1)).pin_memory()
    pkv.swap_blocks(ds.k_pool, ds.v_pool, hk, hv, in_pairs, status=ds.status)
    bt = wl.block_tables.copy()
    pos = 0
    for s in order:
        nb = -(-int(wl.context_lens[s]) // 16)
        bt[s, :nb] = target[pos:pos + nb]
        pos += nb
    ds.block_tables.copy_(torch.from_numpy(bt))
    ds.attend()
    torch.cuda.synchronize()
    assert ds.status_bits() == 0
    ref_k, ref_v = k_dev.copy(), v_dev.copy()
    ref_k[victims] = P.NAN_BITS[wl.dtype]
    ref_v[victims] = P.NAN_BITS[wl.dtype]
    oracle.swap_blocks(ref_k, ref_v, ref_hk, ref_hv, in_pairs.numpy())
    assert np.array_equal(to_bits(ds.k_pool), ref_k) and np.array_equal(to_bits(ds.v_pool), ref_v)
    assert torch.equal(ds.out.view(torch.int32), before.view(torch.int32))


def test_swap_all_layer_blocks():
    """An all-layer pool swaps whole blocks (every layer) in one call."""
    rng = np.random.default_rng(11)
    NB, L, Hkv, D = 24, 4, 2, 128
    pool = torch.from_numpy(rng.integers(-30000, 30000, size=(2, NB, L, 16, Hkv, D), dtype=np.int16)).cuda()
    host = torch.zeros((2, 6, L, 16, Hkv, D), dtype=torch.int16).pin_memory()
    pairs = torch.tensor([[5, 0], [17, 1], [2, 5], [23, 3]], dtype=torch.int32).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.swap_blocks(host[0], host[1], pool[0], pool[1], pairs, status=status)
    torch.cuda.synchronize()
    ref = np.zeros(host.shape, np.int16)
    p = pool.cpu().numpy()
    oracle.swap_blocks(ref[0], ref[1], p[0], p[1], pairs.cpu().numpy())
    assert int(status.item()) == 0 and np.array_equal(host.numpy(), ref)


def test_swap_fp8_codes_and_scales():
    """FP8 pools swap their codes and their per-(block, KV head) scales."""
    wl = P.make_workload(2, poison=True, num_seqs=8, lens=("uniform", 40, 200), partition_size=64, pool_factor=2.0)
    pools = P.make_fp8_pools(wl)
    ds = DeviceStepFp8(wl, pools)
    before = ds.step().clone()
    order, victims = _victims(wl, 2)
    n = victims.size
    hk8 = torch.zeros((n,) + tuple(ds.k8.shape[1:]), dtype=torch.uint8).pin_memory()
    hv8 = torch.zeros_like(hk8).pin_memory()
    hks = torch.zeros((n, wl.num_kv_heads), dtype=torch.float32).pin_memory()
    hvs = torch.zeros_like(hks).pin_memory()
    out_pairs = torch.from_numpy(np.stack([victims, np.arange(n, dtype=np.int32)], 1)).cuda()
    pkv.swap_blocks(hk8, hv8, ds.k8, ds.v8, out_pairs, status=ds.status)
    pkv.swap_blocks(hks, hvs, ds.k_scale, ds.v_scale, out_pairs, status=ds.status)
    target = _free_blocks(wl, n, np.random.default_rng(4))
    vict = torch.from_numpy(victims).cuda().long()
    torch.cuda.synchronize()
    ds.k8[vict] = P.FP8_NAN
    ds.v8[vict] = P.FP8_NAN
    ds.k_scale[vict] = float("nan")
    ds.v_scale[vict] = float("nan")
    in_pairs = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), target], 1)).cuda()
    pkv.swap_blocks(ds.k8, ds.v8, hk8, hv8, in_pairs, status=ds.status)
    pkv.swap_blocks(ds.k_scale, ds.v_scale, hks, hvs, in_pairs, status=ds.status)
    bt = wl.block_tables.copy()
    pos = 0
    for s in order:
        nb = -(-int(wl.context_lens[s]) // 16)
        bt[s, :nb] = target[pos:pos + nb]
        pos += nb
    ds.block_tables.copy_(torch.from_numpy(bt))
    ds.attend()
    assert ds.status_bits() == 0
    assert torch.equal(ds.out.view(torch.int32), before.view(torch.int32))


def test_swap_bad_pair_is_flagged_and_skipped():
    rng = np.random.default_rng(12)
    dev = torch.from_numpy(rng.integers(0, 255, size=(8, 4096), dtype=np.uint8)).cuda()
    host = torch.zeros((4, 4096), dtype=torch.uint8).pin_memory()
    pairs = torch.tensor([[1, 0], [9, 1], [3, 7], [2, 2]], dtype=torch.int32).cuda()  # 9: past 8 blocks; 7: past 4
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.swap_blocks(host, host, dev, dev, pairs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pkv.DEV_ERR_PAIR
    d = dev.cpu().numpy()
    assert np.array_equal(host[0].numpy(), d[1]) and np.array_equal(host[2].numpy(), d[2])
    assert not host[1].numpy().any() and not host[3].numpy().any()


def test_pageable_host_memory_is_refused():
    dev = torch.zeros((4, 4096), dtype=torch.uint8, device="cuda")
    host = torch.zeros((4, 4096), dtype=torch.uint8)  # not pinned
    pairs = torch.tensor([[0, 0]], dtype=torch.int32).cuda()
    with pytest.raises(pkv.PkvError):
        pkv.swap_blocks(host, host, dev, dev, pairs)
    # the same refusal in the C ABI itself (the binding's own check bypassed)
    lib = pkv.load()
    rc = lib.pkv_swap_blocks(host.data_ptr(), host.data_ptr(), 4096, 4, dev.data_ptr(), dev.data_ptr(), 4096, 4,
                             4096, pairs.data_ptr(), 1, None, None)
    assert rc == pkv.PKV_ERR_INVALID_ARG
