"""Blocks of 8, 32 and 64 tokens besides the default 16 ("gpu_paged_kv_cache",
"Fixed-size blocks and the block-table indirection": 16 is the common
default; long sequences tolerate larger blocks, short ones and prefix reuse
want smaller).  The partition kernel's 16-token tiles are a part of one
block (B >= 16) or two 8-token blocks; every path is checked against the
oracle run with the same block size."""
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
    # several partitions of 64 tokens and ragged tails, one warp per unit
    "c2_ps64": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), partition_size=64),
    # partitions that start inside a 64-token block (48 = 3 tiles)
    "c2_ps48": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), partition_size=48),
    # one partition per sequence
    "c2_single": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), partition_size=0),
    # two warps per unit
    "c3_two_warps": dict(cfg=3, num_seqs=256, lens=("uniform", 1, 90), partition_size=32),
    # shared prefix, copy-on-write of partial tail blocks
    "c5_prefix": dict(cfg=5, num_seqs=8, lens=("prefix", 64, 0, 40), partition_size=32),
}


@pytest.mark.parametrize("block_size", [8, 32, 64])
@pytest.mark.parametrize("case", sorted(CASES))
def test_block_size_step_matches_oracle(case, block_size):
    wl = P.make_workload(poison=True, block_size=block_size, **CASES[case])
    k, v, ref = oracle.apply_step(wl)
    ds = DeviceStep(wl)
    out = ds.step().cpu().numpy()
    assert ds.status_bits() == 0
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)
    assert np.all(np.isfinite(out))
    err = float(np.max(np.abs(out - ref)))
    assert err <= ATOL, err


@pytest.mark.parametrize("block_size", [8, 32, 64])
def test_block_size_fused_step_equals_write_then_attend(block_size):
    for case in ("c2_ps64", "c3_two_warps"):
        wl = P.make_workload(poison=True, block_size=block_size, **CASES[case])
        a, b = DeviceStep(wl), DeviceStep(wl)
        out_a = a.step().clone()
        out_b = b.fused_step().clone()
        assert a.status_bits() == 0 and b.status_bits() == 0
        assert torch.equal(out_a.view(torch.int32), out_b.view(torch.int32))
        assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))


@pytest.mark.parametrize("block_size", [8, 64])
def test_block_size_same_tokens_same_result(block_size):
    """The same sequences stored in 16-token blocks and in `block_size`-token
    blocks give outputs within rounding of each other (and each matches the
    oracle): the table, not the block size, decides what is read."""
    kw = dict(num_seqs=10, lens=("uniform", 20, 400), partition_size=64)
    wl16 = P.make_workload(2, poison=True, **kw)
    wlb = P.make_workload(2, poison=True, block_size=block_size, **kw)
    # identical lengths and values: rebuild wlb's pools from wl16's tokens
    assert np.array_equal(wl16.context_lens, wlb.context_lens)
    for pool16, poolb in ((wl16.k_pool, wlb.k_pool), (wl16.v_pool, wlb.v_pool)):
        for s, L in enumerate(wl16.context_lens.tolist()):
            for t in range(L - 1):  # history (the new token is written by the step)
                poolb[wlb.block_tables[s, t // block_size], t % block_size] = \
                    pool16[wl16.block_tables[s, t // 16], t % 16]
    wlb.q, wlb.k_new, wlb.v_new = wl16.q, wl16.k_new, wl16.v_new
    o16 = DeviceStep(wl16).step().cpu().numpy()
    ob = DeviceStep(wlb).step().cpu().numpy()
    assert float(np.max(np.abs(o16 - ob))) <= 1e-5


def test_block_size_all_layer_view():
    """32-token blocks in an all-layer pool: a layer's view has a block
    stride of layers x 32 rows."""
    wl = P.make_workload(2, poison=True, block_size=32, num_seqs=8, lens=("uniform", 1, 200), partition_size=64)
    L = 3
    ld = P.make_layers(wl, L)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    pool = dev(ld.pool)
    out = torch.empty((L,) + wl.q.shape, dtype=torch.float32, device="cuda")
    bt, cl, sm = (torch.from_numpy(x).cuda() for x in (wl.block_tables, wl.context_lens, wl.slot_mapping))
    nb = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.max_context_len, 64)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, kn, vn = dev(ld.q), dev(ld.k_new), dev(ld.v_new)
    for layer in range(L):
        pkv.decode_step(out[layer], q[layer], kn[layer], vn[layer], pool[0, :, layer], pool[1, :, layer], bt, cl, sm,
                        wl.scale, partition_size=64, max_context_len=wl.max_context_len, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    for layer in range(L):
        k, v = ld.pool[0, :, layer].copy(), ld.pool[1, :, layer].copy()
        oracle.write_cache(k, v, ld.k_new[layer], ld.v_new[layer], wl.slot_mapping)
        ref = oracle.decode_attention(ld.q[layer], k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
        assert np.array_equal(got[0, :, layer], k) and np.array_equal(got[1, :, layer], v)
        assert float(np.max(np.abs(out[layer].cpu().numpy() - ref))) <= ATOL
