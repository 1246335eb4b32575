"""FP8 pools in the all-layer layout: codes [NB, layers, 16, H_kv, D] and
scales [NB, layers, H_kv], every layer of a block (and its scales) together
("KV Cache & PagedAttention" section 4; "gpu_paged_kv_cache", "Blocks as
quantization groups": a block's scales move with it).  Copy-on-write moves a
block's codes and scales of every layer at once; the write and the decode
take one layer's views.  Each layer is checked against the oracle run on that
layer's own one-layer pools."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def _layers(wl, L):
    ld = P.make_layers(wl, L)
    pools = [P.make_fp8_pools(wl, seed=100 + layer) for layer in range(L)]
    k8 = np.ascontiguousarray(np.stack([p.k8 for p in pools], 1))
    v8 = np.ascontiguousarray(np.stack([p.v8 for p in pools], 1))
    ks = np.ascontiguousarray(np.stack([p.k_scale for p in pools], 1))
    vs = np.ascontiguousarray(np.stack([p.v_scale for p in pools], 1))
    return ld, pools, k8, v8, ks, vs


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", ["prefix_cow", "uniform"])
def test_fp8_all_layer_step_matches_oracle(case, fused):
    if case == "prefix_cow":
        wl = P.make_workload(5, poison=True, num_seqs=8, lens=("prefix", 64, 0, 40), partition_size=32)
    else:
        wl = P.make_workload(2, poison=True, num_seqs=12, lens=("uniform", 1, 300), partition_size=64)
    L = 3
    ld, pools, k8, v8, ks, vs = _layers(wl, L)
    dk, dv = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    dks, dvs = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    bt, cl, sm = (torch.from_numpy(x).cuda() for x in (wl.block_tables, wl.context_lens, wl.slot_mapping))
    pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, dtype=np.int32)).cuda()
    q, kn, vn = (to_dev(x, wl.dtype) for x in (ld.q, ld.k_new, ld.v_new))
    out = torch.empty((L,) + wl.q.shape, dtype=torch.float32, device="cuda")
    nb = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.max_context_len,
                                    wl.partition_size)
    ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if pairs.shape[0]:
        pkv.copy_blocks_fp8(dk, dv, dks, dvs, pairs, status=status)  # every layer at once
    for layer in range(L):
        kw = dict(partition_size=wl.partition_size, max_context_len=wl.max_context_len, workspace=ws, status=status)
        views = (dk[:, layer], dv[:, layer], dks[:, layer], dvs[:, layer])
        if fused:
            pkv.decode_step_fp8(out[layer], q[layer], kn[layer], vn[layer], *views, bt, cl, sm, wl.scale, **kw)
        else:
            pkv.write_cache_fp8(kn[layer], vn[layer], *views, sm, status=status)
            pkv.decode_attention_fp8(out[layer], q[layer], *views, bt, cl, wl.scale, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_k, got_v, got_ks, got_vs = (t.cpu().numpy() for t in (dk, dv, dks, dvs))
    for layer in range(L):
        wl_l = dataclasses.replace(wl, q=ld.q[layer], k_new=ld.k_new[layer], v_new=ld.v_new[layer])
        rk, rv, rks, rvs, ref = oracle.apply_step_fp8(wl_l, pools[layer])
        assert np.array_equal(got_k[:, layer], rk) and np.array_equal(got_v[:, layer], rv), layer
        assert np.array_equal(got_ks[:, layer], rks, equal_nan=True), layer
        assert np.array_equal(got_vs[:, layer], rvs, equal_nan=True), layer
        err = float(np.max(np.abs(out[layer].cpu().numpy() - ref)))
        assert err <= ATOL, (layer, err)


def test_fp8_layer_views_are_validated():
    """A scale view whose layer count disagrees with the pool's is refused
    before any launch."""
    k = torch.zeros((4, 2, 16, 2, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones((4, 3, 2), dtype=torch.float32, device="cuda")
    kn = torch.zeros((1, 2, 128), dtype=torch.float16, device="cuda")
    sm = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.write_cache_fp8(kn, kn, k[:, 0], k[:, 0], s[:, 0], s[:, 0], sm)
    with pytest.raises(pkv.PkvError):
        pkv.copy_blocks_fp8(k, k, s, s, torch.zeros((1, 2), dtype=torch.int32, device="cuda"))
