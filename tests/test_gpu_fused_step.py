"""pkv_decode_step (the new token's write fused into decode attention) equals
pkv_write_cache followed by pkv_decode_attention, bit for bit, and the oracle
within 2e-3."""
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


CASES = [  # (recipe, overrides, partition size)
    (1, {}, 0),
    (1, {}, 16),
    (2, dict(num_seqs=10), 512),
    (2, dict(num_seqs=10, dtype="f16", num_q_heads=16, num_kv_heads=2), 64),
    (3, dict(num_seqs=24), 512),
    (3, dict(num_seqs=24), pkv.PARTITION_BALANCED),
    (2, dict(num_seqs=3, lens=("fixed", [1, 16, 17])), pkv.PARTITION_BALANCED),
    (5, dict(num_seqs=16, lens=("prefix", 64, 0, 70)), 32),
    (5, dict(num_seqs=16, lens=("prefix", 64, 0, 70)), pkv.PARTITION_BALANCED),
    # a grid of many waves (64 x 4 sequence-heads x 38 partitions): the head-group kernel with four
    # heads a CTA on a GB300; then the same with 32-token blocks (two tiles per block)
    (2, dict(num_seqs=64, num_q_heads=16, num_kv_heads=4, lens=("uniform", 300, 600)), 16),
    (2, dict(num_seqs=64, num_q_heads=16, num_kv_heads=4, lens=("uniform", 300, 600), block_size=32), 16),
]


@pytest.mark.parametrize("cfg,kw,ps", CASES)
def test_fused_step_equals_write_then_attend(cfg, kw, ps):
    wl = P.make_workload(cfg, poison=True, **kw)
    sep = DeviceStep(wl, partition_size=ps)
    ref_out = sep.step().clone()
    fused = DeviceStep(wl, partition_size=ps)
    out = fused.fused_step()
    assert fused.status_bits() == 0
    bits = lambda t: t.view(torch.int16)  # the pools hold NaN poison: compare bit patterns
    assert torch.equal(bits(fused.k_pool), bits(sep.k_pool)) and torch.equal(bits(fused.v_pool), bits(sep.v_pool))
    assert torch.equal(out, ref_out)
    k_ref, v_ref, ref = oracle.apply_step(wl)
    assert np.array_equal(to_bits(fused.k_pool), k_ref)
    assert float(np.max(np.abs(out.cpu().numpy() - ref))) <= ATOL


@pytest.mark.parametrize("ps", [512, pkv.PARTITION_BALANCED])
def test_fused_step_rejects_slots_not_at_the_end(ps):
    """A slot that is not position L-1 is flagged and not written; a -1 slot
    writes nothing.  Attention then reads the pool as it stands."""
    wl = P.make_workload(2, num_seqs=6)
    sm = wl.slot_mapping.copy()
    sm[1] = sm[1] - 1 if sm[1] % 16 else sm[1] + 1  # another slot of the same block
    sm[4] = -1
    ds = DeviceStep(wl, partition_size=ps)
    ds.slot_mapping = torch.from_numpy(sm).cuda()
    out = ds.fused_step().cpu().numpy()
    assert ds.status_bits() & pkv.DEV_ERR_SLOT
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    keep = np.ones(wl.num_seqs, bool)
    keep[[1, 4]] = False
    oracle.write_cache(k, v, wl.k_new[keep], wl.v_new[keep], wl.slot_mapping[keep])
    assert np.array_equal(to_bits(ds.k_pool), k) and np.array_equal(to_bits(ds.v_pool), v)
    ref = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert float(np.max(np.abs(out - ref))) <= ATOL
