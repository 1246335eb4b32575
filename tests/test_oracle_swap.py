"""The swap oracle (block lists moved between a device pool and a host pool)
checked against what swapping must do, without a GPU: the listed blocks move
byte for byte, nothing else changes, a swap out followed by a swap in to other
blocks restores every byte, and a sequence whose table is repointed to the
swapped-in blocks attends exactly as before ("gpu_paged_kv_cache",
"Reclaiming memory: swap versus recompute"; "PagedAttention internals",
section 05)."""
import numpy as np
import pytest

import oracle
import pkv_inputs as P


def _pool(n, rng, shape=(16, 2, 64)):
    return rng.integers(0, 2 ** 16, size=(n,) + shape, dtype=np.uint16)


def test_listed_blocks_move_and_nothing_else():
    rng = np.random.default_rng(1)
    dk, dv = _pool(10, rng), _pool(10, rng)
    hk, hv = _pool(6, rng), _pool(6, rng)
    hk0, hv0 = hk.copy(), hv.copy()
    pairs = np.array([[7, 0], [2, 5], [9, 3]], dtype=np.int32)  # (device block, host slot)
    oracle.swap_blocks(hk, hv, dk, dv, pairs)
    for s, d in pairs.tolist():
        assert np.array_equal(hk[d], dk[s]) and np.array_equal(hv[d], dv[s])
    untouched = [i for i in range(6) if i not in pairs[:, 1]]
    assert np.array_equal(hk[untouched], hk0[untouched]) and np.array_equal(hv[untouched], hv0[untouched])


def test_round_trip_to_other_blocks_restores_every_byte():
    rng = np.random.default_rng(2)
    dk, dv = _pool(12, rng), _pool(12, rng)
    orig = dk.copy(), dv.copy()
    victim = np.array([4, 0, 9, 11], dtype=np.int32)
    hk, hv = np.zeros((4,) + dk.shape[1:], np.uint16), np.zeros((4,) + dv.shape[1:], np.uint16)
    oracle.swap_blocks(hk, hv, dk, dv, np.stack([victim, np.arange(4)], 1))
    dk[victim] = 0xFFFF  # freed and reused by someone else
    dv[victim] = 0xFFFF
    target = np.array([1, 5, 6, 2], dtype=np.int32)
    oracle.swap_blocks(dk, dv, hk, hv, np.stack([np.arange(4), target], 1))
    for i in range(4):
        assert np.array_equal(dk[target[i]], orig[0][victim[i]]) and np.array_equal(dv[target[i]], orig[1][victim[i]])


@pytest.mark.parametrize("cfg", [1])
def test_swapped_in_sequence_attends_as_before(cfg):
    wl = P.make_workload(cfg, poison=True)
    k, v, before = oracle.apply_step(wl)
    s = int(np.argmax(wl.context_lens))
    nblk = -(-int(wl.context_lens[s]) // 16)
    blocks = wl.block_tables[s, :nblk].copy()
    hk = np.zeros((nblk,) + k.shape[1:], np.uint16)
    hv = np.zeros_like(hk)
    oracle.swap_blocks(hk, hv, k, v, np.stack([blocks, np.arange(nblk)], 1))
    k[blocks] = P.NAN_BITS[wl.dtype]  # freed
    v[blocks] = P.NAN_BITS[wl.dtype]
    used = set(wl.block_tables[wl.block_tables >= 0].tolist())
    free = np.array([b for b in range(wl.num_blocks) if b not in used][:nblk], dtype=np.int32)
    oracle.swap_blocks(k, v, hk, hv, np.stack([np.arange(nblk), free], 1))
    bt = wl.block_tables.copy()
    bt[s, :nblk] = free
    after = oracle.decode_attention(wl.q, k, v, bt, wl.context_lens, wl.scale, wl.dtype)
    assert np.array_equal(after, before)
