"""The oracle checked against things other than itself (CPU only)."""
import numpy as np
import pytest

import oracle
import pkv_inputs as P
from tests import oracle_pins as pins


def _oracle_attn(q, kp, vp, bt, cl, scale, dtype):
    return oracle.decode_attention(q, kp, vp, bt, cl, scale, dtype)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(_oracle_attn)


def test_sampled_rows_match_full():
    wl = P.make_workload(1, poison=True)
    k, v, full = oracle.apply_step(wl)
    rows = [(3, 1), (0, 0), (2, 3)]
    part = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, rows=rows)
    for i, (s, h) in enumerate(rows):
        assert np.array_equal(part[i], full[s, h])


def test_thread_count_does_not_change_result():
    wl = P.make_workload(1)
    k, v, _ = oracle.apply_step(wl, attention=False)
    a = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, num_threads=1)
    b = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype, num_threads=7)
    assert np.array_equal(a, b)


def test_oracle_rejects_out_of_range_table():
    wl = P.make_workload(1)
    bt = wl.block_tables.copy()
    bt[3, 1] = wl.num_blocks  # one past the pool
    with pytest.raises(ValueError):
        oracle.decode_attention(wl.q, wl.k_pool, wl.v_pool, bt, wl.context_lens, wl.scale, wl.dtype)


def test_zero_length_sequence_gives_zeros():
    wl = P.make_workload(1)
    cl = wl.context_lens.copy()
    cl[0] = 0
    out = oracle.decode_attention(wl.q, wl.k_pool, wl.v_pool, wl.block_tables, cl, wl.scale, wl.dtype)
    assert np.all(out[0] == 0.0)


def test_write_cache_places_rows_at_slot():
    """slot = block * B + offset: the row lands in that block at that offset, nothing else moves."""
    wl = P.make_workload(1, poison=True)
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.write_cache(k, v, wl.k_new, wl.v_new, wl.slot_mapping)
    changed = np.argwhere(np.any(k != wl.k_pool, axis=(2, 3)))
    assert sorted(map(tuple, changed.tolist())) == sorted((s // 16, s % 16) for s in wl.slot_mapping.tolist())
    for i, slot in enumerate(wl.slot_mapping.tolist()):
        assert np.array_equal(k[slot // 16, slot % 16], wl.k_new[i])
        assert np.array_equal(v[slot // 16, slot % 16], wl.v_new[i])
    # the written slot is position L-1 of its sequence, reached through the table
    for s, L in enumerate(wl.context_lens.tolist()):
        t = L - 1
        assert wl.slot_mapping[s] == wl.block_tables[s, t // 16] * 16 + t % 16


def test_write_cache_skips_negative_slots():
    wl = P.make_workload(1)
    k, v = wl.k_pool.copy(), wl.v_pool.copy()
    sm = wl.slot_mapping.copy()
    sm[1] = -1
    oracle.write_cache(k, v, wl.k_new, wl.v_new, sm)
    s1 = wl.slot_mapping[1]
    assert np.array_equal(k[s1 // 16, s1 % 16], wl.k_pool[s1 // 16, s1 % 16])


def test_copy_on_write_recipe():
    """Prefix-sharing recipe (small): the CoW copy gives each forking sequence a
    private tail identical to the parent's; shared blocks stay untouched."""
    wl = P.make_workload(5, num_seqs=12, lens=("prefix", 64, 0, 40), poison=True)
    assert len(wl.copy_pairs) > 0
    k, v, _ = oracle.apply_step(wl, attention=False)
    kc, vc = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.copy_blocks(kc, vc, wl.copy_pairs)
    for src, dst in wl.copy_pairs.tolist():
        assert kc[dst].tobytes() == wl.k_pool[src].tobytes()
        assert vc[dst].tobytes() == wl.v_pool[src].tobytes()
    prot = wl.protected_blocks
    assert np.array_equal(k[prot].view(np.uint16), wl.k_pool[prot].view(np.uint16))
    assert np.array_equal(v[prot].view(np.uint16), wl.v_pool[prot].view(np.uint16))
    # shared prefix referenced by every table, refcount = number of sequences
    for b in wl.block_tables[0, :4].tolist():
        assert wl.refcount[b] == 12
        assert np.all(wl.block_tables[:, :4] == wl.block_tables[0, :4])
    # NaN-poisoned tails and unused blocks never reach the output of the real recipe
    out = oracle.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert np.all(np.isfinite(out))


def test_generator_recipes_shapes():
    for cfg in (1,):
        wl = P.make_workload(cfg)
        assert wl.k_pool.shape == (wl.num_blocks, 16, wl.num_kv_heads, wl.head_dim)
        assert wl.block_tables.shape[1] == -(-wl.max_context_len // 16)
    wl = P.make_workload(2, num_seqs=5)
    assert wl.context_lens.min() >= 128 and wl.context_lens.max() <= 2048
    # distinct physical blocks across all tables (no sharing in this recipe)
    used = wl.block_tables[wl.block_tables >= 0]
    assert len(np.unique(used)) == len(used)
    # internal waste bounded by B-1 per sequence
    cap = (wl.block_tables >= 0).sum(axis=1) * 16
    assert np.all(cap - wl.context_lens <= 15) and np.all(cap >= wl.context_lens)
