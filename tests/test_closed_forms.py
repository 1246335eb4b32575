"""The pages' printed sizing figures, recomputed from the oracle's closed forms."""
import os

import pytest

from oracle import sizing as Z
from pkv_inputs import BlockPool, SeqState, append_token

import numpy as np

KiB, MiB, GiB = 1024, 1024**2, 1024**3
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_closed_forms.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (x.strip() for x in line.split("="))
            vals[k] = float(v)
    return vals


G = _golden()


def test_per_token_bytes_70b_and_8b():
    assert Z.kv_bytes_per_token(80, 8, 128, 2) == G["kv_bytes_per_token_70b_fp16"] == 320 * KiB
    assert Z.kv_cache_bytes(80, 8, 128, 4096) / GiB == G["reservation_4k_70b_gib"]
    assert Z.kv_bytes_per_token(32, 8, 128, 2) == G["kv_bytes_per_token_8b_fp16"] == 128 * KiB


def test_8b_pool_arithmetic():
    per_block = Z.block_bytes(32, 8, 128, 2, 16)
    assert per_block == G["block_bytes_8b_fp16_b16"] == 2 * MiB
    blocks = Z.pool_blocks(54 * GiB, per_block)
    assert blocks == G["pool_blocks_8b_54gib"]
    assert blocks * 16 == G["pool_tokens_8b_54gib"]


def test_70b_block_slab():
    assert Z.block_bytes(80, 8, 128, 2, 16) / MiB == G["block_bytes_70b_fp16_b16_mib"]


@pytest.mark.parametrize("B", [8, 16, 32, 64, 128])
def test_expected_waste_300_tokens(B):
    w = Z.expected_internal_waste(B)
    assert w == G[f"waste_tokens_b{B}"]
    assert round(100 * w / 300, 1) == G[f"waste_pct_b{B}"]


def test_waste_bound_and_mean():
    for B in (8, 16, 32):
        ws = [Z.internal_waste_tokens(n, B) for n in range(1, 50 * B + 1)]
        assert max(ws) == B - 1 and min(ws) == 0
        # uniform over residues -> mean (B-1)/2
        assert np.mean(ws[: (len(ws) // B) * B]) == Z.expected_internal_waste(B)


def test_table_sizes_and_loop_counts():
    assert Z.blocks_for_tokens(300, 8) == G["table_entries_300_b8"]
    assert Z.blocks_for_tokens(300, 16) == G["table_entries_300_b16"]
    assert Z.blocks_for_tokens(300, 128) == G["table_entries_300_b128"]
    assert Z.blocks_for_tokens(4096, 16) == G["table_entries_4096_b16"]
    assert Z.table_bytes(4096, 16) == G["table_bytes_4096_b16"]
    assert Z.blocks_for_tokens(131072, 16) == G["table_entries_131072_b16"]
    assert Z.table_bytes(131072, 16) == G["table_bytes_131072_b16"]


def test_sharing_examples():
    per_tok = Z.kv_bytes_per_token(80, 8, 128, 2)
    assert round(4 * 2000 * per_tok / GiB, 2) == G["unshared_4x2000_70b_gib"]
    assert 2000 * per_tok / MiB == G["shared_2000_70b_mib"]
    assert Z.blocks_for_tokens(2000, 16) == G["prompt_blocks_2000_b16"]
    assert Z.shared_prefix_blocks(2050, 16) == G["shared_blocks_2050_b16"]
    assert 2050 - 16 * Z.shared_prefix_blocks(2050, 16) == 2
    assert round(500 * 3000 * per_tok / GiB) == G["unshared_500x3000_70b_gib"]
    nb = Z.blocks_for_tokens(3000, 16)
    assert nb == G["shared_3000_blocks_b16"]
    assert round(nb * Z.block_bytes(80, 8, 128, 2, 16) / GiB, 2) == G["shared_3000_70b_gib"]


def test_lattice_script_printout():
    one = Z.kv_cache_bytes(80, 8, 128, 8192, 1, 2) / GiB
    assert round(one, 2) == G["llama70b_8k_1seq_gib"]
    assert round(Z.kv_cache_bytes(80, 8, 128, 8192, 64, 2) / GiB, 2) == G["llama70b_8k_64users_gib"]
    assert round(Z.kv_cache_bytes(80, 64, 128, 8192, 1, 2) / GiB, 2) == G["llama70b_8k_64kvheads_gib"]


def test_fleet_waste_256_sequences():
    assert abs(256 * Z.expected_internal_waste(16) - G["waste_256_seqs_b16_approx"]) < 100


def test_worked_decode_example_300_tokens():
    """300-token prompt -> 19 blocks; token 301 lands in logical block 18, no new block."""
    bm = BlockPool(64, np.random.default_rng(0))
    seq = SeqState()
    for _ in range(300):
        append_token(bm, seq)
    assert len(seq.table) == G["prompt_300_blocks_b16"]
    before = list(seq.table)
    slot, pair = append_token(bm, seq)
    assert pair is None and seq.table == before  # no new block
    logical = 300 // 16
    assert logical == G["token_301_logical_block"]
    assert (logical * 16, logical * 16 + 15) == (G["token_301_block_first"], G["token_301_block_last"])
    assert slot == seq.table[logical] * 16 + 300 % 16
    # every 16 steps one fresh block: 3 more appends fill block 18, the 4th opens block 19
    for _ in range(3):
        append_token(bm, seq)
    assert len(seq.table) == 19
    append_token(bm, seq)
    assert len(seq.table) == 20
