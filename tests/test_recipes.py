"""The seeded workload recipes have the shapes the design states (CPU only):
pool sizes 1.25x the blocks needed, length ranges, and for the
prefix-sharing recipe a 2048-token prompt shared by every sequence with
114 copy-on-write pairs at its seed.  Copy sources are shared tails and
copy destinations fresh blocks that no table held before the step
("PagedAttention internals", section 03: copy-on-write always targets a
fresh block)."""
import numpy as np

import pkv_inputs as P


def test_8b_class_and_70b_class_recipes():
    wl = P.make_workload(2)
    L = wl.context_lens
    assert wl.num_blocks == 5779 and wl.num_seqs == 64 and wl.copy_pairs.shape[0] == 0
    assert L.min() >= 128 and L.max() <= 2048
    need = int(np.sum(-(-L.astype(np.int64) // 16)))
    assert wl.num_blocks == int(np.ceil(1.25 * need))
    wl = P.make_workload(3)
    L = wl.context_lens
    assert wl.num_blocks == 10242 and wl.num_seqs == 256
    assert L.min() >= 1 and L.max() == 4096  # the lognormal's cap is reached at this seed
    assert 250 <= int(np.median(L)) <= 350  # median 300 by construction


def test_prefix_sharing_recipe():
    wl = P.make_workload(5)
    L = wl.context_lens
    assert wl.num_blocks == 2894 and wl.num_seqs == 128
    assert L.min() >= 2049 and L.max() <= 2561  # 2048 shared + U[0, 512] private + the new token
    prompt = wl.block_tables[:, :128]
    assert np.all(prompt == prompt[0])  # every sequence shares the prompt's 128 blocks
    pairs = wl.copy_pairs
    assert pairs.shape == (114, 2)
    src, dst = pairs[:, 0], pairs[:, 1]
    assert len(np.unique(dst)) == len(dst) and not set(dst) & set(src)
    # each copied tail is the block before the append of a sequence whose private suffix ends
    # mid-block; after the step the table holds the destination at that position
    for s_blk, d_blk in pairs:
        rows, cols = np.nonzero(wl.block_tables == d_blk)
        assert len(rows) == 1
        s = rows[0]
        assert cols[0] == (int(L[s]) - 1) // 16 and (int(L[s]) - 1) % 16 != 0
        assert s_blk in wl.protected_blocks
