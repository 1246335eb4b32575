"""bench.py's algorithmic byte counts agree with the workload's own (CPU only)."""
import numpy as np

import bench
import pkv_inputs as P


def test_step_bytes_16bit_and_fp8():
    wl = P.make_workload(1)
    nb = bench.step_bytes(wl)
    assert nb["kv"] == wl.kv_bytes_read()
    f8 = P.make_fp8_pools(wl)
    nb8 = bench.step_bytes_fp8(wl)
    assert nb8["kv"] == f8.kv_bytes_read(wl)
    blocks = int(np.sum((wl.context_lens.astype(np.int64) + 15) // 16))
    # one byte per element instead of two, plus a K and a V scale per (table entry, KV head)
    assert nb8["kv"] == nb["kv"] // 2 + blocks * wl.num_kv_heads * 8
    T = wl.slot_mapping.shape[0]
    assert nb8["write"] == 2 * T * wl.num_kv_heads * wl.head_dim * 3 + T * wl.num_kv_heads * 8 + T * 4
    for d in (nb, nb8):
        assert d["step"] == d["attention"] + d["write"] + d["copy"]


def test_kernel_source_hash_ignores_comments_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  // store\n}\n/* block */\n")
    h0 = bench.kernel_source_hash([str(a)])
    a.write_text("// a different header\n__global__ void k(int* p) {\n    p[0] = 1;\n}\n")
    assert bench.kernel_source_hash([str(a)]) == h0
    a.write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n")
    assert bench.kernel_source_hash([str(a)]) != h0


def test_write_and_copy_bytes_count_rows_and_blocks():
    # one token of the 8B-class row (8 KV heads x 128): K and V rows read (2 B) and written (2 B), one slot
    assert bench.write_bytes(1, 8, 128) == 2 * 1024 * 4 + 4
    # FP8: rows read (2 B), codes written (1 B), the K and V scale of each KV head, one slot
    assert bench.write_bytes(1, 8, 128, fp8=True) == 2 * 1024 * 3 + 8 * 8 + 4
    # one pair of 16-token blocks: K and V block read and written, the pair read
    assert bench.copy_bytes(1, 16, 8, 128) == 2 * 16 * 1024 * 2 * 2 + 8
    assert bench.copy_bytes(1, 16, 8, 128, fp8=True) == 2 * (16 * 1024 + 32) * 2 + 8
    wl = P.make_workload(5, num_seqs=8, lens=("prefix", 64, 0, 40))
    assert wl.copy_pairs.shape[0] > 0
    nb = bench.step_bytes(wl)
    assert nb["copy"] == bench.copy_bytes(wl.copy_pairs.shape[0], 16, wl.num_kv_heads, wl.head_dim)


def test_cache_op_sets_are_disjoint_whole_blocks():
    rng = np.random.default_rng(0)
    slots, nb = bench.cache_op_sets("write", 40, 16, 5, rng)
    assert slots.shape == (5, 40) and slots.dtype == np.int32 and nb == 5 * 3
    assert len(np.unique(slots)) == slots.size and slots.min() >= 0 and slots.max() < nb * 16
    for r in range(5):
        # tokens fill their blocks in order: offset t % 16 within block t // 16 of the set
        assert np.array_equal(slots[r] % 16, np.arange(40) % 16)
        blocks = slots[r] // 16
        assert np.all(blocks[np.arange(40) // 16 * 16] == blocks)
    pairs, nb = bench.cache_op_sets("copy", 7, 16, 4, rng)
    assert pairs.shape == (4, 7, 2) and pairs.dtype == np.int32 and nb == 4 * 2 * 7
    assert len(np.unique(pairs)) == pairs.size and pairs.min() >= 0 and pairs.max() < nb


def test_reference_arm_prints_one_contract_line(capsys):
    """`bench.py --impl reference` (the fp64 oracle on host cores) prints one
    JSON line with the contract's keys, on the same workload description as
    the CUDA arm."""
    import json

    bench.main(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3", "--ref-seconds", "0.5"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True and line["steps"] == 2 and line["warmup"] == 3
    wl = P.make_workload(1)
    assert {k: line["config"][k] for k in bench.workload_config(wl)} == bench.workload_config(wl)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_unique_bytes_count_a_shared_prefix_once():
    """Prefix-sharing recipe: every sequence reads the same 2048-token prefix
    blocks; the distinct slots are the prefix once plus each private suffix
    (copy-on-write tails land in fresh blocks, so they are distinct too)."""
    wl = P.make_workload(5, num_seqs=24)
    L = wl.context_lens.astype(np.int64)
    row = wl.num_kv_heads * wl.head_dim * 2 * 2
    assert bench.unique_kv_bytes(wl) == (2048 + int((L - 2048).sum())) * row
    wl2 = P.make_workload(2, num_seqs=8)  # no sharing: unique == logical
    assert bench.unique_kv_bytes(wl2) == bench.step_bytes(wl2)["kv"]


def test_unique_bytes_fp8_count_codes_and_block_scales_once():
    """FP8 pools: one byte per element, plus a K and a V scale per KV head of
    each distinct block.  Without sharing this is the step's own K/V count."""
    wl = P.make_workload(5, num_seqs=24)
    L = wl.context_lens.astype(np.int64)
    hd = wl.num_kv_heads * wl.head_dim
    blocks = 2048 // 16 + int(np.sum((L - 2048 + 15) // 16))  # prefix blocks once, then each private tail
    assert bench.unique_kv_bytes(wl, 1, 4) == (2048 + int((L - 2048).sum())) * hd * 2 + blocks * wl.num_kv_heads * 8
    wl2 = P.make_workload(2, num_seqs=8)
    assert bench.unique_kv_bytes(wl2, 1, 4) == bench.step_bytes_fp8(wl2)["kv"]


def test_graph_blocks_time_exactly_k_steps():
    for K in (1, 3, 5, 20, 21, 64, 5000, 4999):
        for R in (1, 2, 3):
            b, full, rem = bench.graph_blocks(K, R)
            assert b * full + rem == K and b % R == 0 and b >= 1
            assert rem < b


def test_partition_kernel_names_follow_the_library_rule():
    """The bench names the kernel a recipe runs (its roofline and traffic
    record are that kernel's): on 152 SMs the 70B-class layer overfills one
    wave of warp slots and keeps the per-head kernel, the others run the
    head-group kernel; FP8 write-then-attend runs the FP8 head-group grid."""
    name = bench.partition_kernel_name
    for cfg, expect in ((2, "decode_partitions_hg_kernel"), (3, "decode_partitions_kernel"),
                        (4, "decode_partitions_hg_kernel"), (5, "decode_partitions_hg_kernel")):
        spec = P.CONFIGS[cfg]
        assert name(spec["num_seqs"], spec["num_kv_heads"], spec["partition_size"], 16, False, True, 152) == expect
        assert name(spec["num_seqs"], spec["num_kv_heads"], P.fp8_partition_size(cfg), 16, True, False, 152) == \
            "decode_partitions_fp8_hg_kernel"
        assert name(spec["num_seqs"], spec["num_kv_heads"], P.fp8_partition_size(cfg), 16, True, True, 152) == \
            "decode_partitions_fp8_kernel"
    assert name(64, 8, -1, 16, False, True, 152) == "decode_balanced_kernel"
    assert name(64, 8, -1, 16, True, False, 152) == "decode_balanced_fp8_kernel"
    assert name(64, 8, 512, 8, False, True, 152) == "decode_partitions_kernel"  # 8-token blocks
    assert name(64, 3, 512, 16, False, True, 152) == "decode_partitions_kernel"  # odd H_kv
