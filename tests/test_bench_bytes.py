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
