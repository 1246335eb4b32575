"""Several host threads driving the library at once.

Each thread has its own CUDA stream and its own buffers and runs decode
steps (copy-on-write, fused write + attention, reduce) concurrently with the
others; ctypes releases the GIL for the duration of each C call, so the
library's host code (argument checks, tensor-map and occupancy caches) runs
in parallel.  The threads start together in a fresh process, so the caches
are filled concurrently as well.  Every thread's outputs and pools must match
the oracle."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import oracle, paged_kv_cache_112_gb300 as pkv, pkv_inputs as P
from tests.gpu_util import ATOL, DeviceStep, to_bits

torch.cuda.set_device(0)
pkv.load()
# (recipe, partition size): fixed partitions of two sizes and the balanced split
jobs = [(2, 512), (2, 64), (5, 1024), (3, pkv.PARTITION_BALANCED)]
wls = [P.make_workload(c, num_seqs=20, poison=True) for c, _ in jobs]
refs = [oracle.apply_step(wl) for wl in wls]
steps = [DeviceStep(wl, partition_size=ps) for wl, (_, ps) in zip(wls, jobs)]
start = threading.Barrier(len(jobs))
errors = []

def run(i):
    ds = steps[i]
    stream = torch.cuda.Stream()
    try:
        with torch.cuda.stream(stream):
            start.wait()
            for _ in range(25):
                ds.copy()
                pkv.decode_step(ds.out, ds.q, ds.k_new, ds.v_new, ds.k_pool, ds.v_pool, ds.block_tables,
                                ds.context_lens, ds.slot_mapping, ds.wl.scale, partition_size=ds.partition_size,
                                max_context_len=ds.max_context_len, workspace=ds.workspace, status=ds.status)
        stream.synchronize()
    except Exception as e:  # reported by the main thread
        errors.append((i, repr(e)))

threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
torch.cuda.synchronize()
for i, (ds, (k_ref, v_ref, ref)) in enumerate(zip(steps, refs)):
    assert int(ds.status.item()) == 0, (i, int(ds.status.item()))
    assert np.array_equal(to_bits(ds.k_pool), k_ref) and np.array_equal(to_bits(ds.v_pool), v_ref), i
    err = float(np.max(np.abs(ds.out.cpu().numpy().astype(np.float64) - ref)))
    assert err <= ATOL, (i, err)
print("threads ok")
"""


def test_four_host_threads_on_their_own_streams():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
