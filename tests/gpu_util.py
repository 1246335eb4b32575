"""Moves pkv_inputs workloads onto the GPU and runs one decode step through
the library's C ABI (helpers for the gpu-marked tests)."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_112_gb300 as pkv

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
ATOL = 2e-3  # max-abs error bound on the fp32 attention output vs the fp64 oracle


def to_dev(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DT[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceStep:
    """Device copies of one workload plus output, workspace and status word."""

    def __init__(self, wl, partition_size=None, out_dtype=torch.float32, device="cuda"):
        self.wl = wl
        dt = wl.dtype
        self.q = to_dev(wl.q, dt, device)
        self.k_pool = to_dev(wl.k_pool, dt, device)
        self.v_pool = to_dev(wl.v_pool, dt, device)
        self.k_new = to_dev(wl.k_new, dt, device)
        self.v_new = to_dev(wl.v_new, dt, device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.context_lens = torch.from_numpy(wl.context_lens).to(device)
        self.slot_mapping = torch.from_numpy(wl.slot_mapping).to(device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, dtype=np.int32)).to(device)
        self.partition_size = wl.partition_size if partition_size is None else partition_size
        self.max_context_len = wl.max_context_len
        self.out = torch.empty(wl.q.shape, dtype=out_dtype, device=device)
        nbytes = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, self.max_context_len,
                                            self.partition_size)
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device) if nbytes else None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def copy(self):
        if self.pairs.shape[0]:
            pkv.copy_blocks(self.k_pool, self.v_pool, self.pairs, status=self.status)

    def write(self):
        pkv.write_cache(self.k_new, self.v_new, self.k_pool, self.v_pool, self.slot_mapping, status=self.status)

    def attend(self, out=None):
        pkv.decode_attention(self.out if out is None else out, self.q, self.k_pool, self.v_pool,
                             self.block_tables, self.context_lens, self.wl.scale,
                             partition_size=self.partition_size, max_context_len=self.max_context_len,
                             workspace=self.workspace, status=self.status)

    def step(self):
        self.copy()
        self.write()
        self.attend()
        torch.cuda.synchronize()
        return self.out

    def fused_step(self, out=None):
        """copy_blocks, then the write fused into decode attention (pkv_decode_step)."""
        self.copy()
        pkv.decode_step(self.out if out is None else out, self.q, self.k_new, self.v_new, self.k_pool, self.v_pool,
                        self.block_tables, self.context_lens, self.slot_mapping, self.wl.scale,
                        partition_size=self.partition_size, max_context_len=self.max_context_len,
                        workspace=self.workspace, status=self.status)
        torch.cuda.synchronize()
        return self.out if out is None else out

    def status_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.status.item())


class DeviceStepFp8:
    """Device copies of one workload over FP8 pools (pkv_inputs.Fp8Pools)."""

    def __init__(self, wl, pools, partition_size=None, out_dtype=torch.float32, device="cuda"):
        self.wl = wl
        dt = wl.dtype
        self.q = to_dev(wl.q, dt, device)
        self.k_new = to_dev(wl.k_new, dt, device)
        self.v_new = to_dev(wl.v_new, dt, device)
        self.k8 = torch.from_numpy(pools.k8).to(device)
        self.v8 = torch.from_numpy(pools.v8).to(device)
        self.k_scale = torch.from_numpy(pools.k_scale).to(device)
        self.v_scale = torch.from_numpy(pools.v_scale).to(device)
        self.block_tables = torch.from_numpy(wl.block_tables).to(device)
        self.context_lens = torch.from_numpy(wl.context_lens).to(device)
        self.slot_mapping = torch.from_numpy(wl.slot_mapping).to(device)
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, dtype=np.int32)).to(device)
        self.partition_size = wl.partition_size if partition_size is None else partition_size
        self.max_context_len = wl.max_context_len
        self.out = torch.empty(wl.q.shape, dtype=out_dtype, device=device)
        self.set_workspace(self.max_context_len)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def set_workspace(self, max_context_len):
        self.max_context_len = max_context_len
        wl = self.wl
        nbytes = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, max_context_len,
                                            self.partition_size)
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=self.q.device) if nbytes else None

    def copy(self):
        if self.pairs.shape[0]:
            pkv.copy_blocks_fp8(self.k8, self.v8, self.k_scale, self.v_scale, self.pairs, status=self.status)

    def write(self):
        pkv.write_cache_fp8(self.k_new, self.v_new, self.k8, self.v8, self.k_scale, self.v_scale,
                            self.slot_mapping, status=self.status)

    def attend(self, out=None):
        pkv.decode_attention_fp8(self.out if out is None else out, self.q, self.k8, self.v8, self.k_scale,
                                 self.v_scale, self.block_tables, self.context_lens, self.wl.scale,
                                 partition_size=self.partition_size, max_context_len=self.max_context_len,
                                 workspace=self.workspace, status=self.status)

    def step(self):
        self.copy()
        self.write()
        self.attend()
        torch.cuda.synchronize()
        return self.out

    def fused_step(self, out=None):
        """copy_blocks_fp8, then the quantising write fused into attention (pkv_decode_step_fp8)."""
        self.copy()
        pkv.decode_step_fp8(self.out if out is None else out, self.q, self.k_new, self.v_new, self.k8, self.v8,
                            self.k_scale, self.v_scale, self.block_tables, self.context_lens, self.slot_mapping,
                            self.wl.scale, partition_size=self.partition_size, max_context_len=self.max_context_len,
                            workspace=self.workspace, status=self.status)
        torch.cuda.synchronize()
        return self.out if out is None else out

    def status_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.status.item())
