"""A small serving loop on the GPU driven by the native block manager: prompt
admission with prefix-cache hits (the cached tokens are not written again),
the prefill's bulk write, a fork for parallel sampling, decode steps with
copy-on-write pairs fed to pkv_copy_blocks and the fused write + attention,
and a swap out / in through pinned host memory.  A token's K/V rows are a
function of its whole history, so identical prefixes hold identical bytes
("PagedAttention internals", section 04: equal token prefixes give equal K
and V); every output is checked against the oracle on the
sequence's contiguous history."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL

pytestmark = pytest.mark.gpu

B, NB, HQ, HKV, D, DT = 16, 96, 8, 2, 128, "f16"
SCALE = 1 / np.sqrt(D)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def kv_row(history):
    """K and V rows [H_kv, D] (f16 bits) of the last token of `history`."""
    rng = np.random.default_rng(zlib.crc32(np.asarray(history, np.int32).tobytes()))
    x = rng.standard_normal((2, HKV, D)).astype(np.float32)
    return P.f32_to_bits(x[0], DT), P.f32_to_bits(x[1], DT)


def rows_for(tokens, positions):
    ks, vs = zip(*(kv_row(tokens[: p + 1]) for p in positions)) if positions else ((), ())
    return np.stack(ks) if ks else np.zeros((0, HKV, D), np.uint16), np.stack(vs) if vs else np.zeros((0, HKV, D), np.uint16)


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


class Loop:
    def __init__(self):
        self.bm = pkv.BlockManager(NB, B)
        # unwritten slots hold NaN, so a slot read before it is written would show
        self.k = torch.full((NB, B, HKV, D), P.NAN_BITS[DT], dtype=torch.int16, device="cuda").view(torch.float16)
        self.v = self.k.clone()
        self.tokens = {}
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def admit(self, sid, tokens, extra=0):
        cached, slots = self.bm.add_sequence(sid, tokens, extra)
        todo = [t for t in range(len(tokens)) if slots[t] >= 0]
        k, v = rows_for(tokens, todo)
        if todo:
            pkv.write_cache(dev16(k), dev16(v), self.k, self.v, torch.from_numpy(slots[todo]).cuda(),
                            status=self.status)
        self.tokens[sid] = list(tokens)
        return cached

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])

    def decode(self, rng, sids):
        """One decode step of `sids`: append a token each, copy-on-write,
        fused write + attention; returns {sid: output [H_q, D]}."""
        slots, pairs, knew, vnew = [], [], [], []
        for sid in sids:
            tok = int(rng.integers(0, 1000))
            slot, cow = self.bm.append(sid, tok)
            self.tokens[sid].append(tok)
            slots.append(slot)
            if cow:
                pairs.append(cow)
            k, v = kv_row(self.tokens[sid])
            knew.append(k)
            vnew.append(v)
        if pairs:
            pkv.copy_blocks(self.k, self.v, torch.tensor(pairs, dtype=torch.int32).cuda(), status=self.status)
        tables = [self.bm.block_table(sid) for sid in sids]
        width = max(len(t) for t in tables)
        bt = np.full((len(sids), width), -1, np.int32)
        for i, t in enumerate(tables):
            bt[i, : len(t)] = t
        cl = np.array([self.bm.seq_len(s) for s in sids], np.int32)
        q = P.f32_to_bits(rng.standard_normal((len(sids), HQ, D)).astype(np.float32), DT)
        out = torch.empty((len(sids), HQ, D), dtype=torch.float32, device="cuda")
        ps = 32
        nb = pkv.decode_workspace_bytes(len(sids), HQ, D, int(cl.max()), ps)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
        pkv.decode_step(out, dev16(q), dev16(np.stack(knew)), dev16(np.stack(vnew)), self.k, self.v,
                        torch.from_numpy(bt).cuda(), torch.from_numpy(cl).cuda(),
                        torch.tensor(slots, dtype=torch.int32).cuda(), SCALE, partition_size=ps,
                        max_context_len=int(cl.max()), workspace=ws, status=self.status)
        return self._check(sids, q, out)

    def decode_batch(self, rng, sids):
        """The same step with the whole batch's bookkeeping in one call
        (pkv_bm_decode_step: slots, lengths, padded tables and copy pairs)."""
        toks = [int(x) for x in rng.integers(0, 1000, size=len(sids))]
        width = max(-(-(self.bm.seq_len(s) + 1) // B) for s in sids)
        slots, cl, bt, pairs = self.bm.decode_step(sids, toks, width)
        knew, vnew = [], []
        for sid, tok in zip(sids, toks):
            self.tokens[sid].append(tok)
            k, v = kv_row(self.tokens[sid])
            knew.append(k)
            vnew.append(v)
        if len(pairs):
            pkv.copy_blocks(self.k, self.v, torch.from_numpy(np.ascontiguousarray(pairs, np.int32)).cuda(),
                            status=self.status)
        q = P.f32_to_bits(rng.standard_normal((len(sids), HQ, D)).astype(np.float32), DT)
        out = torch.empty((len(sids), HQ, D), dtype=torch.float32, device="cuda")
        ps = 32
        nb = pkv.decode_workspace_bytes(len(sids), HQ, D, int(cl.max()), ps)
        ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")
        pkv.decode_step(out, dev16(q), dev16(np.stack(knew)), dev16(np.stack(vnew)), self.k, self.v,
                        torch.from_numpy(np.ascontiguousarray(bt)).cuda(), torch.from_numpy(cl).cuda(),
                        torch.from_numpy(slots).cuda(), SCALE, partition_size=ps, max_context_len=int(cl.max()),
                        workspace=ws, status=self.status)
        return self._check(sids, q, out)

    def _check(self, sids, q, out):
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0
        got = out.cpu().numpy()
        for i, sid in enumerate(sids):
            toks = self.tokens[sid]
            k, v = rows_for(toks, list(range(len(toks))))
            n = -(-len(toks) // B)
            kp = np.full((n, B, HKV, D), P.NAN_BITS[DT], np.uint16)
            vp = kp.copy()
            kp.reshape(-1, HKV, D)[: len(toks)] = k
            vp.reshape(-1, HKV, D)[: len(toks)] = v
            ref = oracle.decode_attention(q[i:i + 1], kp, vp, np.arange(n, dtype=np.int32).reshape(1, n),
                                          np.array([len(toks)], np.int32), SCALE, DT)
            assert float(np.max(np.abs(got[i] - ref[0]))) <= ATOL, sid
        return got


def test_serving_loop_with_prefix_cache_fork_cow_and_swap():
    rng = np.random.default_rng(2024)
    loop = Loop()
    system = [int(x) for x in rng.integers(0, 1000, size=2 * B + 3)]  # 2 whole blocks + 3 tokens
    assert loop.admit(1, system + [7, 8, 9, 10]) == 0
    assert loop.admit(2, system + [11] * 20) == 2 * B  # the system prompt's whole blocks are shared
    assert loop.admit(3, system + [7, 8, 9, 10], extra=5) == 0  # another adapter: its own blocks
    shared = loop.bm.block_table(1)[:2]
    assert np.array_equal(loop.bm.block_table(2)[:2], shared)
    assert loop.bm.refcount(int(shared[0])) == 2
    loop.fork(1, 4)  # parallel sample: shares every block, tail included
    for _ in range(3):
        loop.decode(rng, [1, 2, 3, 4])
    # preempt sequence 2: blocks to pinned host memory, released, then resumed elsewhere
    blocks = loop.bm.swap_out(2)
    hk = torch.empty((len(blocks), B, HKV, D), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pkv.swap_blocks(hk, hv, loop.k, loop.v, torch.tensor(np.stack([blocks, np.arange(len(blocks))], 1),
                                                         dtype=torch.int32).cuda(), status=loop.status)
    torch.cuda.synchronize()
    loop.admit(5, [int(x) for x in rng.integers(0, 1000, size=3 * B)])  # someone else takes blocks meanwhile
    loop.decode(rng, [1, 3, 4, 5])
    new = loop.bm.swap_in(2)
    assert len(new) == len(blocks)
    pkv.swap_blocks(loop.k, loop.v, hk, hv, torch.tensor(np.stack([np.arange(len(new)), new], 1),
                                                         dtype=torch.int32).cuda(), status=loop.status)
    for _ in range(2):
        loop.decode(rng, [1, 2, 3, 4, 5])
    for sid in (1, 2, 3, 4, 5):
        loop.bm.free(sid)
    assert loop.bm.available_blocks == NB


def test_serving_loop_with_batched_bookkeeping_and_cached_swap_in():
    """Decode steps whose bookkeeping comes from pkv_bm_decode_step, and a
    resume through swap_in_cached: full blocks still in the prefix cache are
    shared again, only the others come back from the host."""
    rng = np.random.default_rng(77)
    loop = Loop()
    system = [int(x) for x in rng.integers(0, 1000, size=3 * B)]  # 3 whole blocks
    loop.admit(1, system + [int(x) for x in rng.integers(0, 1000, size=B + 5)])
    assert loop.admit(2, system + [int(x) for x in rng.integers(0, 1000, size=9)]) == 3 * B
    loop.fork(2, 3)  # forked tail: the next batch step copies it once
    for _ in range(3):
        loop.decode_batch(rng, [1, 2, 3])
    # preempt sequence 1: every block goes to the host, the blocks are released
    blocks = loop.bm.swap_out(1)
    hk = torch.empty((len(blocks), B, HKV, D), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    pkv.swap_blocks(hk, hv, loop.k, loop.v, torch.tensor(np.stack([blocks, np.arange(len(blocks))], 1),
                                                         dtype=torch.int32).cuda(), status=loop.status)
    torch.cuda.synchronize()
    loop.decode_batch(rng, [2, 3])
    new, from_host = loop.bm.swap_in_cached(1)
    assert len(new) == len(blocks)
    # the system prompt's blocks (held by sequences 2 and 3) and sequence 1's own full
    # prompt block (released to the prefix cache, not evicted) are shared again; only
    # the partial tail block, which is never cached, comes back from the host
    assert list(from_host) == [0, 0, 0, 0, 1]
    assert np.array_equal(new[:3], loop.bm.block_table(2)[:3])
    idx = np.flatnonzero(from_host)
    pkv.swap_blocks(loop.k, loop.v, hk, hv, torch.tensor(np.stack([idx, new[idx]], 1), dtype=torch.int32).cuda(),
                    status=loop.status)
    for _ in range(2):
        loop.decode_batch(rng, [1, 2, 3])
    for sid in (1, 2, 3):
        loop.bm.free(sid)
