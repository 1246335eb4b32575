"""All-layer pools and graph-captured decode steps.

"KV Cache & PagedAttention" section 4 keeps every layer of a block
together, [2][num_blocks][num_layers][16][H_kv][D]; a layer's pool is then a
view whose blocks are num_layers slices apart, which the library takes as a
block stride.  "gpu_paged_kv_cache" ("The write path: slot mapping and
scatter") keeps the tables at fixed addresses, updated in place, so a
captured decode step replays with new contents.  Each layer is checked
against the oracle run on that layer's own contiguous pool."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_112_gb300 as pkv
import pkv_inputs as P
from tests.gpu_util import ATOL, TORCH_DT, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkv.load(build_if_missing=True)


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(TORCH_DT[dtype])


def _oracle_layer(k_pool, v_pool, q, k_new, v_new, bt, cl, sm, pairs, wl):
    k, v = k_pool.copy(), v_pool.copy()
    oracle.copy_blocks(k, v, pairs)
    oracle.write_cache(k, v, k_new, v_new, sm)
    out = oracle.decode_attention(q, k, v, bt, cl, wl.scale, wl.dtype)
    return k, v, out


class LayeredStep:
    """One decode step of every layer over an all-layer pool on the GPU:
    copy-on-write of whole blocks (all layers at once), then per layer the
    fused write + attention and the reduce."""

    def __init__(self, wl, ld, *, extra_cols=0, max_len=None):
        self.wl, self.L = wl, ld.q.shape[0]
        self.pool = _dev(ld.pool, wl.dtype)
        self.q, self.k_new, self.v_new = _dev(ld.q, wl.dtype), _dev(ld.k_new, wl.dtype), _dev(ld.v_new, wl.dtype)
        bt = np.pad(wl.block_tables, ((0, 0), (0, extra_cols)), constant_values=-1)
        self.bt = torch.from_numpy(np.ascontiguousarray(bt)).cuda()
        self.cl = torch.from_numpy(wl.context_lens).cuda()
        self.sm = torch.from_numpy(wl.slot_mapping).cuda()
        self.pairs = torch.from_numpy(np.ascontiguousarray(wl.copy_pairs, dtype=np.int32)).cuda()
        self.out = torch.empty(ld.q.shape, dtype=torch.float32, device="cuda")
        self.max_len = max_len or wl.max_context_len
        nb = pkv.decode_workspace_bytes(wl.num_seqs, wl.num_q_heads, wl.head_dim, self.max_len, wl.partition_size)
        self.ws = torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda") if nb else None
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def layer_pools(self, layer):
        return self.pool[0, :, layer], self.pool[1, :, layer]

    def run(self):
        if self.pairs.shape[0]:
            pkv.copy_blocks(self.pool[0], self.pool[1], self.pairs, status=self.status)
        for layer in range(self.L):
            kp, vp = self.layer_pools(layer)
            pkv.decode_step(self.out[layer], self.q[layer], self.k_new[layer], self.v_new[layer], kp, vp, self.bt,
                            self.cl, self.sm, self.wl.scale, partition_size=self.wl.partition_size,
                            max_context_len=self.max_len, workspace=self.ws, status=self.status)


def _check(step, ref_pools, ref_outs):
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    pool = step.pool.view(torch.int16).cpu().numpy().view(np.uint16)
    for layer, (k, v) in enumerate(ref_pools):
        assert np.array_equal(pool[0, :, layer], k) and np.array_equal(pool[1, :, layer], v), layer
        err = float(np.max(np.abs(step.out[layer].cpu().numpy().astype(np.float64) - ref_outs[layer])))
        assert err <= ATOL, (layer, err)


CASES = {
    "c2_layers": dict(cfg=2, num_seqs=12, lens=("uniform", 1, 300), partition_size=64),
    # copy-on-write of partial tail blocks, moved with every layer
    "c5_layers": dict(cfg=5, num_seqs=8, lens=("prefix", 64, 0, 40), partition_size=32),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_all_layer_pool_step_matches_oracle(case):
    wl = P.make_workload(poison=True, **CASES[case])
    ld = P.make_layers(wl, 3)
    step = LayeredStep(wl, ld)
    step.run()
    refs = [_oracle_layer(ld.pool[0, :, l], ld.pool[1, :, l], ld.q[l], ld.k_new[l], ld.v_new[l], wl.block_tables,
                          wl.context_lens, wl.slot_mapping, wl.copy_pairs, wl) for l in range(3)]
    _check(step, [(k, v) for k, v, _ in refs], [o for _, _, o in refs])


def _advance(bt, cl, num_blocks, rng):
    """The next decode step's bookkeeping: every sequence appends one token;
    a sequence whose last block is full gets a block no table uses."""
    used = set(bt[bt >= 0].tolist())
    free = [b for b in range(num_blocks) if b not in used]
    rng.shuffle(free)
    bt2, cl2 = bt.copy(), cl + 1
    sm2 = np.empty(cl.shape, dtype=np.int32)
    for s, pos in enumerate(cl.tolist()):  # the new token's position is the old length
        blk, off = divmod(pos, 16)
        if off == 0:
            bt2[s, blk] = free.pop()
        sm2[s] = bt2[s, blk] * 16 + off
    return bt2, cl2.astype(np.int32), sm2


def test_graph_replay_with_tables_updated_in_place():
    """A three-layer decode step captured once in a CUDA graph, replayed for
    two consecutive steps: between replays the tables, lengths, slots,
    queries and new rows are rewritten in place in the captured buffers."""
    wl = P.make_workload(2, poison=True, num_seqs=12, lens=("uniform", 1, 300), partition_size=64,
                         pool_factor=1.5)
    L = 3
    ld = P.make_layers(wl, L)
    step = LayeredStep(wl, ld, extra_cols=1, max_len=wl.max_context_len + 1)
    bt1 = step.bt.cpu().numpy()
    # warm-up outside capture (descriptors, function attributes), on an untouched copy of the inputs
    side = torch.cuda.Stream()
    pool0 = step.pool.clone()
    with torch.cuda.stream(side):
        step.run()
    torch.cuda.synchronize()
    step.pool.copy_(pool0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run()
    graph.replay()
    refs = [_oracle_layer(ld.pool[0, :, l], ld.pool[1, :, l], ld.q[l], ld.k_new[l], ld.v_new[l], bt1,
                          wl.context_lens, wl.slot_mapping, wl.copy_pairs, wl) for l in range(L)]
    _check(step, [(k, v) for k, v, _ in refs], [o for _, _, o in refs])

    # step 2: new bookkeeping and values in the same buffers
    rng = np.random.default_rng(5)
    bt2, cl2, sm2 = _advance(bt1, wl.context_lens, wl.num_blocks, rng)
    ld2 = P.make_layers(wl, L, seed=77)
    step.bt.copy_(torch.from_numpy(bt2))
    step.cl.copy_(torch.from_numpy(cl2))
    step.sm.copy_(torch.from_numpy(sm2))
    step.q.copy_(_dev(ld2.q, wl.dtype))
    step.k_new.copy_(_dev(ld2.k_new, wl.dtype))
    step.v_new.copy_(_dev(ld2.v_new, wl.dtype))
    graph.replay()
    refs2 = [_oracle_layer(refs[l][0], refs[l][1], ld2.q[l], ld2.k_new[l], ld2.v_new[l], bt2, cl2, sm2,
                           np.zeros((0, 2), np.int32), wl) for l in range(L)]
    _check(step, [(k, v) for k, v, _ in refs2], [o for _, _, o in refs2])


def test_bulk_prefill_write_then_decode():
    """The pages' worked example ("tm_paged_attention", "End-to-end flow"):
    a 300-token prompt fills 19 blocks through one write of 300 rows (the
    prefill's bulk write), and token 301 lands in logical block 18 with no
    new block; decode then attends over all 301 tokens."""
    rng = np.random.default_rng(301)
    NB, L, Hq, Hkv, D, dtype = 40, 2, 8, 2, 128, "bf16"
    phys = rng.permutation(NB)[:19].astype(np.int32)
    assert -(-300 // 16) == 19 and 300 // 16 == 18 and -(-301 // 16) == 19
    gen = torch.Generator().manual_seed(301)
    nan = P.NAN_BITS[dtype]
    pool = np.full((2, NB, L, 16, Hkv, D), nan, dtype=np.uint16)
    prompt = [P._fill_normal((300, Hkv, D), dtype, gen) for _ in range(2 * L)]  # K, V per layer
    new = [P._fill_normal((1, Hkv, D), dtype, gen) for _ in range(2 * L)]
    q = [P._fill_normal((1, Hq, D), dtype, gen) for _ in range(L)]
    slots = (phys[np.arange(300) // 16] * 16 + np.arange(300) % 16).astype(np.int32)
    bt = phys.reshape(1, 19)
    cl = np.array([301], np.int32)
    slot301 = np.array([phys[18] * 16 + 300 % 16], np.int32)

    dpool = _dev(pool, dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty((L, 1, Hq, D), dtype=torch.float32, device="cuda")
    d_slots, d_bt, d_cl = (torch.from_numpy(x).cuda() for x in (slots, bt, cl))
    d_s301 = torch.from_numpy(slot301).cuda()
    for layer in range(L):
        kp, vp = dpool[0, :, layer], dpool[1, :, layer]
        pkv.write_cache(_dev(prompt[2 * layer], dtype), _dev(prompt[2 * layer + 1], dtype), kp, vp, d_slots,
                        status=status)
        pkv.decode_step(out[layer], _dev(q[layer], dtype), _dev(new[2 * layer], dtype), _dev(new[2 * layer + 1], dtype),
                        kp, vp, d_bt, d_cl, d_s301, 1 / np.sqrt(D), partition_size=0, max_context_len=301,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got_pool = dpool.view(torch.int16).cpu().numpy().view(np.uint16)
    for layer in range(L):
        k, v = pool[0, :, layer].copy(), pool[1, :, layer].copy()
        oracle.write_cache(k, v, prompt[2 * layer], prompt[2 * layer + 1], slots)
        oracle.write_cache(k, v, new[2 * layer], new[2 * layer + 1], slot301)
        assert np.array_equal(got_pool[0, :, layer], k) and np.array_equal(got_pool[1, :, layer], v)
        ref = oracle.decode_attention(q[layer], k, v, bt, cl, 1 / np.sqrt(D), dtype)
        assert float(np.max(np.abs(out[layer].cpu().numpy() - ref))) <= ATOL
