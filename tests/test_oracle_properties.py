"""Property tests of the attention oracle over drawn shapes (CPU only).

For any batch (lengths 0..130, group sizes 1..8, head_dim 8..128, block
sizes 8..64, f16 or bf16, blocks scattered at random through a NaN-poisoned
pool), the oracle equals torch's scaled_dot_product_attention in fp64 on the
contiguous K/V the pool was built from -- paging changes where bytes live,
not what attention computes ("KV Cache & PagedAttention", section 5) -- and
its output is bit-identical when the physical blocks are relabelled
("PagedAttention internals", section 03: reads are oblivious to where a
block sits).  A sequence of length 0 gives a zero row."""
import numpy as np
import pytest
import torch

import oracle
from tests.oracle_pins import _rand_problem, _wid
from tests.oracle_pins_fp8 import Fp8Problem, _widen

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def problems(draw):
    Hkv = draw(st.sampled_from([1, 2, 4]))
    G = draw(st.sampled_from([1, 2, 4, 8]))
    D = draw(st.sampled_from([8, 64, 128]))
    B = draw(st.sampled_from([8, 16, 32, 64]))
    dtype = draw(st.sampled_from(["f16", "bf16"]))
    lens = draw(st.lists(st.integers(0, 130), min_size=1, max_size=4))
    seed = draw(st.integers(0, 2 ** 32 - 1))
    scale = draw(st.sampled_from([0.0, 0.05, 1 / np.sqrt(D), 0.7]))
    return Hkv * G, Hkv, D, B, dtype, lens, seed, scale


@hypothesis.settings(max_examples=60, deadline=None, derandomize=True)
@hypothesis.given(problems())
def test_oracle_equals_sdpa_and_ignores_block_placement(prob):
    Hq, Hkv, D, B, dtype, lens, seed, scale = prob
    rng = np.random.default_rng(seed)
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, lens, Hq, Hkv, D, dtype, nb_extra=3, B=B)
    got = oracle.decode_attention(q, kp, vp, bt, cl, scale, dtype)
    G = Hq // Hkv
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0.0)
            continue
        qs = torch.from_numpy(_wid(q[s], dtype)).reshape(1, Hq, 1, D)
        ks = torch.from_numpy(_wid(K[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        vs = torch.from_numpy(_wid(V[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=scale)[0, :, 0].numpy()
        assert np.max(np.abs(got[s] - ref)) <= 1e-12, s
    # relabel the physical blocks: a permuted pool and the tables mapped through it
    perm = rng.permutation(kp.shape[0])
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    kp2, vp2 = kp[perm], vp[perm]  # new block i holds old block perm[i]
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    got2 = oracle.decode_attention(q, kp2, vp2, bt2, cl, scale, dtype)
    assert np.array_equal(got, got2)


@st.composite
def fp8_problems(draw):
    Hkv = draw(st.sampled_from([1, 2, 4]))
    G = draw(st.sampled_from([1, 2, 4, 8]))
    D = draw(st.sampled_from([16, 64, 128]))
    dtype = draw(st.sampled_from(["f16", "bf16"]))
    lens = draw(st.lists(st.integers(0, 100), min_size=1, max_size=4))
    seed = draw(st.integers(0, 2 ** 32 - 1))
    exact = draw(st.booleans())
    return Hkv * G, Hkv, D, dtype, lens, seed, exact


@hypothesis.settings(max_examples=40, deadline=None, derandomize=True)
@hypothesis.given(fp8_problems())
def test_fp8_oracle_equals_sdpa_on_dequantised_data(prob):
    """The FP8 oracle over drawn shapes, against SDPA in fp64 on the
    contiguous data dequantised through torch's float8_e4m3fn type and each
    logical block's scales ("PagedAttention internals", section 06: the
    block is the quantisation group)."""
    Hq, Hkv, D, dtype, lens, seed, exact = prob
    pr = Fp8Problem(np.random.default_rng(seed), lens, Hq, Hkv, D, dtype, exact=exact)
    got = oracle.decode_attention_fp8(*pr.args())
    G = Hq // Hkv
    for s, L in enumerate(lens):
        if L == 0:
            assert np.all(got[s] == 0.0)
            continue
        K, V = pr.contiguous(s)
        qs = torch.from_numpy(_widen(pr.q[s], dtype)).reshape(1, Hq, 1, D)
        ks = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        vs = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=pr.scale)[0, :, 0].numpy()
        assert np.max(np.abs(got[s] - ref)) <= 1e-12, s
