"""Pins for the attention oracle, written as functions of an implementation.

Each pin takes attn(q, k_pool, v_pool, block_tables, context_lens, scale, dtype)
-> float64 [S, H_q, D] and raises AssertionError when the implementation
disagrees with something the pages or the mathematics fix independently of
it: brute force, a library routine on contiguous data, closed forms,
invariants.  test_oracle_pins runs them on the C++ oracle; test_oracle_mutations
runs them on deliberately broken implementations and checks each is caught.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import pkv_inputs as P
from oracle import brute

B = P.BLOCK_SIZE


def _bits(x, dtype):
    return P.f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


def _wid(b, dtype):
    return P.bits_to_f32(b, dtype).astype(np.float64)


def paged_from_contiguous(K, V, num_blocks, rng, dtype, B=B):
    """Scatter per-sequence contiguous K/V ([L, H_kv, D] bit arrays) into a pool
    of B-token blocks through randomly drawn physical blocks.  Unused slots
    hold NaN."""
    Hkv, D = K[0].shape[1], K[0].shape[2]
    nan = P.NAN_BITS[dtype]
    kp = np.full((num_blocks, B, Hkv, D), nan, dtype=np.uint16)
    vp = np.full_like(kp, nan)
    perm = list(rng.permutation(num_blocks))
    lens = [k.shape[0] for k in K]
    maxb = max(1, max(-(-L // B) for L in lens))
    tables = np.full((len(K), maxb), -1, dtype=np.int32)
    for s, (k, v) in enumerate(zip(K, V)):
        for lb in range(-(-k.shape[0] // B)):
            phys = int(perm.pop())
            tables[s, lb] = phys
            n = min(B, k.shape[0] - lb * B)
            kp[phys, :n] = k[lb * B: lb * B + n]
            vp[phys, :n] = v[lb * B: lb * B + n]
    return kp, vp, tables, np.asarray(lens, dtype=np.int32)


def _rand_problem(rng, lens, Hq, Hkv, D, dtype, nb_extra=5, B=B):
    K = [_bits(rng.standard_normal((L, Hkv, D)), dtype) for L in lens]
    V = [_bits(rng.standard_normal((L, Hkv, D)), dtype) for L in lens]
    q = _bits(rng.standard_normal((len(lens), Hq, D)), dtype)
    nb = sum(-(-L // B) for L in lens) + nb_extra
    kp, vp, bt, cl = paged_from_contiguous(K, V, nb, rng, dtype, B)
    return q, K, V, kp, vp, bt, cl


def pin_block_sizes(attn, dtype="bf16"):
    """Blocks of 8, 32 and 64 tokens: torch SDPA in fp64 on the contiguous K/V
    the pool was built from ("gpu_paged_kv_cache", "Fixed-size blocks": a
    position is found through the table for every block size B)."""
    rng = np.random.default_rng(17)
    lens = [1, 7, 8, 9, 33, 64, 65, 130]
    Hq, Hkv, D = 4, 2, 32
    for bs in (8, 32, 64):
        q, K, V, kp, vp, bt, cl = _rand_problem(rng, lens, Hq, Hkv, D, dtype, B=bs)
        got = attn(q, kp, vp, bt, cl, 0.3, dtype)
        G = Hq // Hkv
        for s, L in enumerate(lens):
            qs = torch.from_numpy(_wid(q[s], dtype)).reshape(1, Hq, 1, D)
            ks = torch.from_numpy(_wid(K[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
            vs = torch.from_numpy(_wid(V[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
            ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=0.3)[0, :, 0].numpy()
            assert np.max(np.abs(got[s] - ref)) <= 1e-12, (bs, s)


def pin_brute_force(attn):
    """Config-1 recipe after its write step, poisoned, vs the pure-Python loop."""
    import oracle

    wl = P.make_workload(1, poison=True)
    k, v, _ = oracle.apply_step(wl, attention=False)
    got = attn(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    ref = np.asarray(brute.decode_attention(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, wl.dtype))
    assert np.max(np.abs(got - ref)) <= 1e-12, np.max(np.abs(got - ref))


def pin_sdpa(attn, dtype="f16"):
    """torch scaled_dot_product_attention in fp64 on the contiguous K/V the pool was built from."""
    rng = np.random.default_rng(11)
    lens = [1, 5, 16, 17, 40, 64]
    Hq, Hkv, D = 6, 2, 32
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, lens, Hq, Hkv, D, dtype)
    scale = 0.37
    got = attn(q, kp, vp, bt, cl, scale, dtype)
    G = Hq // Hkv
    for s, L in enumerate(lens):
        qs = torch.from_numpy(_wid(q[s], dtype)).reshape(1, Hq, 1, D)
        ks = torch.from_numpy(_wid(K[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        vs = torch.from_numpy(_wid(V[s], dtype)).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=scale)[0, :, 0].numpy()
        assert np.max(np.abs(got[s] - ref)) <= 1e-12, (s, np.max(np.abs(got[s] - ref)))


def pin_single_token(attn, dtype="bf16"):
    """L = 1: softmax of one score is 1, the output is v_0 exactly."""
    rng = np.random.default_rng(12)
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, [1, 1, 1], 4, 2, 64, dtype)
    got = attn(q, kp, vp, bt, cl, 1 / 8, dtype)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(got[s, h], _wid(V[s][0, h // 2], dtype)), (s, h)


def pin_zero_scale_mean(attn, dtype="f16"):
    """scale = 0: every weight is 1/L, the output is the mean of the values."""
    rng = np.random.default_rng(13)
    lens = [3, 16, 33]
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, lens, 4, 4, 16, dtype)
    got = attn(q, kp, vp, bt, cl, 0.0, dtype)
    for s, L in enumerate(lens):
        ref = _wid(V[s], dtype).mean(axis=0)  # [H_kv, D]
        assert np.max(np.abs(got[s] - ref)) <= 1e-13


def pin_equal_keys_mean(attn, dtype="f16"):
    """All keys equal: all scores equal, the output is the mean of the values."""
    rng = np.random.default_rng(14)
    lens = [7, 20]
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, lens, 2, 1, 16, dtype)
    row = _bits(rng.standard_normal(16), dtype)
    K2 = [np.broadcast_to(row, k.shape).copy() for k in K]
    kp, vp, bt, cl = paged_from_contiguous(K2, V, 8, np.random.default_rng(1), dtype)
    got = attn(q, kp, vp, bt, cl, 0.25, dtype)
    for s in range(2):
        ref = _wid(V[s], dtype).mean(axis=0)
        assert np.max(np.abs(got[s] - ref)) <= 1e-13


def pin_dominant_key(attn, dtype="f16"):
    """One key aligned with q and a large scale: the output is that key's value."""
    rng = np.random.default_rng(15)
    L, D = 37, 16
    for j in (0, 16, 36):  # first token, a block boundary, the token written this step
        qv = np.zeros((1, 1, D), np.float32)
        qv[0, 0, 0] = 1.0
        k = np.zeros((L, 1, D), np.float32)
        k[j, 0, 0] = 1.0
        q = _bits(qv, dtype)
        K = [_bits(k, dtype)]
        V = [_bits(rng.standard_normal((L, 1, D)), dtype)]
        kp, vp, bt, cl = paged_from_contiguous(K, V, 6, rng, dtype)
        got = attn(q, kp, vp, bt, cl, 100.0, dtype)  # others weigh e^-100
        assert np.max(np.abs(got[0, 0] - _wid(V[0][j, 0], dtype))) <= 1e-12, j


def pin_grouping(attn, dtype="f16"):
    """H_q = 6, H_kv = 3: query heads 2g, 2g+1 read KV head g (contiguous groups)."""
    rng = np.random.default_rng(16)
    L, D = 21, 8
    v = np.zeros((L, 3, D), np.float32)
    for g in range(3):
        v[:, g, :] = g + 1.0
    K = [_bits(rng.standard_normal((L, 3, D)), dtype)]
    V = [_bits(v, dtype)]
    q = _bits(rng.standard_normal((1, 6, D)), dtype)
    kp, vp, bt, cl = paged_from_contiguous(K, V, 4, rng, dtype)
    got = attn(q, kp, vp, bt, cl, 0.3, dtype)
    for h in range(6):
        assert np.allclose(got[0, h], h // 2 + 1.0, atol=1e-12, rtol=0), h


def pin_len_boundary(attn, dtype="f16"):
    """Tokens at positions >= L never count, even finite ones with a huge score,
    and the token at L-1 does count."""
    rng = np.random.default_rng(17)
    L, D = 20, 16
    q, K, V, kp, vp, bt, cl = _rand_problem(rng, [L], 2, 1, D, dtype, nb_extra=0)
    base = attn(q, kp, vp, bt, cl, 0.25, dtype)
    phys = int(bt[0, 1])
    qv = _wid(q[0, 0], dtype)
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[phys, 4:, 0] = _bits(40.0 * np.sign(qv) , dtype)  # slots 20..31: past L, huge scores
    vp2[phys, 4:, 0] = _bits(np.full(D, 7.0), dtype)
    got = attn(q, kp2, vp2, bt, cl, 0.25, dtype)
    assert np.array_equal(got, base)
    cl3 = cl + 1  # now slot 20 is in range: result must move towards 7
    got3 = attn(q, kp2, vp2, bt, cl3, 0.25, dtype)
    assert np.all(np.abs(got3[0, 0] - 7.0) < 1e-6)


def pin_permutation_invariance(attn, dtype="bf16"):
    """Relabelling physical blocks (pool and tables permuted together) changes nothing, bit for bit."""
    import oracle

    wl = P.make_workload(1, poison=True, dtype=dtype)
    k, v, _ = oracle.apply_step(wl, attention=False)
    base = attn(wl.q, k, v, wl.block_tables, wl.context_lens, wl.scale, dtype)
    rng = np.random.default_rng(18)
    pi = rng.permutation(wl.num_blocks)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    bt2 = np.where(wl.block_tables >= 0, pi[np.maximum(wl.block_tables, 0)], -1).astype(np.int32)
    got = attn(wl.q, k2, v2, bt2, wl.context_lens, wl.scale, dtype)
    assert np.array_equal(got, base)


def pin_shared_prefix(attn, dtype="f16"):
    """Sequences whose tables share prefix blocks give the same result as
    sequences holding private copies of those blocks."""
    rng = np.random.default_rng(19)
    Hkv, D, S, pre = 2, 16, 4, 48
    pk = _bits(rng.standard_normal((pre, Hkv, D)), dtype)
    pv = _bits(rng.standard_normal((pre, Hkv, D)), dtype)
    sfx = [0, 5, 16, 23]
    K = [np.concatenate([pk, _bits(rng.standard_normal((n, Hkv, D)), dtype)]) for n in sfx]
    V = [np.concatenate([pv, _bits(rng.standard_normal((n, Hkv, D)), dtype)]) for n in sfx]
    q = _bits(rng.standard_normal((S, 4, D)), dtype)
    kp, vp, bt, cl = paged_from_contiguous(K, V, 40, rng, dtype)  # private copies
    private = attn(q, kp, vp, bt, cl, 0.25, dtype)
    # shared: every sequence points its first 3 entries at sequence 0's prefix blocks
    bt_sh = bt.copy()
    bt_sh[1:, :3] = bt[0, :3]
    for s in range(1, S):  # the private prefix copies become garbage
        kp[bt[s, :3]] = P.NAN_BITS[dtype]
        vp[bt[s, :3]] = P.NAN_BITS[dtype]
    shared = attn(q, kp, vp, bt_sh, cl, 0.25, dtype)
    assert np.array_equal(private, shared)


def pin_poison(attn):
    """NaN in every slot no sequence owns never reaches the output."""
    import oracle

    wl_p = P.make_workload(1, poison=True)
    wl_c = P.make_workload(1, poison=False)
    kp, vp, _ = oracle.apply_step(wl_p, attention=False)
    kc, vc, _ = oracle.apply_step(wl_c, attention=False)
    a = attn(wl_p.q, kp, vp, wl_p.block_tables, wl_p.context_lens, wl_p.scale, wl_p.dtype)
    b = attn(wl_c.q, kc, vc, wl_c.block_tables, wl_c.context_lens, wl_c.scale, wl_c.dtype)
    assert np.all(np.isfinite(a))
    assert np.array_equal(a, b)


ALL_PINS = [pin_brute_force, pin_sdpa, pin_block_sizes, pin_single_token, pin_zero_scale_mean, pin_equal_keys_mean,
            pin_dominant_key, pin_grouping, pin_len_boundary, pin_permutation_invariance,
            pin_shared_prefix, pin_poison]
