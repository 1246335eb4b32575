"""Pins for the FP8-pool oracle, written as functions of an implementation.

FP8 pools hold e4m3 codes with one float32 scale per (physical block, KV head)
for K and one for V ("PagedAttention internals" section 06, "Blocks as
quantization groups"; "KV Cache & PagedAttention" section 5).

  attn8(q, k8, v8, k_scale, v_scale, block_tables, context_lens, scale, dtype)
      -> float64 [S, H_q, D]
  write8(k8, v8, k_scale, v_scale, k_new, v_new, slot_mapping, dtype)   (in place)
  copy8(k8, v8, k_scale, v_scale, pairs)                                 (in place)

Every expectation comes from outside the oracle: torch's float8_e4m3fn type
(decode of a code; float32 -> e4m3 rounding of in-range values), torch's
scaled-dot-product attention on contiguous data, the pinned 16-bit oracle on
pools whose dequantised values are exact in 16 bits, and closed forms of the
format (largest finite 448, saturation, ties to the even code).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pkv_inputs as P

B = P.BLOCK_SIZE


def deq_torch(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes -> float64 through torch's float8_e4m3fn type."""
    c = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def enc_torch(x: np.ndarray) -> np.ndarray:
    """float32 -> e4m3 codes through torch's cast (in-range values only)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _pow2_scales(rng, shape):
    return np.ldexp(1.0, rng.integers(-8, -6, size=shape, endpoint=True)).astype(np.float32)


def _rand_scales(rng, shape):
    return np.exp2(rng.uniform(-7.5, -6.5, size=shape)).astype(np.float32)


class Fp8Problem:
    """A paged FP8 problem built from contiguous per-sequence codes and
    per-logical-block scales, scattered through random physical blocks.
    Unused slots hold NaN codes; unused blocks NaN scales."""

    def __init__(self, rng, lens, Hq, Hkv, D, dtype, exact, nb_extra=5, codes=P.draw_fp8_codes):
        self.lens, self.Hq, self.Hkv, self.D, self.dtype = list(lens), Hq, Hkv, D, dtype
        nblk = [-(-L // B) for L in self.lens]
        NB = sum(nblk) + nb_extra
        scales = _pow2_scales if exact else _rand_scales
        self.K8 = [codes((L, Hkv, D), rng) for L in self.lens]
        self.V8 = [codes((L, Hkv, D), rng) for L in self.lens]
        self.KS = [scales(rng, (n, Hkv)) for n in nblk]
        self.VS = [scales(rng, (n, Hkv)) for n in nblk]
        self.k8 = np.full((NB, B, Hkv, D), P.FP8_NAN, dtype=np.uint8)
        self.v8 = np.full_like(self.k8, P.FP8_NAN)
        self.ks = np.full((NB, Hkv), np.nan, dtype=np.float32)
        self.vs = np.full_like(self.ks, np.nan)
        perm = list(rng.permutation(NB))
        self.bt = np.full((len(self.lens), max(1, max(nblk, default=1))), -1, dtype=np.int32)
        for s, L in enumerate(self.lens):
            for j in range(nblk[s]):
                phys = perm.pop()
                self.bt[s, j] = phys
                n = min(B, L - j * B)
                self.k8[phys, :n] = self.K8[s][j * B:j * B + n]
                self.v8[phys, :n] = self.V8[s][j * B:j * B + n]
                self.ks[phys] = self.KS[s][j]
                self.vs[phys] = self.VS[s][j]
        self.cl = np.asarray(self.lens, dtype=np.int32)
        qf = rng.standard_normal((len(self.lens), Hq, D)).astype(np.float32)
        self.q = P.f32_to_bits(qf, dtype)
        self.scale = 1.0 / np.sqrt(D)

    def args(self):
        return (self.q, self.k8, self.v8, self.ks, self.vs, self.bt, self.cl, self.scale, self.dtype)

    def contiguous(self, s):
        """Dequantised contiguous K, V of sequence s ([L, H_kv, D] float64), via torch."""
        tok_blk = np.arange(self.lens[s]) // B
        K = deq_torch(self.K8[s]) * self.KS[s][tok_blk][:, :, None].astype(np.float64)
        V = deq_torch(self.V8[s]) * self.VS[s][tok_blk][:, :, None].astype(np.float64)
        return K, V


# ------------------------------------------------------------------ attention


def _widen(bits, dtype):
    return P.bits_to_f32(bits, dtype).astype(np.float64)


def pin8_sdpa(attn8, dtype="bf16"):
    """torch scaled_dot_product_attention in fp64 on the contiguous K/V,
    dequantised through torch's float8 type and each logical block's scales
    (random, not powers of two)."""
    rng = np.random.default_rng(81)
    lens = [1, 15, 16, 17, 40, 77]
    Hq, Hkv, D = 8, 2, 32
    pr = Fp8Problem(rng, lens, Hq, Hkv, D, dtype, exact=False)
    got = attn8(*pr.args())
    G = Hq // Hkv
    for s in range(len(lens)):
        K, V = pr.contiguous(s)
        qs = torch.from_numpy(_widen(pr.q[s], dtype)).reshape(1, Hq, 1, D)
        ks = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        vs = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=pr.scale)[0, :, 0].numpy()
        assert np.max(np.abs(got[s] - ref)) <= 1e-12, (s, np.max(np.abs(got[s] - ref)))


def _pools16(codes, scales, dtype):
    """Dequantised pool -> 16-bit patterns; exact when the scales are powers of two."""
    x = deq_torch(codes) * scales.astype(np.float64)[:, None, :, None]
    bad = ~np.isfinite(x)
    x32 = np.where(bad, 0.0, x).astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), np.where(bad, 0.0, x))
    bits = P.f32_to_bits(x32, dtype)
    assert np.array_equal(_widen(bits, dtype), x32.astype(np.float64)), "not exact in 16 bits"
    bits[bad] = P.NAN_BITS[dtype]
    return bits


def pin8_exact_vs_16bit(attn8, dtype="f16"):
    """Power-of-two scales that differ per block, KV head and K/V: every
    dequantised value is exact in 16 bits, so the result equals the pinned
    16-bit oracle's on those values."""
    rng = np.random.default_rng(82)
    lens = [33, 1, 48, 70, 16, 5]
    Hq, Hkv, D = 12, 3, 64
    pr = Fp8Problem(rng, lens, Hq, Hkv, D, dtype, exact=True)
    got = attn8(*pr.args())
    k16 = _pools16(pr.k8, pr.ks, dtype)
    v16 = _pools16(pr.v8, pr.vs, dtype)
    ref = oracle.decode_attention(pr.q, k16, v16, pr.bt, pr.cl, pr.scale, dtype)
    assert np.max(np.abs(got - ref)) <= 1e-13, np.max(np.abs(got - ref))


def pin8_scale_homogeneity(attn8, dtype="bf16"):
    """Output is linear in the V scales; the K scales and the logit scale enter
    only as their product."""
    rng = np.random.default_rng(83)
    pr = Fp8Problem(rng, [20, 3, 50], 4, 2, 32, dtype, exact=True)
    q, k8, v8, ks, vs, bt, cl, scale, dt = pr.args()
    base = attn8(q, k8, v8, ks, vs, bt, cl, scale, dt)
    assert np.all(np.isfinite(base))
    v4 = attn8(q, k8, v8, ks, vs * np.float32(4), bt, cl, scale, dt)
    assert np.array_equal(v4, 4 * base)
    k2 = attn8(q, k8, v8, ks * np.float32(2), vs, bt, cl, scale / 2, dt)
    assert np.max(np.abs(k2 - base)) <= 1e-13


FINITE_CODES = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)


def every_code(shape, rng):
    """Codes covering every finite e4m3 value (subnormals and -0 included), shuffled."""
    n = int(np.prod(shape))
    return rng.permutation(np.resize(FINITE_CODES, max(n, 1)))[:n].reshape(shape)


def pin8_sdpa_every_code(attn8, dtype="f16"):
    """As pin8_sdpa, with K and V running through every finite code."""
    rng = np.random.default_rng(86)
    lens = [8, 9]
    Hq, Hkv, D = 2, 1, 32
    pr = Fp8Problem(rng, lens, Hq, Hkv, D, dtype, exact=False, codes=every_code)
    assert set(np.unique(pr.K8[0])) == set(FINITE_CODES)
    got = attn8(*pr.args())
    for s in range(len(lens)):
        K, V = pr.contiguous(s)
        qs = torch.from_numpy(_widen(pr.q[s], dtype)).reshape(1, Hq, 1, D)
        ks = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(Hq, 0).unsqueeze(0)
        vs = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(Hq, 0).unsqueeze(0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=pr.scale)[0, :, 0].numpy()
        assert np.max(np.abs(got[s] - ref)) <= 1e-12, (s, np.max(np.abs(got[s] - ref)))


def pin8_single_token(attn8, dtype="f16"):
    """L = 1: the output is the dequantised v_0, exactly."""
    rng = np.random.default_rng(84)
    pr = Fp8Problem(rng, [1, 1, 1, 1], 4, 2, 64, dtype, exact=False, codes=every_code)
    got = attn8(*pr.args())
    for s in range(4):
        _, V = pr.contiguous(s)
        for h in range(4):
            assert np.array_equal(got[s, h], V[0, h // 2]), (s, h)


def pin8_empty_sequence(attn8, dtype="f16"):
    """L = 0 reads nothing and writes zeros."""
    rng = np.random.default_rng(85)
    pr = Fp8Problem(rng, [0, 9], 4, 2, 16, dtype, exact=False)
    got = attn8(*pr.args())
    assert np.array_equal(got[0], np.zeros_like(got[0])) and np.all(np.isfinite(got[1]))


ATTN_PINS = [pin8_sdpa, pin8_sdpa_every_code, pin8_exact_vs_16bit, pin8_scale_homogeneity, pin8_single_token, pin8_empty_sequence]


# ------------------------------------------------------------------ write / copy


def _expected_codes(x32: np.ndarray, s32: np.ndarray) -> np.ndarray:
    """e4m3 of float32(x) / float32(s): torch's cast inside the finite range,
    the largest finite code (0x7E, with the sign) beyond it."""
    r = (torch.from_numpy(x32) / torch.from_numpy(s32)).numpy()
    sat = np.abs(r) > 448
    inside = enc_torch(np.where(sat, 0, r).astype(np.float32))
    return np.where(sat, np.where(r < 0, 0xFE, 0x7E), inside).astype(np.uint8)


def pin8_write_torch(write8, dtype="bf16"):
    """Each new row lands in its slot as e4m3(x / scale of its block and KV
    head); rows of other slots, the scales and slot -1 leave the pools alone."""
    rng = np.random.default_rng(91)
    NB, Hkv, D = 6, 3, 16
    k8 = P.draw_fp8_codes((NB, B, Hkv, D), rng)
    v8 = P.draw_fp8_codes((NB, B, Hkv, D), rng)
    ks, vs = _rand_scales(rng, (NB, Hkv)), _rand_scales(rng, (NB, Hkv))
    slots = np.array([5 * B + 3, -1, 0, 2 * B + 15, 5 * B + 4], dtype=np.int32)
    T = slots.size
    k_new = P.f32_to_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 2, dtype)
    v_new = P.f32_to_bits(rng.standard_normal((T, Hkv, D)).astype(np.float32) * 2, dtype)
    k0, v0, ks0, vs0 = k8.copy(), v8.copy(), ks.copy(), vs.copy()
    write8(k8, v8, ks, vs, k_new, v_new, slots, dtype)
    assert np.array_equal(ks, ks0) and np.array_equal(vs, vs0)
    touched = np.zeros((NB, B), dtype=bool)
    n_sat = 0
    for i, slot in enumerate(slots.tolist()):
        if slot < 0:
            continue
        b, o = divmod(slot, B)
        touched[b, o] = True
        for pool, new, sc in ((k8, k_new, ks), (v8, v_new, vs)):
            x = P.bits_to_f32(new[i], dtype)
            want = _expected_codes(x, np.repeat(sc[b][:, None], D, axis=1))
            assert np.array_equal(pool[b, o], want), (i, slot)
            n_sat += int(np.sum((want & 0x7F) == 0x7E))
    assert n_sat > 0, "the draw must reach the saturation branch"
    assert np.array_equal(k8[~touched], k0[~touched]) and np.array_equal(v8[~touched], v0[~touched])


def pin8_write_ties(write8, dtype="f16"):
    """Values exactly halfway between two neighbouring e4m3 values (times a
    power-of-two scale) take the code with the even mantissa; values on a
    representable point take that point's code."""
    pos = deq_torch(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448 ascending
    mids = (pos[:-1] + pos[1:]) / 2
    even = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F)).astype(np.uint8)
    vals = np.concatenate([mids, -mids, pos, -pos[1:]])
    want = np.concatenate([even, even | 0x80, np.arange(0x7F), np.arange(1, 0x7F) | 0x80]).astype(np.uint8)
    D = 32
    n = -(-vals.size // D) * D
    vals = np.pad(vals, (0, n - vals.size))
    want = np.pad(want, (0, n - want.size))
    T = n // D
    s = np.float32(2.0 ** -7)
    x = (vals * float(s)).astype(np.float32)
    bits = P.f32_to_bits(x, dtype)
    assert np.array_equal(P.bits_to_f32(bits, dtype).astype(np.float64), vals * float(s))
    k8 = np.zeros((T, B, 1, D), dtype=np.uint8)
    v8 = np.zeros_like(k8)
    ks = np.full((T, 1), s, dtype=np.float32)
    vs = ks.copy()
    new = bits.reshape(T, 1, D)
    slots = (np.arange(T) * B + 7).astype(np.int32)
    write8(k8, v8, ks, vs, new, new, slots, dtype)
    assert np.array_equal(k8[:, 7, 0].reshape(-1), want)
    assert np.array_equal(v8[:, 7, 0].reshape(-1), want)


def pin8_copy(copy8):
    """Each destination block becomes its source: codes and scales, K and V;
    nothing else moves."""
    rng = np.random.default_rng(92)
    NB, Hkv, D = 9, 2, 16
    k8 = P.draw_fp8_codes((NB, B, Hkv, D), rng)
    v8 = P.draw_fp8_codes((NB, B, Hkv, D), rng)
    ks, vs = _rand_scales(rng, (NB, Hkv)), _rand_scales(rng, (NB, Hkv))
    pairs = np.array([[1, 7], [4, 2], [0, 8]], dtype=np.int32)
    k0, v0, ks0, vs0 = k8.copy(), v8.copy(), ks.copy(), vs.copy()
    copy8(k8, v8, ks, vs, pairs)
    src, dst = pairs[:, 0], pairs[:, 1]
    keep = np.setdiff1d(np.arange(NB), dst)
    for a, a0 in ((k8, k0), (v8, v0), (ks, ks0), (vs, vs0)):
        assert np.array_equal(a[dst], a0[src])
        assert np.array_equal(a[keep], a0[keep])


WRITE_PINS = [pin8_write_torch, pin8_write_ties]
COPY_PINS = [pin8_copy]
