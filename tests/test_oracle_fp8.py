"""The FP8-pool oracle checked against things other than itself (CPU only),
and each plausible mistake planted in an implementation of its definition
(on the CPU, in this file only) caught by at least one pin."""
import math

import numpy as np
import pytest

import oracle
import pkv_inputs as P
from tests import oracle_pins_fp8 as p8

B = P.BLOCK_SIZE


# ------------------------------------------------------------------ e4m3 codec


def test_decode_closed_forms():
    """Values fixed by the format: bias 7, 3 mantissa bits, subnormals below
    2^-6, largest finite 448, NaN at S.1111.111, no infinities."""
    d = oracle.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x40, 0x77, 0x7E, 0x80, 0xB8, 0xFE],
                                    dtype=np.uint8))
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 2.0, 240.0, 448.0, -0.0, -1.0, -448.0]
    assert d.tolist() == want
    assert math.copysign(1.0, d[9]) == -1.0
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_decode_matches_torch_every_code():
    codes = np.arange(256, dtype=np.uint8)
    got, ref = oracle.e4m3_decode(codes), p8.deq_torch(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(200_000) * 60, rng.standard_normal(50_000) * 1e-2,
                        rng.uniform(-448, 448, 50_000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(x), p8.enc_torch(x))


def test_encode_saturates_and_keeps_nan():
    """Beyond 448 the code saturates to the largest finite value (the format
    has no infinity); NaN stays NaN."""
    x = np.array([448.0, 463.99, 464.0, 1e4, np.inf, -500.0, -np.inf, np.nan], dtype=np.float32)
    assert oracle.e4m3_encode(x).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_encode_decode_round_trip_every_code():
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(p8.FINITE_CODES).astype(np.float32)),
                          p8.FINITE_CODES)


# ------------------------------------------------------------------ pins on the oracle


@pytest.mark.parametrize("pin", p8.ATTN_PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    pin(oracle.decode_attention_fp8)


@pytest.mark.parametrize("pin", p8.WRITE_PINS, ids=lambda f: f.__name__)
def test_write_pin(pin):
    pin(oracle.write_cache_fp8)


@pytest.mark.parametrize("pin", p8.COPY_PINS, ids=lambda f: f.__name__)
def test_copy_pin(pin):
    pin(oracle.copy_blocks_fp8)


def test_sampled_rows_match_full():
    wl = P.make_workload(1, poison=True)
    pools = P.make_fp8_pools(wl)
    k8, v8, ks, vs, full = oracle.apply_step_fp8(wl, pools)
    rows = [(3, 1), (0, 0), (2, 3)]
    part = oracle.decode_attention_fp8(wl.q, k8, v8, ks, vs, wl.block_tables, wl.context_lens, wl.scale,
                                       wl.dtype, rows=rows)
    for i, (s, h) in enumerate(rows):
        assert np.array_equal(part[i], full[s, h])


def test_step_copies_before_writing():
    """Prefix-sharing recipe, poisoned: a copy-on-write destination's scales
    are NaN until the copy, so a write quantising with them (or an attention
    reading them) before the copy would leave NaN behind."""
    wl = P.make_workload(5, poison=True, num_seqs=6, num_q_heads=4, num_kv_heads=2, head_dim=32,
                         lens=("prefix", 32, 0, 40))
    assert wl.copy_pairs.size
    pools = P.make_fp8_pools(wl)
    k8, v8, ks, vs, out = oracle.apply_step_fp8(wl, pools)
    assert np.all(np.isfinite(out))
    for i, slot in enumerate(wl.slot_mapping.tolist()):
        b, o = divmod(slot, B)
        assert not np.isnan(ks[b]).any()
        x = P.bits_to_f32(wl.k_new[i], wl.dtype)
        want = p8._expected_codes(x, np.repeat(ks[b][:, None], wl.head_dim, axis=1))
        assert np.array_equal(k8[b, o], want)
    src, dst = wl.copy_pairs[:, 0], wl.copy_pairs[:, 1]
    assert np.array_equal(ks[dst], pools.k_scale[src]) and np.array_equal(vs[dst], pools.v_scale[src])


def test_generator_never_draws_nan_and_poisons_dead_slots():
    wl = P.make_workload(1, poison=True)
    pools = P.make_fp8_pools(wl)
    live = wl.live
    assert not np.any((pools.k8[live] & 0x7F) == 0x7F)
    assert np.all(pools.k8[~live] == P.FP8_NAN) and np.all(pools.v8[~live] == P.FP8_NAN)
    clean = P.make_fp8_pools(wl, poison=False)
    assert not np.any((clean.k8 & 0x7F) == 0x7F) and np.all(np.isfinite(clean.k_scale))


# ------------------------------------------------------------------ planted mistakes


def _planted_decode(codes, mutation):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    if mutation == "sign_ignored":
        sign = np.ones_like(sign)
    e, m = (c >> 3) & 0xF, c & 0x7
    bias = 8 if mutation == "exponent_bias_8" else 7
    normal = np.ldexp((8 + m).astype(np.float64), e - bias - 3)
    sub = np.ldexp(m.astype(np.float64), -bias - 2)
    if mutation == "subnormal_as_normal":
        sub = np.ldexp((8 + m).astype(np.float64), -bias - 3)
    v = np.where(e == 0, sub, normal)
    return sign * np.where((e == 15) & (m == 7), np.nan, v)


def _planted_attn8(mutation):
    def attn8(q, k8, v8, ks, vs, bt, cl, scale, dtype):
        qf = P.bits_to_f32(q, dtype).astype(np.float64)
        S, Hq, D = qf.shape
        NB, _, Hkv, _ = k8.shape
        G = Hq // Hkv
        out = np.zeros((S, Hq, D))
        for s in range(S):
            L = int(cl[s])
            if L <= 0:
                continue
            t = np.arange(L)
            phys, off = bt[s, t // B], t % B
            for g in range(Hkv):
                kf, vf = ks[phys, g].astype(np.float64), vs[phys, g].astype(np.float64)
                if mutation == "k_scale_for_v":
                    vf = kf
                if mutation == "scale_by_logical_block":
                    kf, vf = ks[t // B, g].astype(np.float64), vs[t // B, g].astype(np.float64)
                if mutation == "scale_index_transposed":
                    kf = ks.reshape(-1)[(g * NB + phys) % ks.size].astype(np.float64)
                    vf = vs.reshape(-1)[(g * NB + phys) % vs.size].astype(np.float64)
                if mutation == "v_scale_of_head_0":
                    vf = vs[phys, 0].astype(np.float64)
                if mutation == "no_k_scale":
                    kf = np.ones_like(kf)
                if mutation == "divide_by_scale":
                    kf, vf = 1 / kf, 1 / vf
                K = _planted_decode(k8[phys, off, g], mutation) * kf[:, None]
                V = _planted_decode(v8[phys, off, g], mutation) * vf[:, None]
                for h in range(g * G, (g + 1) * G):
                    z = K @ qf[s, h] * scale
                    w = np.exp(z - z.max())
                    out[s, h] = (w / w.sum()) @ V
        return out

    return attn8


ATTN_MUTATIONS = ["sign_ignored", "exponent_bias_8", "subnormal_as_normal", "k_scale_for_v",
                  "scale_by_logical_block", "scale_index_transposed", "v_scale_of_head_0", "no_k_scale",
                  "divide_by_scale"]


def _planted_encode(r, mutation):
    r = np.asarray(r, dtype=np.float64)
    pos = p8.deq_torch(np.arange(0x7F, dtype=np.uint8))
    a = np.abs(r)
    over = a > 448
    a = np.minimum(a, 448.0)
    hi = np.clip(np.searchsorted(pos, a), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    dlo, dhi = a - pos[lo], pos[hi] - a
    tie = hi if mutation == "ties_away" else np.where(lo % 2 == 0, lo, hi)
    code = np.where(dhi < dlo, hi, np.where(dlo < dhi, lo, tie))
    if mutation == "truncate":
        code = np.where(dhi == 0, hi, lo)
    if mutation == "nan_on_overflow":
        code = np.where(over, 0x7F, code)
    if mutation != "no_sign":
        code = code | (np.signbit(r).astype(np.int64) << 7)
    return code.astype(np.uint8)


def _planted_write8(mutation):
    def write8(k8, v8, ks, vs, k_new, v_new, slots, dtype):
        for i, slot in enumerate(np.asarray(slots).tolist()):
            if slot < 0:
                if mutation != "negative_slot_wraps":
                    continue
                slot %= k8.shape[0] * B
            b, o = divmod(slot, B)
            if mutation == "offset_major_slots":
                o, b = divmod(slot, k8.shape[0])
            for pool, sc, new in ((k8, ks, k_new), (v8, vs, v_new)):
                if mutation == "k_only" and pool is v8:
                    continue
                x = P.bits_to_f32(new[i], dtype).astype(np.float32)
                sb = sc[0] if mutation == "scale_of_block_0" else sc[b]
                r = x * sb[:, None] if mutation == "multiply_by_scale" else x / sb[:, None]
                pool[b, o] = _planted_encode(r, mutation)

    return write8


WRITE_MUTATIONS = ["ties_away", "truncate", "nan_on_overflow", "no_sign", "negative_slot_wraps",
                   "offset_major_slots", "k_only", "scale_of_block_0", "multiply_by_scale"]


def _planted_copy8(mutation):
    def copy8(k8, v8, ks, vs, pairs):
        for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
            if mutation == "direction_swapped":
                src, dst = dst, src
            k8[dst] = k8[src]
            v8[dst] = v8[src]
            if mutation != "codes_only":
                ks[dst] = ks[src]
                if mutation != "k_scale_only":
                    vs[dst] = vs[src]

    return copy8


COPY_MUTATIONS = ["direction_swapped", "codes_only", "k_scale_only"]


def _caught(pins, impl):
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, IndexError, ValueError):
            return pin.__name__
    return None


def test_unmutated_statements_pass_all_pins():
    assert _caught(p8.ATTN_PINS, _planted_attn8(None)) is None
    assert _caught(p8.WRITE_PINS, _planted_write8(None)) is None
    assert _caught(p8.COPY_PINS, _planted_copy8(None)) is None


@pytest.mark.parametrize("mutation", ATTN_MUTATIONS)
def test_planted_attention_mistake_is_caught(mutation):
    assert _caught(p8.ATTN_PINS, _planted_attn8(mutation)) is not None, mutation


@pytest.mark.parametrize("mutation", WRITE_MUTATIONS)
def test_planted_write_mistake_is_caught(mutation):
    assert _caught(p8.WRITE_PINS, _planted_write8(mutation)) is not None, mutation


@pytest.mark.parametrize("mutation", COPY_MUTATIONS)
def test_planted_copy_mistake_is_caught(mutation):
    assert _caught(p8.COPY_PINS, _planted_copy8(mutation)) is not None, mutation
