"""The pins are sharp: each plausible mistake planted in an implementation of
the oracle's definition (on the CPU, in this file only) fails at least one pin."""
import math

import numpy as np
import pytest

import pkv_inputs as P
from tests import oracle_pins as pins


def _planted(mutation):
    """A numpy statement of paged decode attention with one planted mistake."""

    def attn(q, kp, vp, bt, cl, scale, dtype):
        qf = P.bits_to_f32(q, dtype).astype(np.float64)
        kf = P.bits_to_f32(kp, dtype).astype(np.float64)
        vf = P.bits_to_f32(vp, dtype).astype(np.float64)
        S, Hq, D = qf.shape
        NB, B, Hkv, _ = kf.shape
        G = Hq // Hkv
        out = np.zeros((S, Hq, D))
        for s in range(S):
            L = int(cl[s])
            if mutation == "drop_last_token":
                L -= 1
            if mutation == "one_extra_token":
                L = min(L + 1, bt.shape[1] * B)
            if L <= 0:
                continue
            t = np.arange(L)
            if mutation == "swap_block_and_offset":
                phys, off = bt[s, t % B % bt.shape[1]], t // B % B
            else:
                phys, off = bt[s, t // B], t % B
            for h in range(Hq):
                g = h % Hkv if mutation == "interleaved_groups" else h // G
                K = kf[phys, off, g]
                V = vf[phys, off, g]
                if mutation == "keys_values_swapped":
                    K, V = V, K
                z = K @ qf[s, h]
                if mutation != "no_scale":
                    z = z * scale
                if mutation == "sign_flip":
                    z = -z
                w = np.exp(z - z.max())
                if mutation != "no_normalisation":
                    w = w / w.sum()
                if mutation == "uniform_weights":
                    w = np.full(L, 1.0 / L)
                out[s, h] = w @ V
        return out

    return attn


MUTATIONS = ["drop_last_token", "one_extra_token", "swap_block_and_offset", "interleaved_groups",
             "keys_values_swapped", "no_scale", "sign_flip", "no_normalisation", "uniform_weights"]


def _caught(attn):
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(attn)
        except (AssertionError, IndexError, ValueError):
            return pin.__name__
    return None


def test_unmutated_statement_passes_all_pins():
    assert _caught(_planted(None)) is None


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_planted_mistake_is_caught(mutation):
    assert _caught(_planted(mutation)) is not None, mutation
