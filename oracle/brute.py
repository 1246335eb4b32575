"""Pure-Python brute force of paged decode attention -- TEST INFRASTRUCTURE ONLY.

An independent restatement (Python floats, math.exp, struct decoding) of the
same definition the C++ oracle implements, used only on tiny inputs to pin
it.  Token t of sequence s is read from physical block
block_tables[s][t // B] at offset t % B ("PagedAttention internals",
section 02 "Block tables"); query head h reads KV head h // (H_q / H_kv);
the result is softmax(scale * q.K^T) V over all L tokens.
"""
from __future__ import annotations

import math
import struct


def widen(bits: int, dtype: str) -> float:
    if dtype == "f16":
        return struct.unpack("<e", struct.pack("<H", bits))[0]
    return struct.unpack("<f", struct.pack("<I", bits << 16))[0]


def decode_attention(q, k_pool, v_pool, block_tables, context_lens, scale, dtype):
    """Nested lists / arrays in, list [S][H_q][D] of Python floats out."""
    S, Hq, D = len(q), len(q[0]), len(q[0][0])
    B, Hkv = len(k_pool[0]), len(k_pool[0][0])
    G = Hq // Hkv
    out = []
    for s in range(S):
        L = int(context_lens[s])
        rows = []
        for h in range(Hq):
            g = h // G
            keys, vals = [], []
            for t in range(L):
                b = int(block_tables[s][t // B])
                keys.append([widen(int(x), dtype) for x in k_pool[b][t % B][g]])
                vals.append([widen(int(x), dtype) for x in v_pool[b][t % B][g]])
            qh = [widen(int(x), dtype) for x in q[s][h]]
            if L == 0:
                rows.append([0.0] * D)
                continue
            scores = [scale * sum(a * c for a, c in zip(qh, k)) for k in keys]
            top = max(scores)
            w = [math.exp(z - top) for z in scores]
            tot = sum(w)
            rows.append([sum(w[t] * vals[t][d] for t in range(L)) / tot for d in range(D)])
        out.append(rows)
    return out
