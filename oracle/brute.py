"""Exact brute force of the lightning-indexer top-k for tiny inputs.

Test infrastructure only. Pure Python with `fractions.Fraction`: every input
is decoded exactly (bf16 = upper half of a binary32; f16 = IEEE binary16 and
E4M3 from their definitions, written again here independently of the C
oracle; an E4M3 element is its row scale times its code's value), every
product and sum is exact, and the full list of keys is ordered by
(score descending, key index ascending). A masked (-inf) score is represented
as None and ranks below every finite score.

Definition (llama.cpp issue 25468, root-cause comment; llama.cpp PR 22378,
collapse-Q revert commit; fairydreaming/llama.cpp PR 2, API-change note):
    I[t,s] = sum_h w[t,h] * relu(sum_d q[t,h,d] k[s,d]) + mask[t,s].
"""
from __future__ import annotations

import struct
from fractions import Fraction


def bf16_exact(b: int) -> Fraction:
    (f,) = struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))
    return Fraction(f)


def f16_exact(b: int):
    """Fraction for finite values, +/-float('inf') for infinities."""
    sign = -1 if (b >> 15) & 1 else 1
    e = (b >> 10) & 0x1F
    m = b & 0x3FF
    if e == 31:
        if m:
            raise ValueError("NaN is outside the input contract")
        return sign * float("inf")
    if e == 0:
        return sign * Fraction(m, 1 << 24)
    return sign * Fraction(1024 + m, 1024) * (Fraction(2) ** (e - 15))


def f32_exact(x: float) -> Fraction:
    (f,) = struct.unpack("<f", struct.pack("<f", x))
    return Fraction(f)


def e4m3_exact(b: int) -> Fraction:
    """OCP E4M3 (no infinities) from its definition: bias 7, 3 fraction bits,
    exponent field 0 subnormal; S.1111.111 (NaN) is outside the input contract."""
    sign = -1 if (b >> 7) & 1 else 1
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 15 and m == 7:
        raise ValueError("NaN is outside the input contract")
    if e == 0:
        return sign * Fraction(m, 1 << 9)
    return sign * Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))


def score_rows(q_bits, k_bits, w, mask, n_q, n_kv, H, D, dtype="bf16"):
    """Exact scores: list of rows, each a list of Fraction or None (-inf)."""
    dec = f16_exact if dtype == "f16" else bf16_exact
    qf = [[[dec(int(q_bits[t][h][d])) for d in range(D)] for h in range(H)] for t in range(n_q)]
    kf = [[dec(int(k_bits[s][d])) for d in range(D)] for s in range(n_kv)]
    return _score_values(qf, kf, w, mask, n_q, n_kv, H, D)


def score_rows_e4m3(q8, q_scale, k8, k_scale, w, mask, n_q, n_kv, H, D):
    """Exact scores of the quantised form: q = q_scale[t,h] * e4m3(q8[t,h,d]),
    k = k_scale[s] * e4m3(k8[s,d])."""
    qf = [[[f32_exact(float(q_scale[t][h])) * e4m3_exact(int(q8[t][h][d])) for d in range(D)]
           for h in range(H)] for t in range(n_q)]
    kf = [[f32_exact(float(k_scale[s])) * e4m3_exact(int(k8[s][d])) for d in range(D)] for s in range(n_kv)]
    return _score_values(qf, kf, w, mask, n_q, n_kv, H, D)


def _score_values(qf, kf, w, mask, n_q, n_kv, H, D):
    rows = []
    for t in range(n_q):
        row = []
        for s in range(n_kv):
            total = Fraction(0)
            for h in range(H):
                dot = sum((qf[t][h][d] * kf[s][d] for d in range(D)), Fraction(0))
                total += f32_exact(float(w[t][h])) * max(dot, Fraction(0))
            if mask is not None:
                m = f16_exact(int(mask[t][s]))
                if m == float("-inf"):
                    row.append(None)
                    continue
                if m == float("inf"):
                    raise ValueError("+inf mask is outside the input contract")
                total += m
            row.append(total)
        rows.append(row)
    return rows


def topk(q_bits, k_bits, w, mask, n_q, n_kv, H, D, top_k, dtype="bf16"):
    """Per row: list of (index, score) with score a Fraction or None (-inf);
    padded with (-1, None) when n_kv < top_k."""
    return _select(score_rows(q_bits, k_bits, w, mask, n_q, n_kv, H, D, dtype), n_kv, top_k)


def topk_e4m3(q8, q_scale, k8, k_scale, w, mask, n_q, n_kv, H, D, top_k):
    """`topk` of the quantised form (see `score_rows_e4m3`)."""
    return _select(score_rows_e4m3(q8, q_scale, k8, k_scale, w, mask, n_q, n_kv, H, D), n_kv, top_k)


def _select(score_rows_list, n_kv, top_k):
    out = []
    for row in score_rows_list:
        finite = sorted((s for s in range(n_kv) if row[s] is not None), key=lambda s: (-row[s], s))
        masked = [s for s in range(n_kv) if row[s] is None]  # already index-ascending
        order = finite + masked
        sel = [(s, row[s]) for s in order[:top_k]]
        sel += [(-1, None)] * (top_k - len(sel))
        out.append(sel)
    return out
