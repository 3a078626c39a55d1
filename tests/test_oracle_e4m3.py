"""Pins of the oracle's quantised (E4M3) form against things other than itself.

The form: q and k arrive as OCP E4M3 codes with one f32 scale per row, an
element's value being scale * code value; the score is the indexer formula
on those values. Sources: "llama.cpp DeepSeek v4 Flash experimental
inference", section "Plan: Implement CUDA Kernels for DeepSeek v4 (DSV4)
Operations", kernel 3 (dsv4_fp8_kv_quantize: rows quantised to E4M3 against
their amax); "deepseek v4 support" (llama.cpp PR 22378), batched-prefill
commit (the indexer's queries are quantised on its scoring path).

Pins: the decoder against torch's float8_e4m3fn on all 256 codes; the whole
form against exact rational brute force (whose decoder is written again from
the format's definition); the reduction to the 16-bit form when every
dequantised value is a bf16 value; and the exact scale identities of the
formula. `test_oracle_mutants.py` plants slips in these parts and checks that
one of the pins here fails.
"""
import math
import os

import numpy as np
import pytest
import torch

import lid_inputs as li
import oracle
from oracle import brute

NEG_INF = 0xFC00
NAN_CODES = (0x7F, 0xFF)


def _brute_as_arrays(res):
    idx = np.array([[i for i, _ in row] for row in res], dtype=np.int64)
    sc = np.array([[(-math.inf if v is None else float(v)) for _, v in row] for row in res])
    return idx, sc


def _random_codes(rng, shape):
    """Uniform over the 254 non-NaN codes."""
    c = rng.integers(0, 254, size=shape)
    return np.where(c >= 0x7F, c + 1, c).astype(np.uint8)  # skip 0x7F; 0xFF is never drawn


def _random_case(seed, n_q, n_kv, H, D):
    rng = np.random.default_rng(1000 + seed)
    q8 = _random_codes(rng, (n_q, H, D))
    k8 = _random_codes(rng, (n_kv, D))
    qs = rng.uniform(0.01, 2.0, size=(n_q, H)).astype(np.float32)
    ks = rng.uniform(0.01, 2.0, size=n_kv).astype(np.float32)
    ks[rng.integers(0, n_kv)] = 0.0  # an all-zero key row
    w = rng.standard_normal((n_q, H)).astype(np.float32)
    r = rng.random((n_q, n_kv))
    mask = np.where(r < 0.2, np.uint16(NEG_INF), np.where(r < 0.3, li.f16_bits(np.float32(-1.5)), np.uint16(0)))
    return q8, qs, k8, ks, w, mask.astype(np.uint16)


def test_decode_e4m3_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.decode_e4m3(b)
        if b in NAN_CODES:
            assert math.isnan(got) and math.isnan(ref[b])
        else:
            assert got == ref[b], hex(b)
            assert float(brute.e4m3_exact(b)) == ref[b], hex(b)
    assert oracle.decode_e4m3(0x7E) == 448.0 and oracle.decode_e4m3(0x01) == 2.0 ** -9


@pytest.mark.parametrize("seed", range(5))
def test_e4m3_oracle_matches_exact_brute_force(seed):
    n_q, n_kv, H, D = 2, 30 + seed, 1 + seed % 3, 4 + 2 * (seed % 3)
    top_k = [4, 13, 40][seed % 3]  # 40 > n_kv: padding
    q8, qs, k8, ks, w, mask = _random_case(seed, n_q, n_kv, H, D)
    if seed % 2:
        mask = None
    bi, bs = _brute_as_arrays(brute.topk_e4m3(q8, qs, k8, ks, w, mask, n_q, n_kv, H, D, top_k))
    oi, os_ = oracle.topk_e4m3(q8, qs, k8, ks, w, mask, H, D, top_k)
    assert np.array_equal(oi, bi)
    fin = np.isfinite(bs)
    assert np.array_equal(np.isfinite(os_), fin)
    assert np.all(np.abs(os_[fin] - bs[fin]) <= 1e-12 * np.maximum(1.0, np.abs(bs[fin])))
    exact = brute.score_rows_e4m3(q8, qs, k8, ks, w, mask, n_q, n_kv, H, D)
    got = oracle.scores_e4m3(q8, qs, k8, ks, w, mask, H, D)
    for t in range(n_q):
        for s in range(n_kv):
            if exact[t][s] is None:
                assert got[t, s] == -math.inf
            else:
                assert got[t, s] == pytest.approx(float(exact[t][s]), rel=1e-12, abs=1e-12)


def test_e4m3_form_reduces_to_the_16_bit_form():
    # power-of-two scales, distinct per q row (t, h) and per key row: every
    # dequantised value is a bf16 value, so both forms score the same numbers
    rng = np.random.default_rng(7)
    n_q, n_kv, H, D, top_k = 3, 70, 4, 16, 20
    q8 = _random_codes(rng, (n_q, H, D))
    k8 = _random_codes(rng, (n_kv, D))
    qs = np.exp2(rng.integers(-6, 4, size=(n_q, H))).astype(np.float32)
    ks = np.exp2(rng.integers(-6, 4, size=n_kv)).astype(np.float32)
    w = rng.standard_normal((n_q, H)).astype(np.float32)
    mask = li.causal_mask(n_q, n_kv, 50)
    qv = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.float32).numpy() * qs[:, :, None]
    kv = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float32).numpy() * ks[:, None]
    qb, kb = li.f32_to_bf16_bits(qv), li.f32_to_bf16_bits(kv)
    # (the rounding to bf16 is exact: 3 fraction bits and a small exponent range)
    assert np.array_equal((qb.astype(np.uint32) << 16).view(np.float32), qv)
    assert np.array_equal((kb.astype(np.uint32) << 16).view(np.float32), kv)
    i8, s8 = oracle.topk_e4m3(q8, qs, k8, ks, w, mask, H, D, top_k)
    i16, s16 = oracle.topk(qb, kb, w, mask, H, D, top_k, "bf16")
    assert np.array_equal(i8, i16)
    assert np.array_equal(s8, s16)


def test_scale_identities_hold_exactly():
    # w[t,h] * q_scale[t,h] is what the formula uses: moving a power of two from
    # one to the other changes nothing; key scales multiply unmasked scores
    q8, qs, k8, ks, w, _ = _random_case(11, 2, 50, 3, 8)
    base = oracle.scores_e4m3(q8, qs, k8, ks, w, None, 3, 8)
    j = np.array([[1, -2, 3], [0, 2, -1]])
    moved = oracle.scores_e4m3(q8, (qs * np.exp2(j)).astype(np.float32), k8, ks,
                               (w * np.exp2(-j)).astype(np.float32), None, 3, 8)
    assert np.array_equal(moved, base)
    twice = oracle.scores_e4m3(q8, qs, k8, (ks * 4).astype(np.float32), w, None, 3, 8)
    assert np.array_equal(twice, 4 * base)
    # a key row with scale 0 is all zeros: its score is 0 + mask
    assert np.all(base[:, ks == 0] == 0.0)


def test_quantised_inputs_reconstruct_within_half_a_step():
    inp = li.e4m3_inputs("q", 3, 500, 8, 128, 16, seed=4)
    qv = torch.from_numpy(inp.q_bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    kv = torch.from_numpy(inp.k_bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    # every row reaches the format's largest magnitude exactly once scaled
    assert np.all(np.abs(qv).max(axis=-1) == 448.0) and np.all(np.abs(kv).max(axis=-1) == 448.0)
    q = li.normal(li.stream_seed(4, li.STREAM_Q), 3 * 8 * 128).astype(np.float32).reshape(3, 8, 128)
    rel = np.abs(qv * inp.q_scale[:, :, None] - q)
    # nearest rounding: within half the spacing (2^-3 relative for normals,
    # 2^-9 absolute below 2^-6) of the scaled value
    bound = np.maximum(np.abs(q) * 2.0 ** -4, inp.q_scale[:, :, None].astype(np.float64) * 2.0 ** -10)
    assert np.all(rel <= bound * (1 + 1e-6))


def test_hand_worked_golden_example():
    """tests/golden/hand_worked_e4m3.txt is computed by hand (see the file)."""
    g = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked_e4m3.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                key, vals = ln.split(":", 1)
                g[key.strip()] = vals.split()
    q8 = np.array([int(x, 16) for x in g["q8"]], np.uint8).reshape(1, 2, 2)
    k8 = np.array([int(x, 16) for x in g["k8"]], np.uint8).reshape(-1, 2)
    qs = np.array([float(x) for x in g["q_scale"]], np.float32).reshape(1, 2)
    ks = np.array([float(x) for x in g["k_scale"]], np.float32)
    w = np.array([float(x) for x in g["w"]], np.float32).reshape(1, 2)
    idx, sc = oracle.topk_e4m3(q8, qs, k8, ks, w, None, 2, 2, int(g["top_k"][0]))
    assert [int(x) for x in g["idx"]] == list(idx[0])
    assert [float(x) for x in g["score"]] == list(sc[0])
