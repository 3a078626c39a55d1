"""Pins of the oracle's sparse attention over the selected latent rows (the
consumer of the top-k; llama.cpp issue 25468, root-cause comment: the top-512
feeds the CSA attention; llama.cpp PR 22378, batched-prefill commit: Q*K^T ->
softmax -> *V over the V4 MLA latent KV, masked slots contribute zero).

Each pin comes from outside the oracle's own formula: closed forms (identical
rows, zero queries, one selection, a two-key case with weights 3/4 and 1/4),
invariances (order of the selections, removing excluded ones), a limit (a
dominant score selects its row), and the textbook reduction to scipy's
softmax / logsumexp on random inputs.
"""
import math

import numpy as np
import pytest

import lid_inputs as li
import oracle


def _bf16(x):
    return li.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _dec(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_identical_rows_give_that_row_and_zero_queries_the_mean():
    rng = np.random.default_rng(1)
    Dc, Ha = 16, 3
    v = rng.integers(-4, 5, Dc).astype(np.float32)
    kv = np.tile(v, (40, 1))
    qa = rng.integers(-3, 4, (2, Ha, Dc)).astype(np.float32)
    idx = np.array([[3, 7, 11, 19], [0, 1, 2, 39]], np.int32)
    out, lse = oracle.sparse_attn(_bf16(qa), _bf16(kv), idx, None, Ha, Dc, 0.25)
    assert np.allclose(out, v[None, None, :], rtol=0, atol=1e-12)
    # zero queries: uniform weights over the selection
    kv2 = rng.integers(-4, 5, (40, Dc)).astype(np.float32)
    out, lse = oracle.sparse_attn(_bf16(np.zeros_like(qa)), _bf16(kv2), idx, None, Ha, Dc, 0.7)
    for t in range(2):
        assert np.allclose(out[t], kv2[idx[t]].mean(axis=0)[None, :], rtol=0, atol=1e-12)
        assert np.allclose(lse[t], math.log(4.0), rtol=0, atol=1e-12)


def test_single_selection_and_two_keys_three_to_one():
    Dc = 8
    kv = np.zeros((10, Dc), np.float32)
    kv[2, 0], kv[5, 0] = 2.0, 1.0
    kv[2, 1], kv[5, 1] = 5.0, -7.0
    qa = np.zeros((1, 1, Dc), np.float32)
    qa[0, 0, 0] = 1.0
    # one selection: its row; lse = scale * s
    out, lse = oracle.sparse_attn(_bf16(qa), _bf16(kv), np.array([[5, -1, -1]], np.int32), None, 1, Dc, 0.5)
    assert np.allclose(out[0, 0], kv[5]) and lse[0, 0] == pytest.approx(0.5 * 1.0, abs=1e-15)
    # s_2 - s_5 = 1: with scale ln 3 the weights are 3/4 and 1/4
    scale = math.log(3.0)
    out, lse = oracle.sparse_attn(_bf16(qa), _bf16(kv), np.array([[5, 2]], np.int32), None, 1, Dc, scale)
    assert np.allclose(out[0, 0], 0.75 * kv[2] + 0.25 * kv[5], rtol=0, atol=1e-12)
    assert lse[0, 0] == pytest.approx(scale * 2.0 + math.log(1.0 + 1.0 / 3.0), abs=1e-12)


def test_exclusions_and_order_do_not_change_the_result():
    a = li.attn_inputs("x", 4, 300, 3, 32, 24, seed=3, n_invalid=6)
    out, lse = oracle.sparse_attn(a.qa_bits, a.kv_bits, a.idx, a.sel_score, a.Ha, a.Dc, a.scale)
    # the same selections without the excluded ones, in reversed order, padded with -1
    kept = np.full_like(a.idx, -1)
    for t in range(a.n_q):
        good = [int(s) for s, sc in zip(a.idx[t], a.sel_score[t]) if s >= 0 and sc != -np.inf]
        kept[t, :len(good)] = good[::-1]
    out2, lse2 = oracle.sparse_attn(a.qa_bits, a.kv_bits, kept, None, a.Ha, a.Dc, a.scale)
    assert np.allclose(out, out2, rtol=0, atol=1e-12) and np.allclose(lse, lse2, rtol=0, atol=1e-12)
    # an index past n_kv counts as no selection too
    bad = kept.copy()
    bad[:, -1] = a.n_kv + 5
    out3, _ = oracle.sparse_attn(a.qa_bits, a.kv_bits, bad, None, a.Ha, a.Dc, a.scale)
    assert np.allclose(out3, out2, rtol=0, atol=1e-12)


def test_no_selection_gives_zeros_and_minus_inf():
    a = li.attn_inputs("x", 2, 100, 2, 16, 8, seed=4)
    idx = a.idx.copy()
    idx[1] = -1
    sc = a.sel_score.copy()
    sc[0] = -np.inf
    out, lse = oracle.sparse_attn(a.qa_bits, a.kv_bits, idx, sc, a.Ha, a.Dc, a.scale)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_dominant_score_selects_its_row():
    Dc = 16
    rng = np.random.default_rng(5)
    kv = rng.integers(-3, 4, (50, Dc)).astype(np.float32)
    qa = np.zeros((1, 1, Dc), np.float32)
    qa[0, 0] = kv[17]
    idx = np.array([[3, 17, 9, 40, 22]], np.int32)
    s = kv[idx[0]].astype(np.float64) @ kv[17].astype(np.float64)
    assert np.argmax(s) == 1 and np.sort(s)[-1] - np.sort(s)[-2] >= 1.0
    out, _ = oracle.sparse_attn(_bf16(qa), _bf16(kv), idx, None, 1, Dc, 60.0)  # weights of the others < e^-60
    assert np.allclose(out[0, 0], kv[17], rtol=0, atol=1e-20 + 1e-12 * np.abs(kv).max())


def test_reduces_to_scipy_softmax_attention():
    special = pytest.importorskip("scipy.special")
    a = li.attn_inputs("x", 5, 400, 4, 48, 40, seed=6, n_invalid=3)
    out, lse = oracle.sparse_attn(a.qa_bits, a.kv_bits, a.idx, a.sel_score, a.Ha, a.Dc, a.scale)
    q = _dec(a.qa_bits)
    k = _dec(a.kv_bits)
    for t in range(a.n_q):
        sel = [int(s) for s, sc in zip(a.idx[t], a.sel_score[t]) if s >= 0 and sc != -np.inf]
        K = k[sel]
        for h in range(a.Ha):
            logits = a.scale * (K @ q[t, h])
            p = special.softmax(logits)
            assert np.allclose(out[t, h], p @ K, rtol=1e-12, atol=1e-12)
            assert lse[t, h] == pytest.approx(special.logsumexp(logits), rel=1e-12, abs=1e-12)


def test_heads_and_rows_use_their_own_queries():
    """Distinct one-hot queries per (t, h) pick distinct closed-form rows."""
    Dc, Ha = 8, 2
    kv = np.zeros((6, Dc), np.float32)
    for s in range(6):
        kv[s, s] = 1.0
    qa = np.zeros((2, Ha, Dc), np.float32)
    qa[0, 0, 0] = qa[0, 1, 1] = qa[1, 0, 2] = qa[1, 1, 3] = 1.0
    idx = np.array([[0, 1, 2, 3], [0, 1, 2, 3]], np.int32)
    out, _ = oracle.sparse_attn(_bf16(qa), _bf16(kv), idx, None, Ha, Dc, 100.0)
    for t, h, s in ((0, 0, 0), (0, 1, 1), (1, 0, 2), (1, 1, 3)):
        assert np.allclose(out[t, h], kv[s], atol=1e-12)
