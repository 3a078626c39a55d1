"""Pins of the fp64 CPU oracle against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped ReLU, a
wrong sign, a head weight paired with the wrong head, a transposed q/k
operand, a wrong tie order, a dropped mask or padding) fails at least one of
them; `test_oracle_mutants.py` plants such slips in a copy of the oracle and
checks exactly that.

Definition pinned (llama.cpp issue 25468, root-cause comment; llama.cpp PR
22378, collapse-Q revert commit; fairydreaming/llama.cpp PR 2, API note):
    I[t,s] = sum_h w[t,h] relu(q[t,h,:] . k[s,:]) + mask[t,s], top_k per t.
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
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _brute_as_arrays(res):
    idx = np.array([[i for i, _ in row] for row in res], dtype=np.int64)
    sc = np.array([[(-math.inf if v is None else float(v)) for _, v in row] for row in res])
    return idx, sc


def _random_tiny(seed, dtype, n_q, n_kv, H, D, top_k, kind):
    rng = np.random.default_rng(seed)
    if kind == "int":
        q = rng.integers(-3, 4, size=(n_q, H, D)).astype(np.float32)
        k = rng.integers(-3, 4, size=(n_kv, D)).astype(np.float32)
        w = rng.integers(-3, 4, size=(n_q, H)).astype(np.float32)
    else:
        q = rng.standard_normal((n_q, H, D)).astype(np.float32)
        k = rng.standard_normal((n_kv, D)).astype(np.float32)
        w = (rng.standard_normal((n_q, H)) / math.sqrt(H)).astype(np.float32)
    enc = li.f16_bits if dtype == "f16" else li.f32_to_bf16_bits
    # mask: mostly 0, some -inf, some other finite f16 values (simply added)
    r = rng.random((n_q, n_kv))
    mvals = li.f16_bits(rng.integers(-4, 5, size=(n_q, n_kv)).astype(np.float32) * 0.5)
    mask = np.where(r < 0.25, np.uint16(NEG_INF), np.where(r < 0.4, mvals, np.uint16(0))).astype(np.uint16)
    return enc(q), enc(k), w, mask


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("kind", ["int", "float"])
def test_oracle_matches_exact_brute_force(seed, dtype, kind):
    n_q, n_kv, H, D = 3, 40 + seed, 1 + seed % 4, 4 + 2 * (seed % 3)
    top_k = [5, 17, 64][seed % 3]  # includes top_k > n_kv (padding)
    q, k, w, mask = _random_tiny(seed, dtype, n_q, n_kv, H, D, top_k, kind)
    if seed % 2:
        mask = None
    bi, bs = _brute_as_arrays(brute.topk(q, k, w, mask, n_q, n_kv, H, D, top_k, dtype))
    oi, os_ = oracle.topk(q, k, w, mask, H, D, top_k, dtype)
    assert np.array_equal(oi, bi)
    fin = np.isfinite(bs)
    assert np.array_equal(np.isfinite(os_), fin)
    # integer inputs are exact in fp64; float inputs round once per product/sum
    tol = 0.0 if kind == "int" else 1e-12
    assert np.all(np.abs(os_[fin] - bs[fin]) <= tol * np.maximum(1.0, np.abs(bs[fin])))


def test_oracle_score_rows_match_brute_force():
    q, k, w, mask = _random_tiny(99, "bf16", 2, 30, 3, 6, 8, "float")
    exact = brute.score_rows(q, k, w, mask, 2, 30, 3, 6, "bf16")
    got = oracle.scores(q, k, w, mask, 3, 6, "bf16")
    for t in range(2):
        for s in range(30):
            if exact[t][s] is None:
                assert got[t, s] == -math.inf
            else:
                assert got[t, s] == pytest.approx(float(exact[t][s]), rel=1e-13, abs=1e-13)


def test_decode_f16_matches_numpy_on_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in range(0, 65536, 1):
        r = ref[b]
        if np.isnan(r):
            continue
        got = oracle.decode_f16(b)
        assert got == r, hex(b)


def test_decode_bf16_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for b, r in zip(bits, ref):
        if np.isnan(r):
            continue
        assert oracle.decode_bf16(int(b)) == r


# ---------------------------------------------------------------- hand cases

def _one_row(n_kv, H, D):
    return (np.zeros((1, H, D), np.uint16), np.zeros((n_kv, D), np.uint16), np.zeros((1, H), np.float32))


def test_all_masked_row_takes_lowest_indices_with_neg_inf():
    q, k, w = _one_row(100, 2, 4)
    q[:] = li.f32_to_bf16_bits(np.ones((1, 2, 4), np.float32))
    k[:] = li.f32_to_bf16_bits(np.arange(400, dtype=np.float32).reshape(100, 4))
    w[:] = 1.0
    mask = np.full((1, 100), NEG_INF, np.uint16)
    idx, sc = oracle.topk(q, k, w, mask, 2, 4, 10)
    assert list(idx[0]) == list(range(10))
    assert np.all(sc == -math.inf)


def test_zero_weights_give_first_indices_with_zero_score():
    q, k, w = _one_row(50, 3, 4)
    q[:] = li.f32_to_bf16_bits(np.full((1, 3, 4), 2.0, np.float32))
    k[:] = li.f32_to_bf16_bits(np.full((50, 4), 1.5, np.float32))
    idx, sc = oracle.topk(q, k, w, None, 3, 4, 8)
    assert list(idx[0]) == list(range(8)) and np.all(sc == 0.0)


def test_fewer_keys_than_top_k_pads_with_minus_one():
    q, k, w = _one_row(5, 1, 2)
    q[:] = li.f32_to_bf16_bits(np.array([[[1.0, 0.0]]], np.float32))
    k[:] = li.f32_to_bf16_bits(np.array([[3, 0], [1, 0], [4, 0], [1, 0], [5, 0]], np.float32))
    w[:] = 1.0
    idx, sc = oracle.topk(q, k, w, None, 1, 2, 8)
    assert list(idx[0]) == [4, 2, 0, 1, 3, -1, -1, -1]
    assert list(sc[0]) == [5, 4, 3, 1, 1] + [-math.inf] * 3


def test_ties_order_by_index():
    """Equal scores (here all the zero-ReLU keys) come out lowest index first."""
    q, k, w = _one_row(6, 1, 2)
    q[:] = li.f32_to_bf16_bits(np.array([[[1.0, 0.0]]], np.float32))
    k[:] = li.f32_to_bf16_bits(np.array([[0, 1], [0, 2], [-1, 0], [0, 0], [2, 0], [0, 5]], np.float32))
    w[:] = -1.0
    idx, sc = oracle.topk(q, k, w, None, 1, 2, 6)
    # key 4 has dot 2 -> score -2; every other key scores zero and they tie
    assert list(idx[0]) == [0, 1, 2, 3, 5, 4]
    assert list(sc[0]) == [0, 0, 0, 0, 0, -2]


def test_masked_keys_rank_after_every_finite_score():
    q, k, w = _one_row(8, 1, 1)
    q[:] = li.f16_bits(np.ones((1, 1, 1), np.float32))
    k[:] = li.f16_bits(np.array([[-3], [2], [-1], [7], [0], [1], [-2], [5]], np.float32))
    w[:] = 1.0
    mask = np.zeros((1, 8), np.uint16)
    mask[0, [3, 7]] = NEG_INF
    mask[0, 1] = li.f16_bits(np.array([-10.0], np.float32))[0]  # finite mask values are added
    idx, sc = oracle.topk(q, k, w, mask, 1, 1, 8, dtype="f16")
    # relu scores: [0,2,0,7,0,1,0,5] + mask -> [0,-8,0,-inf,0,1,0,-inf]
    assert list(idx[0]) == [5, 0, 2, 4, 6, 1, 3, 7]
    assert list(sc[0]) == [1, 0, 0, 0, 0, -8, -math.inf, -math.inf]


# ------------------------------------------------ textbook reductions / closed forms

def test_single_head_unit_weight_is_topk_of_relu_matmul():
    """H=1, w=1, no mask: the top-k of relu(k q), i.e. a matrix product followed
    by numpy's stable argsort on (-score) -- a library routine."""
    n_kv, D, top_k = 3000, 16, 100
    rng = np.random.default_rng(3)
    q = li.f32_to_bf16_bits(rng.standard_normal((1, 1, D)).astype(np.float32))
    k = li.f32_to_bf16_bits(rng.standard_normal((n_kv, D)).astype(np.float32))
    w = np.ones((1, 1), np.float32)
    qf = torch.from_numpy(q.view(np.int16).copy()).view(torch.bfloat16).double().numpy().reshape(D)
    kf = torch.from_numpy(k.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    ref = np.maximum(kf @ qf, 0.0)
    order = np.argsort(-ref, kind="stable")[:top_k]
    idx, sc = oracle.topk(q, k, w, None, 1, D, top_k)
    assert np.array_equal(idx[0], order)
    assert np.allclose(sc[0], ref[order], rtol=1e-14, atol=0)


def test_one_hot_queries_closed_form():
    """Head 0 reads feature 0, head 1 reads feature 1 (one-hot q), so
    I[s] = w0 relu(k[s,0]) + w1 relu(k[s,1]) in closed form."""
    n_kv = 97
    f = [(s * 7) % 13 - 6 for s in range(n_kv)]
    g = [(s * 5) % 11 - 4 for s in range(n_kv)]
    k = np.zeros((n_kv, 4), np.float32)
    k[:, 0], k[:, 1], k[:, 2] = f, g, 100.0  # feature 2 must not leak in
    q = np.zeros((1, 2, 4), np.float32)
    q[0, 0, 0] = 1.0
    q[0, 1, 1] = 1.0
    w = np.array([[3.0, -2.0]], np.float32)
    expect = [3 * max(f[s], 0) - 2 * max(g[s], 0) for s in range(n_kv)]
    order = sorted(range(n_kv), key=lambda s: (-expect[s], s))[:20]
    idx, sc = oracle.topk(li.f16_bits(q), li.f16_bits(k), w, None, 2, 4, 20, dtype="f16")
    assert list(idx[0]) == order
    assert list(sc[0]) == [expect[s] for s in order]


# ------------------------------------------------------------------- invariants

def test_positive_scaling_of_w_keeps_indices():
    """The older API's 1/sqrt(D) and 1/sqrt(H) factors (llama.cpp issue 25468,
    fused-op comment) were dropped later (fairydreaming/llama.cpp PR 2): a
    positive scale changes scores, not the selection."""
    inp = li.float_inputs("t", 3, 700, 8, 32, 50, seed=4)
    i0, s0 = oracle.topk_inputs(inp)
    for c in (0.125, 1.0 / 64, 4.0):  # powers of two: exact scaling
        i1, s1 = oracle.topk(inp.q_bits, inp.k_bits, inp.w * np.float32(c), None, 8, 32, 50)
        assert np.array_equal(i0, i1)
        assert np.array_equal(s1, s0 * c)


def test_key_permutation_permutes_indices():
    inp = li.float_inputs("t", 2, 500, 4, 16, 40, seed=8)
    perm = np.random.default_rng(0).permutation(500)
    i0, s0 = oracle.topk_inputs(inp)
    i1, s1 = oracle.topk(inp.q_bits, inp.k_bits[perm], inp.w, None, 4, 16, 40)
    inv = np.argsort(perm)
    assert np.array_equal(perm[i1], i0) and np.array_equal(s0, s1)
    assert np.array_equal(i1, inv[i0])


def test_collapse_q_is_not_the_method():
    """llama.cpp PR 22378 reverts collapse-Q (summing q and w over queries
    before the contraction) because ReLU does not commute with the sum. The
    oracle must select per query, so its result differs on this case."""
    q = np.array([[[1.0, 0.0]], [[-1.0, 0.0]]], np.float32)  # two queries, one head
    k = np.array([[2.0, 0.0], [-3.0, 0.0], [0.0, 1.0]], np.float32)
    w = np.ones((2, 1), np.float32)
    idx, sc = oracle.topk(li.f16_bits(q), li.f16_bits(k), w, None, 1, 2, 1, dtype="f16")
    assert list(idx[:, 0]) == [0, 1]  # per query: key 0 for t=0, key 1 for t=1
    # collapse-Q: sum_q q = 0 -> all dots 0 -> key 0 for both queries
    qsum = q.sum(axis=0)
    collapsed = np.maximum(k @ qsum[0], 0) * w.sum()
    assert int(np.argsort(-collapsed, kind="stable")[0]) == 0
    assert list(idx[:, 0]) != [0, 0]


def test_shape_reading_reproduces_the_reported_buffer_sizes():
    """llama.cpp issue 25468, root-cause comment: lid_kq is 4096 MiB per CSA
    layer at ctx 131072 and 512 MiB at ctx 16384 (ubatch 512), lid_score is
    64 MiB and lid_top_k 1 MiB; the indexer cache is 168 MiB at ctx 131072
    (KV-cache comment). Read as: compression ratio 4, H = 64 heads, f32
    scores, int32 indices, k = 512, D = 128 two-byte features over 21 layers."""
    MiB = 1 << 20
    for ctx, want in ((131072, 4096), (16384, 512)):
        assert (ctx // 4) * 64 * 512 * 4 == want * MiB
    assert (131072 // 4) * 512 * 4 == 64 * MiB
    assert 512 * 512 * 4 == 1 * MiB
    assert 21 * (131072 // 4) * 128 * 2 == 168 * MiB


# --------------------------------------------------------------------- golden

def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            rows[key.strip()] = vals.split()
    return rows


def test_hand_worked_golden_example():
    """tests/golden/hand_worked.txt is computed by hand (see the file)."""
    g = _read_golden("hand_worked.txt")
    q = np.array([float(x) for x in g["q"]], np.float32).reshape(1, 2, 2)
    k = np.array([float(x) for x in g["k"]], np.float32).reshape(-1, 2)
    w = np.array([float(x) for x in g["w"]], np.float32).reshape(1, 2)
    mask = li.f16_bits(np.array([float(x) for x in g["mask"]], np.float32)).reshape(1, -1)
    top_k = int(g["top_k"][0])
    idx, sc = oracle.topk(li.f16_bits(q), li.f16_bits(k), w, mask, 2, 2, top_k, dtype="f16")
    assert [int(x) for x in g["idx"]] == list(idx[0])
    assert [float(x) for x in g["score"]] == list(sc[0])


def test_tiny_workload_golden():
    """tests/golden/tiny_topk.txt was written by tests/golden/make_golden.py
    (oracle only) and guards the oracle against silent changes."""
    g = _read_golden("tiny_topk.txt")
    inp = li.workload("tiny")
    idx, sc = oracle.topk_inputs(inp)
    for t in range(inp.n_q):
        assert [int(x) for x in g[f"idx{t}"]] == list(idx[t])
        assert [float(x) for x in g[f"score{t}"]] == list(sc[t])
