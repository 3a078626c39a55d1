"""Property test of the oracle against exact brute force over random tiny
shapes (hypothesis): every operand form (bf16, f16, E4M3 with row scales),
masks with -inf and other finite values, negative weights, top_k above and
below n_kv. Integer-valued operands make every fp64 step exact, so indices and
scores must be equal, not close."""
import math

import numpy as np
import pytest

import lid_inputs as li
import oracle
from oracle import brute

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def cases(draw):
    form = draw(st.sampled_from(["bf16", "f16", "e4m3"]))
    n_q = draw(st.integers(1, 3))
    n_kv = draw(st.integers(0, 24))
    H = draw(st.integers(1, 4))
    D = draw(st.integers(1, 6))
    top_k = draw(st.integers(1, 30))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return form, n_q, n_kv, H, D, top_k, seed


def _arrays(form, n_q, n_kv, H, D, seed):
    rng = np.random.default_rng(seed)
    qv = rng.integers(-3, 4, size=(n_q, H, D)).astype(np.float32)
    kv = rng.integers(-3, 4, size=(n_kv, D)).astype(np.float32)
    w = rng.integers(-3, 4, size=(n_q, H)).astype(np.float32)
    r = rng.random((n_q, n_kv))
    mask = np.where(r < 0.25, np.uint16(0xFC00),
                    np.where(r < 0.4, li.f16_bits(np.float32(-2.5)), np.uint16(0))).astype(np.uint16)
    if form == "e4m3":
        qs = np.exp2(rng.integers(-3, 3, size=(n_q, H))).astype(np.float32)
        ks = np.exp2(rng.integers(-3, 3, size=n_kv)).astype(np.float32)
        return (li.e4m3_codes(qv), qs, li.e4m3_codes(kv), ks), w, mask
    enc = li.f16_bits if form == "f16" else li.f32_to_bf16_bits
    return (enc(qv), enc(kv)), w, mask


@hypothesis.settings(max_examples=80, deadline=None)
@hypothesis.given(cases())
def test_oracle_equals_brute_force_on_random_tiny_cases(case):
    form, n_q, n_kv, H, D, top_k, seed = case
    ops, w, mask = _arrays(form, n_q, n_kv, H, D, seed)
    if form == "e4m3":
        q8, qs, k8, ks = ops
        exact = brute.topk_e4m3(q8, qs, k8, ks, w, mask, n_q, n_kv, H, D, top_k)
        oi, os_ = oracle.topk_e4m3(q8, qs, k8, ks, w, mask, H, D, top_k)
    else:
        q, k = ops
        exact = brute.topk(q, k, w, mask, n_q, n_kv, H, D, top_k, form)
        oi, os_ = oracle.topk(q, k, w, mask, H, D, top_k, form)
    bi = np.array([[i for i, _ in row] for row in exact], dtype=np.int64)
    bs = np.array([[(-math.inf if v is None else float(v)) for _, v in row] for row in exact])
    assert np.array_equal(oi, bi)
    assert np.array_equal(os_, bs)
