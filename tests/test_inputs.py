"""The seeded input generator: determinism, published SplitMix64 values, encodings, masks."""
import numpy as np
import torch

import lid_inputs as li


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of Vigna's reference generator
    # (next() adds the golden gamma before mixing), as widely tabulated.
    v = li.splitmix64(0, 0, 3)
    assert [int(x) for x in v] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_offsets_agree():
    a = li.splitmix64(123, 0, 100)
    b = li.splitmix64(123, 37, 20)
    assert np.array_equal(a[37:57], b)


def test_normal_moments_and_determinism():
    x = li.normal(5, 200_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.array_equal(x[:1000], li.normal(5, 1000))
    y = li.normal(5, 200_000, std=0.125)
    assert abs(y.std() - 0.125) < 0.002


def test_uniform_int_range_inclusive():
    x = li.uniform_int(7, 100_000, -3, 3)
    assert x.min() == -3 and x.max() == 3
    counts = np.bincount(x + 3)
    assert counts.min() > 13_000


def test_bf16_rounding_matches_torch():
    x = li.normal(11, 50_000).astype(np.float32) * 37.0
    ours = li.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_masks():
    m = li.causal_mask(4, 2048, 2044)
    assert m.dtype == np.uint16 and m.shape == (4, 2048)
    for t in range(4):
        assert np.all(m[t, :2045 + t] == 0) and np.all(m[t, 2045 + t:] == 0xFC00)
    r = li.range_mask(4, 64, 16)
    assert np.array_equal((r == 0).sum(axis=1), [16] * 4)
    assert np.all(r[2, 32:48] == 0) and np.all(r[2, :32] == 0xFC00)


def test_tiny_workload_recipe():
    inp = li.workload("tiny")
    assert inp.q_bits.shape == (4, 8, 64) and inp.k_bits.shape == (2048, 64)
    q = inp.q_bits.view(np.float16).astype(np.float64)
    assert set(np.unique(q)) <= set(range(-3, 4))
    assert set(np.unique(inp.w)) <= {0.0, 1.0, 2.0, 3.0}
    assert np.array_equal(inp.q_bits, li.workload("tiny").q_bits)


def test_ranges_describe_the_same_masks():
    """The per-row ranges that lid_topk_ranges takes are the dense masks of the
    workloads, written as [lo, hi) (checked where the mask is small enough)."""
    for name in ("tiny", "decode", "prefill", "multiseq"):
        inp = li.workload(name)
        lo, hi = li.workload_ranges(name)
        m = li.mask_from_ranges(lo, hi, inp.n_kv)
        expect = np.zeros((inp.n_q, inp.n_kv), np.uint16) if inp.mask is None else inp.mask
        assert np.array_equal(m, expect), name
    lo, hi = li.causal_ranges(3, 10)
    assert np.array_equal(li.mask_from_ranges(lo, hi, 16), li.causal_mask(3, 16, 10))
    # clamping: negative lo, hi past the end, empty range
    m = li.mask_from_ranges(np.array([-5, 3, 7], np.int32), np.array([2, 99, 7], np.int32), 8)
    assert list(m[0] == 0) == [True, True] + [False] * 6
    assert list(m[1] == 0) == [False] * 3 + [True] * 5
    assert not (m[2] == 0).any()


def test_e4m3_codes_match_torch_rounding():
    # nearest E4M3 value, ties to even, sign kept; includes exact ties, subnormals,
    # zeros of both signs and magnitudes past the largest finite value (saturated)
    import torch
    x = (li.normal(7, 1 << 16) * 40).astype(np.float32)
    edge = np.array([0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11, -2.0 ** -10, 448, 464, 1e6, -1e6,
                     1.0625, 1.1875, 17.0, 19.0], np.float32)  # 2^-10, 1.0625, 17: ties
    x = np.concatenate([x, edge])
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = li.e4m3_codes(x)
    assert np.array_equal(got, ref)
    assert li.e4m3_codes(np.float32(1.0625)) == 0x38 and li.e4m3_codes(np.float32(1.1875)) == 0x3A


def test_e4m3_workload_recipe():
    inp = li.e4m3_inputs("x", 2, 300, 8, 128, 16, seed=3)
    assert inp.dtype == "e4m3" and inp.q_bits.dtype == np.uint8 and inp.k_bits.dtype == np.uint8
    assert inp.q_scale.shape == (2, 8) and inp.k_scale.shape == (300,)
    assert inp.q_scale.dtype == np.float32 and np.all(inp.k_scale > 0)
    assert not np.any((inp.k_bits & 0x7F) == 0x7F)  # no NaN codes
    # same draws as the bf16 form: the scale is each row's amax / 448 of those values
    k = li.normal(li.stream_seed(3, li.STREAM_K), 300 * 128).astype(np.float32).reshape(300, 128)
    assert np.array_equal(inp.k_scale, np.abs(k).max(axis=1) / np.float32(448))
    again = li.e4m3_inputs("x", 2, 300, 8, 128, 16, seed=3)
    assert np.array_equal(again.k_bits, inp.k_bits) and np.array_equal(again.q_scale, inp.q_scale)
    assert li.SHAPES["decode_e4m3"] == li.SHAPES["decode"]
    assert [np.array_equal(a, b) for a, b in zip(li.workload_ranges("multiseq_e4m3"),
                                                 li.workload_ranges("multiseq"))] == [True, True]


def test_integer_e4m3_inputs_are_exact_small_integers_and_powers_of_two():
    import torch
    inp = li.int_e4m3_inputs("i", 3, 200, 16, 128, 8, seed=9)
    qv = torch.from_numpy(inp.q_bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert set(np.unique(qv).tolist()) <= set(range(-3, 4))
    for s in (inp.q_scale, inp.k_scale):
        m, e = np.frexp(s)
        assert np.all(m == 0.5) and np.all((e - 1 >= -2) & (e - 1 <= 2))
