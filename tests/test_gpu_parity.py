"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Bit-exact on integer-valued inputs; within the stated tolerance on float
inputs (see tests/parity.py). Covers every supported H and D, both dtypes,
ragged key counts and query groups, forced and planned key splits, the
edge cases of the method, the five workload shapes at full size (sampled
rows), the host-buffer entry point, and the error paths.
"""
import ctypes

import numpy as np
import pytest
import torch

import lid_inputs as li
import oracle
import sparse_attention_lightning_lid_gb300 as lid
from tests.parity import check_exact, check_tolerance, run_gpu, to_device

pytestmark = pytest.mark.gpu

NEG_INF = np.uint16(0xFC00)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lid.load()
    lid.device_error(reset=True)
    yield
    assert lid.device_error() == 0, "a bounded device-side wait timed out during the tests"


def _random_mask(n_q, n_kv, seed, p_inf=0.3):
    rng = np.random.default_rng(seed)
    m = np.where(rng.random((n_q, n_kv)) < p_inf, NEG_INF, np.uint16(0)).astype(np.uint16)
    # keep at least a few visible keys per row
    m[:, :4] = 0
    return m


def _mask(kind, n_q, n_kv, seed):
    if kind == "none":
        return None
    if kind == "causal":
        return li.causal_mask(n_q, n_kv, max(0, n_kv - n_q))
    return _random_mask(n_q, n_kv, seed)


INT_CASES = [
    # H, D, dtype, n_q, n_kv, top_k, splits, mask, w_range
    (8, 64, "f16", 4, 2048, 64, 0, "causal", (0, 3)),
    (64, 128, "bf16", 1, 5000, 512, 0, "none", (0, 3)),
    (64, 128, "bf16", 5, 3001, 100, 1, "random", (-3, 3)),
    (64, 128, "f16", 9, 4099, 512, 4, "causal", (0, 3)),
    (32, 128, "bf16", 7, 1000, 256, 0, "random", (-3, 3)),
    (16, 64, "f16", 20, 2500, 33, 3, "causal", (0, 3)),
    (8, 128, "bf16", 1, 777, 64, 0, "none", (-3, 3)),
    (64, 64, "bf16", 3, 130, 2048, 0, "none", (0, 3)),
    (64, 128, "bf16", 2, 100, 1, 0, "none", (0, 3)),
    (8, 64, "f16", 33, 640, 16, 2, "random", (0, 3)),
    (64, 128, "bf16", 4, 20000, 512, 0, "random", (-3, 3)),
    (32, 64, "f16", 3, 9000, 1000, 5, "none", (0, 3)),
]


@pytest.mark.parametrize("case", INT_CASES, ids=[f"H{c[0]}D{c[1]}{c[2]}q{c[3]}kv{c[4]}k{c[5]}s{c[6]}{c[7]}"
                                                 for c in INT_CASES])
def test_integer_inputs_bit_exact(case):
    H, D, dtype, n_q, n_kv, top_k, splits, mkind, wr = case
    inp = li.int_inputs("int", n_q, n_kv, H, D, top_k, seed=n_kv + H, mask=_mask(mkind, n_q, n_kv, n_kv),
                        dtype=dtype, w_range=wr)
    opt = lid.Options(force_splits=splits) if splits else None
    g_idx, g_sc = run_gpu(inp, options=opt)
    check_exact(g_idx, g_sc, inp)


def test_tiny_workload_bit_exact():
    inp = li.workload("tiny")
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)


@pytest.mark.parametrize("splits", [0, 1, 3, 40])
def test_float_prefill_shape_all_rows(splits):
    inp = li.float_inputs("f", 40, 6000, 64, 128, 512, seed=3, mask=li.causal_mask(40, 6000, 5960))
    opt = lid.Options(force_splits=splits) if splits else None
    g_idx, g_sc = run_gpu(inp, options=opt)
    check_tolerance(g_idx, g_sc, inp, range(inp.n_q))


def test_float_small_heads_and_f16():
    inp = li.float_inputs("f", 6, 3000, 16, 64, 128, seed=5, mask=_random_mask(6, 3000, 1))
    g_idx, g_sc = run_gpu(inp)
    check_tolerance(g_idx, g_sc, inp, range(inp.n_q))


@pytest.mark.parametrize("splits", [512, 64])
def test_many_splits_merge(splits):
    """The merge at its largest split count, and with most splits fully masked
    for each query (as when sequences share one key cache)."""
    n_q, n_kv = 4, 65536
    inp = li.float_inputs("s", n_q, n_kv, 64, 128, 512, seed=21, mask=li.range_mask(n_q, n_kv, n_kv // n_q))
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=splits))
    check_tolerance(g_idx, g_sc, inp, range(n_q))
    inp = li.int_inputs("s", 2, n_kv, 64, 128, 300, seed=22, dtype="bf16", w_range=(-3, 3))
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=splits))
    check_exact(g_idx, g_sc, inp)



def test_ranked_merge_of_a_few_lists():
    """The merge of a few per-split lists (each key placed by its count of
    larger keys): fewer keys than top_k (padded lists and rows), its largest
    list count and total, and one split more (the general merge)."""
    inp = li.int_inputs("r", 3, 300, 64, 128, 512, seed=31, dtype="bf16")
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=3))
    check_exact(g_idx, g_sc, inp)
    assert np.all(g_idx[:, 300:] == -1) and np.all(np.isneginf(g_sc[:, 300:]))
    inp = li.int_inputs("r", 2, 5000, 64, 128, 2048, seed=32, dtype="bf16", w_range=(-3, 3))
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=2))
    check_exact(g_idx, g_sc, inp)
    inp = li.float_inputs("r", 5, 9000, 64, 128, 512, seed=33, mask=li.causal_mask(5, 9000, 8995))
    for splits in (8, 9):
        g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=splits))
        check_tolerance(g_idx, g_sc, inp, range(5))

# ------------------------------------------------------------ edge cases

def test_ascending_scores_force_constant_compaction():
    """Each key beats every earlier one: every tile inserts into the candidate
    buffer and the radix-select compaction runs over and over."""
    n_kv, H, D = 2048, 64, 64
    k = np.zeros((n_kv, D), np.float32)
    k[:, 0] = np.arange(n_kv)
    q = np.zeros((2, H, D), np.float32)
    q[0, :, 0] = 1.0
    q[1, :, 0] = -1.0  # second query: all scores zero -> ties, lowest indices
    inp = li.Inputs("asc", "f16", 2, n_kv, H, D, 512, li.f16_bits(q), li.f16_bits(k),
                    np.ones((2, H), np.float32), None)
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=1))
    check_exact(g_idx, g_sc, inp)
    assert list(g_idx[0, :3]) == [2047, 2046, 2045]
    assert list(g_idx[1, :3]) == [0, 1, 2]


def test_all_masked_rows_and_zero_weights():
    inp = li.int_inputs("m", 3, 1500, 64, 128, 200, seed=2, dtype="bf16")
    inp.mask = np.zeros((3, 1500), np.uint16)
    inp.mask[0, :] = NEG_INF            # every key masked: lowest indices, -inf
    inp.mask[1, 700:] = NEG_INF         # fewer visible keys than... still > top_k
    inp.w[2, :] = 0.0                   # all scores 0: lowest indices
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)
    assert list(g_idx[0]) == list(range(200)) and np.all(np.isneginf(g_sc[0]))
    assert list(g_idx[2]) == list(range(200)) and np.all(g_sc[2] == 0)


def test_fewer_visible_than_top_k():
    inp = li.int_inputs("m", 2, 3000, 64, 128, 512, seed=4, dtype="bf16")
    inp.mask = np.full((2, 3000), NEG_INF, np.uint16)
    inp.mask[0, 100:400] = 0  # 300 visible keys, then masked keys by index
    inp.mask[1, 2990:] = 0
    g_idx, g_sc = run_gpu(inp, options=lid.Options(force_splits=3))
    check_exact(g_idx, g_sc, inp)


def test_no_keys_gives_padding():
    q = torch.zeros((3, 64, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((3, 64), dtype=torch.float32, device="cuda")
    idx, sc = lid.topk(q, k, w, None, 16)
    torch.cuda.synchronize()
    assert torch.all(idx == -1) and torch.all(torch.isneginf(sc))


def test_no_queries_is_a_no_op():
    q = torch.zeros((0, 64, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    idx, sc = lid.topk(q, k, w, None, 16)
    assert idx.shape == (0, 16)


def test_max_top_k_and_tiny_key_count():
    inp = li.int_inputs("k", 2, 5000, 64, 128, 2048, seed=9, dtype="bf16", w_range=(-3, 3))
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)
    inp = li.int_inputs("k", 3, 7, 8, 64, 16, seed=9, dtype="f16")
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)


def test_side_stream_and_determinism():
    inp = li.float_inputs("d", 8, 8192, 64, 128, 512, seed=11, mask=_random_mask(8, 8192, 3))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = run_gpu(inp, stream=s)
        b = run_gpu(inp, stream=s)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    check_tolerance(a[0], a[1], inp, range(8))


def test_host_buffer_entry_point():
    inp = li.workload("tiny")
    idx, sc = lid.topk_host(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.top_k, dtype="f16")
    check_exact(idx, sc, inp)
    inp = li.float_inputs("h", 5, 5000, 64, 128, 256, seed=12, mask=li.causal_mask(5, 5000, 4995))
    idx, sc = lid.topk_host(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.top_k)
    check_tolerance(idx, sc, inp, range(5))


def test_host_async_two_streams():
    # several calls in flight, each with its own pinned result buffers: every one of them equals
    # the synchronous host call, which the oracle checks
    inp = li.float_inputs("ha", 6, 9000, 64, 128, 256, seed=13, mask=li.causal_mask(6, 9000, 8994))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hq = pin(inp.q_bits.view(np.int16))
    hk = pin(inp.k_bits.view(np.int16))
    hw = pin(inp.w)
    hm = pin(inp.mask.view(np.int16))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ref_i, ref_s = lid.topk_host(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.top_k)
    check_tolerance(ref_i, ref_s, inp, range(6))
    # five calls back to back on one stream (the library's copy stream runs ahead of it, with at most
    # three calls' staging alive), then five alternating between two streams
    for pick in (lambda i: streams[0], lambda i: streams[i % 2]):
        outs = [(torch.full((6, 256), -7, dtype=torch.int32).pin_memory(),
                 torch.full((6, 256), 7.0, dtype=torch.float32).pin_memory()) for _ in range(5)]
        for i, (oi, os_) in enumerate(outs):
            lid.topk_host_async(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, oi, os_, stream=pick(i))
        for s in streams:
            s.synchronize()
        for oi, os_ in outs:
            assert np.array_equal(oi.numpy(), ref_i) and np.array_equal(os_.numpy(), ref_s)



def test_host_async_recorded_in_a_graph():
    # inside a stream capture the copies stay on the captured stream: a graph of the call,
    # replayed, copies the pinned inputs in and the result out each time
    inp = li.float_inputs("hg", 3, 5000, 64, 128, 128, seed=14, mask=li.causal_mask(3, 5000, 4997))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    hq, hk, hw, hm = (pin(inp.q_bits.view(np.int16)), pin(inp.k_bits.view(np.int16)), pin(inp.w),
                      pin(inp.mask.view(np.int16)))
    ref_i, ref_s = lid.topk_host(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.top_k)
    check_tolerance(ref_i, ref_s, inp, range(3))
    oi = torch.empty((3, 128), dtype=torch.int32).pin_memory()
    os_ = torch.empty((3, 128), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    lid.topk_host_async(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, oi, os_, stream=s)  # eager first
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        lid.topk_host_async(hq, hk, hw, hm, inp.H, inp.D, inp.top_k, oi, os_, stream=s)
    for _ in range(2):
        oi.fill_(-7)
        os_.fill_(7.0)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(oi.numpy(), ref_i) and np.array_equal(os_.numpy(), ref_s)
    assert lid.device_error() == 0

# ------------------------------------------------- full-size workload shapes

def _sample_rows(n_q, n):
    if n_q <= n:
        return list(range(n_q))
    rng = np.random.default_rng(0)
    return sorted(set([0, n_q - 1] + rng.choice(n_q, n - 2, replace=False).tolist()))


@pytest.mark.parametrize("name,n_rows,path", [("decode", 1, 0), ("prefill", 512, 0), ("long", 64, 0),
                                              ("multiseq", 4, 0), ("decode", 1, 1), ("multiseq", 4, 1)])
def test_workloads_full_size_sampled(name, n_rows, path):
    """Planned launch configuration (path 0: what bench.py times) and, where
    that is the one-launch path, also the two-launch split merge (path 1).
    Every row of prefill and 64 rows of the long prefill (both ends and 62
    drawn at random) are compared with the oracle; the worst ratio of a score
    error to its tolerance is printed."""
    inp = li.workload(name)
    g_idx, g_sc = run_gpu(inp, options=lid.Options(path=path) if path else None)
    rows = np.arange(inp.n_q) if n_rows >= inp.n_q else _sample_rows(inp.n_q, n_rows)
    worst = check_tolerance(g_idx, g_sc, inp, rows)
    print(f"{name} path {path}: {len(rows)} rows, worst score error / tolerance = {worst:.4f}")
    # properties that hold at any size, on every row
    assert np.all((g_idx >= 0) & (g_idx < inp.n_kv))
    assert np.all(np.diff(g_sc, axis=1) <= 0)
    if inp.mask is not None:
        rows = np.arange(inp.n_q)[:, None]
        assert np.all(inp.mask[rows, g_idx] == 0), "a masked key was selected although enough keys are visible"


def test_workspace_is_never_n_q_by_n_kv():
    for name in li.WORKLOADS:
        n_q, n_kv, H, D, top_k = li.SHAPES[name]
        p = lid.plan(n_q, n_kv, H, D, top_k)
        assert p["workspace_bytes"] < 64 << 20
        assert p["workspace_bytes"] < n_q * n_kv * 4 or n_q * n_kv * 4 < (1 << 20)


# ------------------------------------------------------------ error paths

def _raw_call(q, k, w, mask, n_q, n_kv, H, D, top_k, oi, os_, opt=None, dtype=0):
    L = lid.load()
    return L.lid_topk_ex(q, k, w, mask, n_q, n_kv, H, D, top_k, oi, os_, None, dtype,
                         ctypes.byref(opt) if opt is not None else None)


def test_error_paths_launch_nothing_and_leave_outputs():
    q = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((300, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((2, 64), dtype=torch.float32, device="cuda")
    oi = torch.full((2, 16), 7, dtype=torch.int32, device="cuda")
    os_ = torch.full((2, 16), 3.5, dtype=torch.float32, device="cuda")
    P = lambda t: t.data_ptr()  # noqa: E731
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 12, 128, 16, P(oi), P(os_)) == lid.LID_ERR_UNSUPPORTED
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 64, 96, 16, P(oi), P(os_)) == lid.LID_ERR_UNSUPPORTED
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 64, 128, 0, P(oi), P(os_)) == lid.LID_ERR_UNSUPPORTED
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 64, 128, 4096, P(oi), P(os_)) == lid.LID_ERR_UNSUPPORTED
    assert _raw_call(P(q), P(k), P(w), None, -1, 300, 64, 128, 16, P(oi), P(os_)) == lid.LID_ERR_INVALID_ARG
    assert _raw_call(None, P(k), P(w), None, 2, 300, 64, 128, 16, P(oi), P(os_)) == lid.LID_ERR_INVALID_ARG
    assert _raw_call(P(q) + 2, P(k), P(w), None, 2, 300, 64, 128, 16, P(oi), P(os_)) == lid.LID_ERR_INVALID_ARG
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 64, 128, 16, P(oi), P(os_), dtype=7) == lid.LID_ERR_INVALID_ARG
    opt = lid.Options(force_splits=2, fault_inject=1)
    assert _raw_call(P(q), P(k), P(w), None, 2, 300, 64, 128, 16, P(oi), P(os_), opt) == lid.LID_ERR_OOM
    torch.cuda.synchronize()
    assert torch.all(oi == 7) and torch.all(os_ == 3.5)
    with pytest.raises(lid.LidError):
        lid.topk(q, k, w, None, 0)
    assert "unsupported" in lid.status_string(lid.LID_ERR_UNSUPPORTED)


def test_bounded_device_wait_reports_and_context_survives():
    """Fault injection without faulting the GPU: each scoring CTA's epilogue
    waits on a barrier that nothing completes. The wait gives up after its
    short limit, the CTA aborts cleanly (its MMAs and copies drained), the
    device error word names the stuck role (3: the epilogue's wait; 2: the MMA
    issuer's wait for the epilogue; 1: the copy issuer's wait for the MMA,
    whichever limit runs out first), and the context stays usable."""
    inp = li.int_inputs("f", 4, 3000, 64, 128, 64, seed=41, dtype="bf16")
    q, k, w, m = to_device(inp)
    lid.device_error(reset=True)
    lid.topk(q, k, w, m, inp.top_k, options=lid.Options(force_splits=1, fault_inject=2))
    assert lid.device_error(reset=True) in (1, 2, 3)
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)
    assert lid.device_error() == 0


# ------------------------------------------------- one-launch split path

ONE_LAUNCH_CASES = [
    # H, D, dtype, n_q, n_kv, top_k, splits (0: planned), mask, w_range
    (64, 128, "bf16", 1, 5000, 512, 0, "none", (0, 3)),
    (64, 128, "f16", 9, 4099, 512, 0, "causal", (0, 3)),
    (32, 128, "bf16", 7, 1000, 256, 3, "random", (-3, 3)),
    (16, 64, "f16", 20, 2500, 33, 0, "causal", (0, 3)),
    (8, 64, "f16", 33, 640, 16, 2, "random", (0, 3)),
    (8, 128, "bf16", 1, 777, 64, 0, "none", (-3, 3)),
    (64, 64, "bf16", 3, 2600, 2048, 0, "none", (0, 3)),
    (64, 128, "bf16", 2, 300, 1, 0, "none", (0, 3)),
    (32, 64, "f16", 3, 9000, 1000, 5, "none", (0, 3)),
    (64, 128, "bf16", 1, 131072, 512, 0, "random", (-3, 3)),
    # one query: two epilogue groups stream while two run the early steps; with
    # a forced small split count the candidate buffer needs cuts (one streaming group)
    (64, 128, "bf16", 1, 131072, 512, 8, "none", (0, 3)),
    (32, 64, "f16", 1, 50000, 256, 0, "causal", (0, 3)),
    (16, 64, "bf16", 1, 30000, 128, 0, "none", (-3, 3)),
]


@pytest.mark.parametrize("case", ONE_LAUNCH_CASES,
                         ids=[f"H{c[0]}D{c[1]}{c[2]}q{c[3]}kv{c[4]}k{c[5]}s{c[6]}{c[7]}" for c in ONE_LAUNCH_CASES])
def test_one_launch_path_bit_exact(case):
    H, D, dtype, n_q, n_kv, top_k, splits, mkind, wr = case
    assert lid.plan(n_q, n_kv, H, D, top_k, options=lid.Options(path=2, force_splits=splits))["fused"] >= 1
    inp = li.int_inputs("one", n_q, n_kv, H, D, top_k, seed=n_kv + 7 * H, mask=_mask(mkind, n_q, n_kv, n_kv + 1),
                        dtype=dtype, w_range=wr)
    g_idx, g_sc = run_gpu(inp, options=lid.Options(path=2, force_splits=splits))
    check_exact(g_idx, g_sc, inp)


SINGLE_QUERY_CASES = [c for c in ONE_LAUNCH_CASES if c[3] == 1 and c[0] >= 16]


@pytest.mark.parametrize("case", SINGLE_QUERY_CASES,
                         ids=[f"H{c[0]}D{c[1]}{c[2]}kv{c[4]}k{c[5]}s{c[6]}{c[7]}" for c in SINGLE_QUERY_CASES])
def test_single_query_shapes_on_both_one_launch_kernels(case):
    """One query per CTA: the planned single-query kernel (fused = 2) where
    every key of a CTA fits its buffer, and the general one-launch kernel
    (path 3: early steps, tile-parallel groups, cuts), both bit-exact."""
    H, D, dtype, n_q, n_kv, top_k, splits, mkind, wr = case
    inp = li.int_inputs("sq", n_q, n_kv, H, D, top_k, seed=n_kv + 11 * H, mask=_mask(mkind, n_q, n_kv, n_kv + 2),
                        dtype=dtype, w_range=wr)
    for path in (2, 3):
        opt = lid.Options(path=path, force_splits=splits)
        kind = lid.plan(n_q, n_kv, H, D, top_k, options=opt)["fused"]
        assert kind == (1 if path == 3 else kind) and kind >= 1
        g_idx, g_sc = run_gpu(inp, options=opt)
        check_exact(g_idx, g_sc, inp)


def test_one_launch_degenerate_rows_take_the_histogram_rounds():
    """Rows whose certified bound lets far more than the gather capacity
    through (ties broken by index over tens of thousands of keys), so the
    CTAs narrow the bound with shared digit histograms before gathering."""
    n_q, n_kv = 4, 60000
    inp = li.int_inputs("deg", n_q, n_kv, 64, 128, 512, seed=77, dtype="bf16")
    inp.mask = np.zeros((n_q, n_kv), np.uint16)
    inp.mask[0, :] = NEG_INF            # every key -inf: the 512 lowest indices
    inp.w[1, :] = 0.0                   # every score 0: the 512 lowest indices
    inp.mask[2, :59000] = NEG_INF       # 1000 visible keys at the end, then -inf keys by index
    inp.mask[3, 30000:30100] = NEG_INF  # an ordinary row beside them
    g_idx, g_sc = run_gpu(inp, options=lid.Options(path=2))
    check_exact(g_idx, g_sc, inp)
    assert list(g_idx[0]) == list(range(512)) and list(g_idx[1]) == list(range(512))


def test_one_launch_fewer_keys_than_top_k_pads():
    inp = li.int_inputs("pad", 2, 700, 64, 128, 1024, seed=5, dtype="bf16")
    g_idx, g_sc = run_gpu(inp, options=lid.Options(path=2))
    check_exact(g_idx, g_sc, inp)
    assert np.all(g_idx[:, 700:] == -1) and np.all(np.isneginf(g_sc[:, 700:]))


def test_planned_paths():
    assert lid.plan(*li.SHAPES["decode"])["fused"] == 2           # the single-query kernel
    assert lid.plan(*li.SHAPES["decode"], options=lid.Options(path=3))["fused"] == 1
    assert lid.plan(*li.SHAPES["multiseq"])["fused"] == 1
    assert lid.plan(*li.SHAPES["long"])["fused"] == 0
    assert lid.plan(*li.SHAPES["decode"], options=lid.Options(path=1))["fused"] == 0
    # one CTA per SM: a group cannot use more splits than there are SMs
    with pytest.raises(lid.LidError):
        lid.plan(1, 131072, 64, 128, 512, options=lid.Options(path=2, force_splits=1000))


def test_one_launch_bounded_group_barrier_reports_and_context_survives():
    """The first group barrier waits for one CTA more than the group has: every
    CTA gives up after the short limit, records code 4 and exits; the context
    stays usable."""
    inp = li.int_inputs("fb", 1, 20000, 64, 128, 64, seed=43, dtype="bf16")
    q, k, w, m = to_device(inp)
    lid.device_error(reset=True)
    lid.topk(q, k, w, m, inp.top_k, options=lid.Options(path=2, fault_inject=3))
    assert lid.device_error(reset=True) == 4
    g_idx, g_sc = run_gpu(inp, options=lid.Options(path=2))
    check_exact(g_idx, g_sc, inp)
    assert lid.device_error() == 0


def test_one_launch_barrier_slots_across_streams_and_graphs():
    """The one-launch path's group-barrier counters live in slots that each
    launch leaves at zero: calls alternating over two streams, back-to-back
    calls on one stream, and a CUDA graph replayed several times all give the
    exact result (a slot left dirty would let a barrier pass early or time out)."""
    inp = li.int_inputs("sl", 2, 20000, 64, 128, 64, seed=47, dtype="bf16")
    assert lid.plan(inp.n_q, inp.n_kv, inp.H, inp.D, inp.top_k)["fused"] == 1
    q, k, w, m = to_device(inp)
    o_idx, o_sc = oracle.topk_inputs(inp)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for it in range(6):
        s = streams[it % 2]
        with torch.cuda.stream(s):
            outs.append(lid.topk(q, k, w, m, inp.top_k, stream=s))
    torch.cuda.synchronize()
    for idx, sc in outs:
        assert np.array_equal(idx.cpu().numpy(), o_idx)
        assert np.array_equal(sc.cpu().numpy().astype(np.float64), o_sc)
    s = torch.cuda.Stream()
    oi = torch.empty((inp.n_q, inp.top_k), dtype=torch.int32, device="cuda")
    os_ = torch.empty((inp.n_q, inp.top_k), dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        lid.topk(q, k, w, m, inp.top_k, out_idx=oi, out_score=os_, stream=s)  # eager first
        s.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            lid.topk(q, k, w, m, inp.top_k, out_idx=oi, out_score=os_, stream=s)
            lid.topk(q, k, w, m, inp.top_k, out_idx=oi, out_score=os_, stream=s)
    for _ in range(3):
        oi.fill_(7)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(oi.cpu().numpy(), o_idx)
        assert np.array_equal(os_.cpu().numpy().astype(np.float64), o_sc)
    assert lid.device_error() == 0


# ------------------------------------------------ per-row visible key ranges

def _run_ranges(inp, lo, hi, options=None):
    q, k, w, _ = to_device(inp)
    idx, sc = lid.topk_ranges(q, k, w, torch.from_numpy(lo).cuda(), torch.from_numpy(hi).cuda(), inp.top_k,
                              options=options)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


RANGE_CASES = [
    # H, D, dtype, n_q, n_kv, top_k, ranges
    (64, 128, "bf16", 9, 4099, 512, "causal"),
    (64, 128, "bf16", 4, 40000, 256, "blocks"),      # one row per CTA, each streams its own tiles only
    (16, 64, "f16", 3, 30000, 100, "blocks"),
    (8, 64, "f16", 6, 5000, 64, "blocks"),           # two rows per CTA (H = 8)
    (64, 128, "bf16", 4, 20000, 512, "odd"),         # short, empty and out-of-bounds ranges
    (32, 128, "bf16", 20, 3000, 64, "causal"),
]


def _case_ranges(kind, n_q, n_kv):
    if kind == "causal":
        return li.causal_ranges(n_q, n_kv - n_q)
    if kind == "blocks":
        return li.block_ranges(n_q, n_kv // n_q)
    lo = np.array([-7, 100, 5000, 19990], np.int32)[:n_q]
    hi = np.array([300, 100, 25000, 20000], np.int32)[:n_q]  # 300 visible < top_k; empty; past the end; 10
    return lo, hi


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("case", RANGE_CASES, ids=[f"H{c[0]}D{c[1]}q{c[3]}kv{c[4]}k{c[5]}{c[6]}" for c in RANGE_CASES])
def test_ranges_bit_exact(case, path):
    """lid_topk_ranges equals the oracle run on the dense mask the ranges
    describe, on both split paths."""
    H, D, dtype, n_q, n_kv, top_k, kind = case
    lo, hi = _case_ranges(kind, n_q, n_kv)
    inp = li.int_inputs("rg", n_q, n_kv, H, D, top_k, seed=n_kv + 3, dtype=dtype,
                        mask=li.mask_from_ranges(lo, hi, n_kv))
    g_idx, g_sc = _run_ranges(inp, lo, hi, lid.Options(path=path) if path else None)
    check_exact(g_idx, g_sc, inp)


def test_ranges_multiseq_full_size_sampled():
    inp = li.workload("multiseq")
    lo, hi = li.workload_ranges("multiseq")
    g_idx, g_sc = _run_ranges(inp, lo, hi)
    check_tolerance(g_idx, g_sc, inp, range(4))
    assert all(np.all((g_idx[j] >= lo[j]) & (g_idx[j] < hi[j])) for j in range(4))


def test_ranges_argument_errors():
    q = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((300, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.ones((2, 64), dtype=torch.float32, device="cuda")
    lo = torch.zeros(2, dtype=torch.int32, device="cuda")
    oi = torch.full((2, 16), 7, dtype=torch.int32, device="cuda")
    os_ = torch.full((2, 16), 3.5, dtype=torch.float32, device="cuda")
    L = lid.load()
    rc = L.lid_topk_ranges(q.data_ptr(), k.data_ptr(), w.data_ptr(), lo.data_ptr(), None, 2, 300, 64, 128, 16,
                           oi.data_ptr(), os_.data_ptr(), None, 0, None)
    assert rc == lid.LID_ERR_INVALID_ARG
    rc = L.lid_topk_ranges(q.data_ptr(), k.data_ptr(), w.data_ptr(), lo.data_ptr() + 2, lo.data_ptr(), 2, 300, 64,
                           128, 16, oi.data_ptr(), os_.data_ptr(), None, 0, None)
    assert rc == lid.LID_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(oi == 7) and torch.all(os_ == 3.5)


# ------------------------------------------- quantised operands (E4M3 codes)

E4M3_CASES = [
    # H, n_q, n_kv, top_k, mask, path, force_splits
    (64, 1, 5000, 512, "none", 0, 0),
    (64, 5, 3001, 100, "random", 1, 4),
    (64, 9, 4099, 512, "causal", 0, 0),
    (32, 7, 1000, 256, "random", 0, 0),
    (16, 20, 2500, 33, "causal", 0, 3),
    (8, 33, 640, 16, "random", 0, 2),
    (64, 4, 20000, 512, "random", 2, 0),
    (64, 2, 100, 300, "none", 0, 0),     # fewer keys than top_k: padding
]


@pytest.mark.parametrize("case", E4M3_CASES, ids=[f"H{c[0]}q{c[1]}kv{c[2]}k{c[3]}{c[4]}p{c[5]}s{c[6]}"
                                                  for c in E4M3_CASES])
def test_e4m3_integer_codes_bit_exact(case):
    """E4M3 codes of small integers with power-of-two row scales (distinct per
    q row and key row): every step is exact, so the CUDA path must equal the
    oracle slot by slot -- which also pins the scale of each q row (t, h) and
    key row to its own row."""
    H, n_q, n_kv, top_k, mkind, path, splits = case
    inp = li.int_e4m3_inputs("e4", n_q, n_kv, H, 128, top_k, seed=n_kv + H, mask=_mask(mkind, n_q, n_kv, n_kv + 1),
                             w_range=(-3, 3) if mkind == "random" else (0, 3))
    opt = lid.Options(force_splits=splits, path=path) if (splits or path) else None
    g_idx, g_sc = run_gpu(inp, options=opt)
    check_exact(g_idx, g_sc, inp)


def test_e4m3_ranges_bit_exact():
    n_q, n_kv = 4, 40000
    lo, hi = li.block_ranges(n_q, n_kv // n_q)
    inp = li.int_e4m3_inputs("e4r", n_q, n_kv, 64, 128, 256, seed=5, mask=li.mask_from_ranges(lo, hi, n_kv))
    g_idx, g_sc = run_gpu(inp, ranges=(lo, hi))
    check_exact(g_idx, g_sc, inp)


@pytest.mark.parametrize("name", ["decode_e4m3", "multiseq_e4m3"])
def test_e4m3_workloads_full_size(name):
    """The quantised decode and multi-sequence shapes at full size (float
    codes from N(0,1) draws), within the float tolerance of the oracle; the
    multi-sequence rows through their visible ranges."""
    inp = li.workload(name)
    ranges = li.workload_ranges(name) if name.startswith("multiseq") else None
    g_idx, g_sc = run_gpu(inp, ranges=ranges)
    check_tolerance(g_idx, g_sc, inp, range(inp.n_q))
    if ranges is not None:
        lo, hi = ranges
        assert all(np.all((g_idx[j] >= lo[j]) & (g_idx[j] < hi[j])) for j in range(inp.n_q))


def test_e4m3_argument_errors():
    L = lid.load()
    q8 = torch.zeros((2, 64, 128), dtype=torch.uint8, device="cuda")
    k8 = torch.zeros((300, 128), dtype=torch.uint8, device="cuda")
    qs = torch.ones((2, 64), dtype=torch.float32, device="cuda")
    ks = torch.ones(300, dtype=torch.float32, device="cuda")
    w = torch.ones((2, 64), dtype=torch.float32, device="cuda")
    oi = torch.full((2, 16), 7, dtype=torch.int32, device="cuda")
    os_ = torch.full((2, 16), 3.5, dtype=torch.float32, device="cuda")

    def call(q_scale, k_scale, D=128, mask=None, lo=None, hi=None):
        return L.lid_topk_e4m3(q8.data_ptr(), q_scale, k8.data_ptr(), k_scale, w.data_ptr(), mask, lo, hi, 2, 300,
                               64, D, 16, oi.data_ptr(), os_.data_ptr(), None, None)

    assert call(None, ks.data_ptr()) == lid.LID_ERR_INVALID_ARG
    assert call(qs.data_ptr(), None) == lid.LID_ERR_INVALID_ARG
    assert call(qs.data_ptr() + 2, ks.data_ptr()) == lid.LID_ERR_INVALID_ARG  # misaligned scale
    assert call(qs.data_ptr(), ks.data_ptr(), D=64) == lid.LID_ERR_UNSUPPORTED
    lo = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert call(qs.data_ptr(), ks.data_ptr(), lo=lo.data_ptr()) == lid.LID_ERR_INVALID_ARG  # lo without hi
    # the 16-bit entry points refuse the 8-bit dtype code
    assert L.lid_topk_ex(q8.data_ptr(), k8.data_ptr(), w.data_ptr(), None, 2, 300, 64, 128, 16, oi.data_ptr(),
                         os_.data_ptr(), None, lid.DTYPE_E4M3, None) == lid.LID_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(oi == 7) and torch.all(os_ == 3.5)


# ----------------------------------------------- caller-owned workspace

WS_CASES = [
    # H, D, dtype, n_q, n_kv, top_k, options, mask: every merge form through lid_topk_ws
    (64, 128, "bf16", 1, 131072, 512, {}, "none"),            # one launch, early steps, per-split regions
    (64, 128, "bf16", 1, 131072, 512, {"path": 1}, "random"),  # per-split lists + merge kernel
    (64, 128, "f16", 9, 4099, 512, {"path": 2}, "causal"),     # one launch, several queries per CTA
    (32, 64, "f16", 1, 50000, 256, {"early_tiles": 1}, "causal"),
    (8, 64, "f16", 4, 2048, 64, {}, "causal"),                 # no split: no workspace needed
]


@pytest.mark.parametrize("case", WS_CASES, ids=[f"H{c[0]}q{c[3]}kv{c[4]}{c[6]}{c[7]}" for c in WS_CASES])
def test_caller_workspace_bit_exact_and_reusable(case):
    """lid_topk_ws with one zeroed workspace reused by consecutive calls (its
    counter area must be left zero by every call) gives the oracle's result
    bit for bit."""
    H, D, dtype, n_q, n_kv, top_k, o, mkind = case
    inp = li.int_inputs("ws", n_q, n_kv, H, D, top_k, seed=n_kv + 3 * H, mask=_mask(mkind, n_q, n_kv, n_kv + 5),
                        dtype=dtype, w_range=(-3, 3))
    opt = lid.Options(**o)
    q, k, w, m = to_device(inp)
    ws = lid.workspace(n_q, n_kv, H, D, top_k, opt)
    if ws is None:
        assert lid.plan(n_q, n_kv, H, D, top_k, opt)["workspace_bytes"] == 0
    o_idx, o_sc = oracle.topk_inputs(inp)
    for _ in range(3):
        idx, sc = lid.topk_ws(q, k, w, top_k, ws, mask=m, options=opt)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), o_idx)
        assert np.array_equal(sc.cpu().numpy().astype(np.float64), o_sc)
    if ws is not None:
        assert torch.count_nonzero(ws[:1024]).item() == 0, "the counter area was not left zero"


def test_caller_workspace_ranges_and_e4m3_forms():
    n_q, n_kv = 4, 40000
    inp = li.int_inputs("wr", n_q, n_kv, 64, 128, 256, seed=91, dtype="bf16", w_range=(-3, 3))
    lo, hi = li.block_ranges(n_q, n_kv // n_q)
    inp_m = li.Inputs(inp.name, inp.dtype, n_q, n_kv, 64, 128, 256, inp.q_bits, inp.k_bits, inp.w,
                      li.mask_from_ranges(lo, hi, n_kv))
    q, k, w, _ = to_device(inp)
    opt = lid.Options(plan_ranges=1)  # the plan of the range form
    ws = lid.workspace(n_q, n_kv, 64, 128, 256, opt)
    idx, sc = lid.topk_ws(q, k, w, 256, ws, row_lo=torch.from_numpy(lo).cuda(), row_hi=torch.from_numpy(hi).cuda())
    torch.cuda.synchronize()
    check_exact(idx.cpu().numpy(), sc.cpu().numpy(), inp_m)
    e = li.int_e4m3_inputs("we", 2, 30000, 64, 128, 128, seed=92, mask=li.causal_mask(2, 30000, 29998))
    q8, k8, w8, m8 = to_device(e)
    qs, ks = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (e.q_scale, e.k_scale))
    ws = lid.workspace(2, 30000, 64, 128, 128)
    idx, sc = lid.topk_ws(q8, k8, w8, 128, ws, mask=m8, q_scale=qs, k_scale=ks)
    torch.cuda.synchronize()
    check_exact(idx.cpu().numpy(), sc.cpu().numpy(), e)


def test_caller_workspace_errors_launch_nothing():
    n_q, n_kv, H, D, top_k = li.SHAPES["decode"]
    q = torch.zeros((n_q, H, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((n_kv, D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((n_q, H), dtype=torch.float32, device="cuda")
    need = lid.plan(n_q, n_kv, H, D, top_k)["workspace_bytes"]
    oi = torch.full((n_q, top_k), 7, dtype=torch.int32, device="cuda")
    os_ = torch.full((n_q, top_k), 3.5, dtype=torch.float32, device="cuda")
    small = torch.zeros(need - 8, dtype=torch.uint8, device="cuda")
    for ws in (None, small):
        with pytest.raises(lid.LidError) as e:
            lid.topk_ws(q, k, w, top_k, ws, out_idx=oi, out_score=os_)
        assert e.value.status == lid.LID_ERR_SCRATCH_TOO_SMALL
    big = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(lid.LidError) as e:  # misaligned start
        lid.topk_ws(q, k, w, top_k, big[8:], out_idx=oi, out_score=os_)
    assert e.value.status == lid.LID_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(oi == 7) and torch.all(os_ == 3.5)


def test_one_launch_region_overflow_falls_back_exactly():
    """Every key of the top-512 sits in the last split (equal scores at the end
    of the key range), so that split's region of keys above the bound
    overflows and every CTA takes the general gather instead; the result is
    still the oracle's, ties broken by index."""
    n_kv, H, D = 131072, 64, 128
    k = np.zeros((n_kv, D), np.float32)
    k[n_kv - 600:, 0] = 1.0
    q = np.zeros((1, H, D), np.float32)
    q[0, :, 0] = 1.0
    inp = li.Inputs("ovf", "bf16", 1, n_kv, H, D, 512, li.f32_to_bf16_bits(q), li.f32_to_bf16_bits(k),
                    np.ones((1, H), np.float32), None)
    for path, kind in ((0, 2), (3, 1)):  # the single-query kernel, then the general one-launch kernel
        assert lid.plan(1, n_kv, H, D, 512, options=lid.Options(path=path))["fused"] == kind
        g_idx, g_sc = run_gpu(inp, options=lid.Options(path=path))
        check_exact(g_idx, g_sc, inp)
        assert list(g_idx[0, :4]) == [n_kv - 600, n_kv - 599, n_kv - 598, n_kv - 597]


def test_single_query_overflow_beyond_top_k_takes_each_splits_own_top():
    """Ascending scores over the whole key range: the last split alone holds
    every key of the top-512 and more than 512 keys above the bound, so it
    cuts its overflow list to its own top 512 (a radix select) before the
    ranking; still the oracle's result."""
    n_kv, H, D = 131072, 64, 128
    k = np.zeros((n_kv, D), np.float32)
    k[:, 0] = np.repeat(np.arange(n_kv // 512, dtype=np.float32), 512)  # 256 levels, exact in bf16
    q = np.zeros((1, H, D), np.float32)
    q[0, :, 0] = 1.0
    inp = li.Inputs("asc1", "bf16", 1, n_kv, H, D, 512, li.f32_to_bf16_bits(q), li.f32_to_bf16_bits(k),
                    np.ones((1, H), np.float32), None)
    assert lid.plan(1, n_kv, H, D, 512)["fused"] == 2
    g_idx, g_sc = run_gpu(inp)
    check_exact(g_idx, g_sc, inp)


def test_one_launch_slots_survive_stream_destroy_and_reuse():
    """Streams created and destroyed between back-to-back one-launch calls,
    the next one created while the previous call may still run (a new stream
    can get the destroyed one's handle): the barrier-counter slots are keyed
    by stream ID, so the calls never share counters, and every result is the
    oracle's."""
    libcuda = ctypes.CDLL("libcuda.so.1")
    inp = li.int_inputs("sd", 1, 131072, 64, 128, 512, seed=97, dtype="bf16", w_range=(-3, 3))
    assert lid.plan(1, 131072, 64, 128, 512)["fused"] == 2
    q, k, w, m = to_device(inp)
    o_idx, o_sc = oracle.topk_inputs(inp)
    torch.cuda.synchronize()
    outs, handles = [], []
    for _ in range(8):
        h = ctypes.c_void_p()
        assert libcuda.cuStreamCreate(ctypes.byref(h), 1) == 0  # non-blocking stream
        handles.append(h.value)
        oi = torch.empty((1, 512), dtype=torch.int32, device="cuda")
        os_ = torch.empty((1, 512), dtype=torch.float32, device="cuda")
        rc = lid.load().lid_topk_ex(q.data_ptr(), k.data_ptr(), w.data_ptr(), None, 1, 131072, 64, 128, 512,
                                    oi.data_ptr(), os_.data_ptr(), h.value, lid.DTYPE_BF16, None)
        assert rc == lid.LID_OK, lid.status_string(rc)
        outs.append((oi, os_))
        assert libcuda.cuStreamDestroy_v2(h) == 0  # its work still completes
    torch.cuda.synchronize()
    for oi, os_ in outs:
        assert np.array_equal(oi.cpu().numpy(), o_idx)
        assert np.array_equal(os_.cpu().numpy().astype(np.float64), o_sc)
    assert lid.device_error() == 0


def test_no_n_q_by_n_kv_buffer_is_allocated_measured():
    """Device memory actually taken by a long-prefill call (2048 queries x
    131072 keys, whose score matrix would be 1 GiB in f32 and 64 GiB per head):
    the free-memory drop across the call, with inputs and outputs allocated
    beforehand, is the library's workspace only."""
    n_q, n_kv, H, D, top_k = li.SHAPES["long"]
    q = torch.zeros((n_q, H, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((n_kv, D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((n_q, H), dtype=torch.float32, device="cuda")
    oi = torch.empty((n_q, top_k), dtype=torch.int32, device="cuda")
    os_ = torch.empty((n_q, top_k), dtype=torch.float32, device="cuda")
    small = li.int_inputs("warm", 2, 3000, 64, 128, 64, seed=1, dtype="bf16")
    run_gpu(small)  # module and pool set up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    lid.topk(q, k, w, None, top_k, out_idx=oi, out_score=os_)
    torch.cuda.synchronize()
    grew = free0 - torch.cuda.mem_get_info()[0]
    score_matrix = n_q * n_kv * 4
    assert grew < 64 << 20, f"device memory grew by {grew} bytes during the call"
    assert grew < score_matrix // 16
    need = lid.plan(n_q, n_kv, H, D, top_k)["workspace_bytes"]
    assert need < 64 << 20


def test_mask_alignment_and_ragged_key_counts_bit_exact():
    """Several queries per CTA with the mask as a 16-byte aligned tensor and as
    a view 2 bytes into a larger buffer (aligned only to its elements), key
    counts a multiple of 8 and not, planned and forced splits: every result is
    the oracle's."""
    for n_kv in (6000, 6001):
        inp = li.int_inputs("ring", 9, n_kv, 64, 128, 256, seed=n_kv, mask=_random_mask(9, n_kv, 5), dtype="bf16",
                            w_range=(-3, 3))
        o_idx, o_sc = oracle.topk_inputs(inp)
        q, k, w, m = to_device(inp)
        # the same mask bits 2 bytes into a larger buffer: aligned to 2, not to 16
        big = torch.empty(m.numel() + 8, dtype=torch.float16, device="cuda")
        m_off = big[1:1 + m.numel()].view(m.shape)
        m_off.copy_(m)
        for mask in (m, m_off):
            for opt in (None, lid.Options(force_splits=3)):
                idx, sc = lid.topk(q, k, w, mask, inp.top_k, options=opt)
                torch.cuda.synchronize()
                assert np.array_equal(idx.cpu().numpy(), o_idx)
                assert np.array_equal(sc.cpu().numpy().astype(np.float64), o_sc)
