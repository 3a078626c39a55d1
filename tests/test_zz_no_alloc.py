"""lid_topk_static: the entry point that allocates nothing.

Some callers cannot allocate device memory while a step runs (an engine that
reserves all device memory up front under its own allocator, or a path that
may not risk an allocation failing or stalling mid-step). lid_topk_static
keeps the split workspace in a fixed array the library defines in device
memory. These tests call it through the C ABI, twice in a row, and compare
with lid_topk_ex (which allocates its workspace per call) under the parity
tolerance the other GPU tests use, and with the CPU oracle bit for bit on
integer-valued inputs: the tiny workload, a one-launch shape (its certificates,
candidates and barrier counters in the array) and a two-launch shape (its
per-split lists in the array, read by the merge kernel). The file is named to
be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import lid_inputs as li
import sparse_attention_lightning_lid_gb300 as lid
from tests.parity import REL, check_exact, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lid.load()
    yield


def _call_static(q, k, w, m, top_k, dtype):
    n_q, H, D = q.shape
    oi = torch.full((n_q, top_k), 7, dtype=torch.int32, device="cuda")
    os_ = torch.full((n_q, top_k), 3.5, dtype=torch.float32, device="cuda")
    rc = lid.load().lid_topk_static(q.data_ptr(), k.data_ptr(), w.data_ptr(), None if m is None else m.data_ptr(),
                                    n_q, k.shape[0], H, D, top_k, oi.data_ptr(), os_.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream, dtype)
    return rc, oi, os_


def _same_within_tolerance(a_idx, a_sc, b_idx, b_sc):
    """Two GPU results agree: scores within REL of each other slot by slot, and
    the index sets differ only where the scores tie within REL of the k-th."""
    assert a_idx.shape == b_idx.shape
    for r in range(a_idx.shape[0]):
        fin = np.isfinite(b_sc[r])
        assert np.array_equal(np.isfinite(a_sc[r]), fin)
        kth = abs(b_sc[r][fin][-1]) if fin.any() else 0.0
        scale = np.maximum(np.abs(b_sc[r][fin]), kth)
        assert np.all(np.abs(a_sc[r][fin] - b_sc[r][fin]) <= REL * scale)
        diff = set(a_idx[r].tolist()) ^ set(b_idx[r].tolist())
        if diff:
            score_of = dict(zip(a_idx[r].tolist(), a_sc[r].tolist()))
            score_of.update(zip(b_idx[r].tolist(), b_sc[r].tolist()))
            for s in diff:
                assert abs(score_of[s] - b_sc[r][fin][-1]) <= REL * kth


@pytest.mark.parametrize("name", ["decode", "multiseq_small", "tiny"])
def test_static_scratch_matches_allocating_entry_point(name):
    if name == "multiseq_small":
        inp = li.float_inputs("m", 4, 262144, 64, 128, 512, seed=31, mask=li.range_mask(4, 262144, 65536))
    else:
        inp = li.workload(name)
    q, k, w, m = to_device(inp)
    dtype = lid.DTYPE_F16 if inp.dtype == "f16" else lid.DTYPE_BF16
    ref_idx, ref_sc = lid.topk(q, k, w, m, inp.top_k)
    torch.cuda.synchronize()
    ref_idx, ref_sc = ref_idx.cpu().numpy(), ref_sc.cpu().numpy()
    for _ in range(2):  # the scratch keeps the previous call's contents
        rc, oi, os_ = _call_static(q, k, w, m, inp.top_k, dtype)
        assert rc == lid.LID_OK, lid.status_string(rc)
        torch.cuda.synchronize()
        _same_within_tolerance(oi.cpu().numpy(), os_.cpu().numpy(), ref_idx, ref_sc)
    assert lid.device_error() == 0


def test_static_scratch_rejects_shapes_beyond_its_size():
    n_q, n_kv, H, D, top_k = li.SHAPES["long"]
    need = lid.plan(n_q, n_kv, H, D, top_k)["workspace_bytes"]
    assert need > 8 << 20
    q = torch.zeros((n_q, H, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((n_kv, D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((n_q, H), dtype=torch.float32, device="cuda")
    rc, oi, os_ = _call_static(q, k, w, None, top_k, lid.DTYPE_BF16)
    assert rc == lid.LID_ERR_SCRATCH_TOO_SMALL
    assert "8 MiB" in lid.status_string(rc)
    torch.cuda.synchronize()
    assert torch.all(oi == 7) and torch.all(os_ == 3.5)  # nothing was launched


def _static_twice_exact(inp, rows=None):
    q, k, w, m = to_device(inp)
    dtype = lid.DTYPE_F16 if inp.dtype == "f16" else lid.DTYPE_BF16
    for _ in range(2):  # the second call finds the first one's contents in the array
        rc, oi, os_ = _call_static(q, k, w, m, inp.top_k, dtype)
        assert rc == lid.LID_OK, lid.status_string(rc)
        torch.cuda.synchronize()
        g_idx, g_sc = oi.cpu().numpy(), os_.cpu().numpy()
        check_exact(g_idx, g_sc, inp, rows)
        assert np.all(np.diff(g_sc, axis=1) <= 0)
    assert lid.device_error() == 0


def test_static_scratch_tiny_workload_bit_exact_vs_oracle():
    _static_twice_exact(li.workload("tiny"))


def test_static_scratch_one_launch_bit_exact_vs_oracle():
    inp = li.int_inputs("s1", 1, 131072, 64, 128, 512, seed=61, dtype="bf16", w_range=(-3, 3))
    p = lid.plan(1, 131072, 64, 128, 512)
    assert p["fused"] >= 1 and p["splits"] > 1 and 0 < p["workspace_bytes"] <= 8 << 20
    _static_twice_exact(inp)


def test_static_scratch_two_launch_lists_bit_exact_vs_oracle():
    n_q, n_kv, H, D, top_k = 400, 65536, 64, 128, 512
    p = lid.plan(n_q, n_kv, H, D, top_k)
    assert p["fused"] == 0 and p["splits"] > 1 and 0 < p["workspace_bytes"] <= 8 << 20, p
    mask = li.causal_mask(n_q, n_kv, n_kv - n_q)
    inp = li.int_inputs("s2", n_q, n_kv, H, D, top_k, seed=62, mask=mask, dtype="bf16", w_range=(-3, 3))
    _static_twice_exact(inp, rows=np.array([0, 1, 3, 4, 57, 199, 200, 398, 399]))
