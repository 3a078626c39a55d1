"""The C-ABI library builds, loads without a GPU, and exports every function
that include/lid.h declares. No compute call is made here."""
import ctypes
import os
import re

import sparse_attention_lightning_lid_gb300 as lid

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lid.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(lid_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_expected_entry_points():
    names = _declared_functions()
    assert set(names) == set(lid.EXPORTS), names


def test_library_builds_loads_and_exports_every_declared_symbol():
    path = lid.build()
    handle = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(handle, name), f"{name} declared in lid.h but not exported"
    L = lid.load()
    assert L.lid_status_string(0) == b"ok"
    assert b"unsupported" in L.lid_status_string(2)


def test_options_struct_layout_matches_header():
    # four ints, two pointers, four more ints (path, early_tiles, plan_ranges, reserved)
    assert ctypes.sizeof(lid.Options) == 4 * 4 + 2 * ctypes.sizeof(ctypes.c_void_p) + 4 * 4
    assert lid.PlanInfo.workspace_bytes.offset == 40


def test_enum_values_match_header():
    text = open(HEADER).read()
    for name, value in (("LID_DTYPE_BF16", lid.DTYPE_BF16), ("LID_DTYPE_F16", lid.DTYPE_F16),
                        ("LID_DTYPE_E4M3", lid.DTYPE_E4M3), ("LID_OK", lid.LID_OK),
                        ("LID_ERR_INVALID_ARG", lid.LID_ERR_INVALID_ARG),
                        ("LID_ERR_UNSUPPORTED", lid.LID_ERR_UNSUPPORTED),
                        ("LID_ERR_SCRATCH_TOO_SMALL", lid.LID_ERR_SCRATCH_TOO_SMALL)):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == value, name


def test_e4m3_binding_checks_arguments_before_the_library():
    # host-side validation of the Python binding (no GPU needed: it raises first)
    import pytest
    import torch
    q8 = torch.zeros((2, 8, 128), dtype=torch.uint8)
    k8 = torch.zeros((50, 128), dtype=torch.uint8)
    qs, ks = torch.ones((2, 8)), torch.ones(50)
    w = torch.ones((2, 8))
    with pytest.raises(ValueError, match="shape"):
        lid.topk_e4m3(q8, qs, k8, torch.ones(49), w, None, 16)
    with pytest.raises(TypeError, match="8-bit"):
        lid.topk_e4m3(q8.to(torch.int16), qs, k8, ks, w, None, 16)
    with pytest.raises(TypeError, match="float32"):
        lid.topk_e4m3(q8, qs.double(), k8, ks, w, None, 16)
    with pytest.raises(ValueError, match="together"):
        lid.topk_e4m3(q8, qs, k8, ks, w, None, 16, row_lo=torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        lid.topk_e4m3(q8, qs, k8, ks, w, None, 16)


def test_host_entry_points_reject_bad_arguments_before_any_device_call():
    # argument errors return before anything is enqueued (nothing here touches a GPU)
    import numpy as np
    L = lid.load()
    q = np.zeros((2, 64, 128), np.uint16)
    k = np.zeros((300, 128), np.uint16)
    w = np.zeros((2, 64), np.float32)
    oi = np.zeros((2, 16), np.int32)
    os_ = np.zeros((2, 16), np.float32)
    P = lambda a: a.ctypes.data
    for fn in (L.lid_topk_host, L.lid_topk_host_async):
        call = lambda n_q=2, n_kv=300, H=64, D=128, top_k=16, out_i=P(oi), out_s=P(os_), dtype=lid.DTYPE_BF16: fn(
            P(q), P(k), P(w), None, n_q, n_kv, H, D, top_k, out_i, out_s, None, dtype)
        assert call(n_q=-1) == lid.LID_ERR_INVALID_ARG
        assert call(H=48) == lid.LID_ERR_UNSUPPORTED
        assert call(top_k=0) == lid.LID_ERR_UNSUPPORTED
        assert call(dtype=lid.DTYPE_E4M3) == lid.LID_ERR_INVALID_ARG
        assert call(out_i=None) == lid.LID_ERR_INVALID_ARG
        assert call(n_q=0) == lid.LID_OK
