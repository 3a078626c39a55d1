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
    # four ints, two pointers, four reserved ints
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
