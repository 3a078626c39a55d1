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
