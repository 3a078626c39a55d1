"""CPU oracle of the lightning-indexer top-k (test infrastructure only).

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package. It shares no code with the CUDA path.

Two implementations live here:
  * `lid_oracle.c` -- the fp64 oracle: full score rows, then a full sort
    (compiled with gcc + OpenMP by `build()`; loaded with ctypes);
  * `brute.py` -- exact rational arithmetic in pure Python for tiny inputs,
    used to pin the C oracle.

The method (DeepSeek-V4-Flash lightning indexer; llama.cpp issue 25468,
root-cause comment; llama.cpp PR 22378, collapse-Q revert commit;
fairydreaming/llama.cpp PR 2, API-change note):
    I[t,s] = sum_h w[t,h] * relu(q[t,h,:] . k[s,:]) + mask[t,s]
and per query the top_k keys by (I descending, key index ascending).
`topk_e4m3` / `scores_e4m3` take q and k as E4M3 codes with one f32 scale
per row (value = scale * code) and compute the same on the decoded values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lid_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblid_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle in-tree (gcc -O2 -fopenmp). Returns the .so path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def use_library(path):
    """Point this module at another build of lid_oracle.c (the mutation
    tests load deliberately broken copies); None restores the real one.
    Returns the previously bound library handle."""
    global _lib
    prev = _lib
    _lib = None if path is None else _bind(ctypes.CDLL(path))
    return prev


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I = ctypes.c_int
    lib.lid_oracle_scores.argtypes = [P, P, P, P, I64, I64, I, I, I, P, I64, P]
    lib.lid_oracle_scores.restype = I
    lib.lid_oracle_topk.argtypes = [P, P, P, P, I64, I64, I, I, I, I, P, I64, P, P]
    lib.lid_oracle_topk.restype = I
    lib.lid_oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.lid_oracle_decode_bf16.restype = ctypes.c_double
    lib.lid_oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.lid_oracle_decode_f16.restype = ctypes.c_double
    lib.lid_oracle_scores_e4m3.argtypes = [P, P, P, P, P, P, I64, I64, I, I, P, I64, P]
    lib.lid_oracle_scores_e4m3.restype = I
    lib.lid_oracle_topk_e4m3.argtypes = [P, P, P, P, P, P, I64, I64, I, I, I, P, I64, P, P]
    lib.lid_oracle_topk_e4m3.restype = I
    lib.lid_oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
    lib.lid_oracle_decode_e4m3.restype = ctypes.c_double
    lib.lid_oracle_sparse_attn.argtypes = [P, P, P, P, I64, I64, I, I, I, I, ctypes.c_double, P, I64, P, P]
    lib.lid_oracle_sparse_attn.restype = I
    lib.lid_oracle_threads.argtypes = []
    lib.lid_oracle_threads.restype = I
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(q_bits, k_bits, w, mask, rows, n_q):
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    wf = np.ascontiguousarray(w, dtype=np.float32)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint16)
    r = np.arange(n_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    return q, k, wf, m, r


def scores(q_bits, k_bits, w, mask, H, D, dtype="bf16", rows=None):
    """fp64 score rows [len(rows)][n_kv] (all rows if rows is None)."""
    n_q = q_bits.size // (H * D)
    n_kv = k_bits.size // D
    q, k, wf, m, r = _prep(q_bits, k_bits, w, mask, rows, n_q)
    out = np.empty((r.size, n_kv), dtype=np.float64)
    rc = _load().lid_oracle_scores(_ptr(q), _ptr(k), _ptr(wf), _ptr(m), n_q, n_kv, H, D,
                                   int(dtype == "f16"), _ptr(r), r.size, _ptr(out))
    if rc:
        raise RuntimeError(f"lid_oracle_scores failed with code {rc}")
    return out


def topk(q_bits, k_bits, w, mask, H, D, top_k, dtype="bf16", rows=None):
    """(idx int64 [rows][top_k], score fp64 [rows][top_k]) by (score desc, idx asc)."""
    n_q = q_bits.size // (H * D)
    n_kv = k_bits.size // D
    q, k, wf, m, r = _prep(q_bits, k_bits, w, mask, rows, n_q)
    idx = np.empty((r.size, top_k), dtype=np.int64)
    sc = np.empty((r.size, top_k), dtype=np.float64)
    rc = _load().lid_oracle_topk(_ptr(q), _ptr(k), _ptr(wf), _ptr(m), n_q, n_kv, H, D, top_k,
                                 int(dtype == "f16"), _ptr(r), r.size, _ptr(idx), _ptr(sc))
    if rc:
        raise RuntimeError(f"lid_oracle_topk failed with code {rc}")
    return idx, sc


def _prep_e4m3(q8, q_scale, k8, k_scale, w, mask, rows, n_q, H, D):
    q = np.ascontiguousarray(q8, dtype=np.uint8)
    k = np.ascontiguousarray(k8, dtype=np.uint8)
    qs = np.ascontiguousarray(q_scale, dtype=np.float32)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    wf = np.ascontiguousarray(w, dtype=np.float32)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint16)
    r = np.arange(n_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    if qs.size != n_q * H or ks.size != k.size // D:
        raise ValueError("one scale per q row (t, h) and per key row is expected")
    return q, qs, k, ks, wf, m, r


def scores_e4m3(q8, q_scale, k8, k_scale, w, mask, H, D, rows=None):
    """fp64 score rows of the quantised form: q8 [n_q, H, D] and k8 [n_kv, D]
    E4M3 codes, q_scale [n_q, H] and k_scale [n_kv] f32."""
    n_q = q8.size // (H * D)
    n_kv = k8.size // D
    q, qs, k, ks, wf, m, r = _prep_e4m3(q8, q_scale, k8, k_scale, w, mask, rows, n_q, H, D)
    out = np.empty((r.size, n_kv), dtype=np.float64)
    rc = _load().lid_oracle_scores_e4m3(_ptr(q), _ptr(qs), _ptr(k), _ptr(ks), _ptr(wf), _ptr(m), n_q, n_kv,
                                        H, D, _ptr(r), r.size, _ptr(out))
    if rc:
        raise RuntimeError(f"lid_oracle_scores_e4m3 failed with code {rc}")
    return out


def topk_e4m3(q8, q_scale, k8, k_scale, w, mask, H, D, top_k, rows=None):
    """`topk` of the quantised form (arguments as in `scores_e4m3`)."""
    n_q = q8.size // (H * D)
    n_kv = k8.size // D
    q, qs, k, ks, wf, m, r = _prep_e4m3(q8, q_scale, k8, k_scale, w, mask, rows, n_q, H, D)
    idx = np.empty((r.size, top_k), dtype=np.int64)
    sc = np.empty((r.size, top_k), dtype=np.float64)
    rc = _load().lid_oracle_topk_e4m3(_ptr(q), _ptr(qs), _ptr(k), _ptr(ks), _ptr(wf), _ptr(m), n_q, n_kv,
                                      H, D, top_k, _ptr(r), r.size, _ptr(idx), _ptr(sc))
    if rc:
        raise RuntimeError(f"lid_oracle_topk_e4m3 failed with code {rc}")
    return idx, sc


def topk_inputs(inp, rows=None):
    """`topk` (or `topk_e4m3`) on a `lid_inputs.Inputs` record."""
    if inp.dtype == "e4m3":
        return topk_e4m3(inp.q_bits, inp.q_scale, inp.k_bits, inp.k_scale, inp.w, inp.mask, inp.H, inp.D,
                         inp.top_k, rows)
    return topk(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.top_k, inp.dtype, rows)


def scores_inputs(inp, rows=None):
    """`scores` (or `scores_e4m3`) on a `lid_inputs.Inputs` record."""
    if inp.dtype == "e4m3":
        return scores_e4m3(inp.q_bits, inp.q_scale, inp.k_bits, inp.k_scale, inp.w, inp.mask, inp.H, inp.D, rows)
    return scores(inp.q_bits, inp.k_bits, inp.w, inp.mask, inp.H, inp.D, inp.dtype, rows)


def sparse_attn(qa_bits, kv_bits, idx, sel_score, Ha, Dc, scale, dtype="bf16", rows=None):
    """fp64 sparse attention over the selected latent rows (the consumer of the
    top-k): qa_bits [n_q, Ha, Dc] and kv_bits [n_kv, Dc] bf16/f16 bits, idx
    [n_q, top_k] int32 (-1: none), sel_score [n_q, top_k] f32 or None (-inf:
    not a selection). Returns (out [rows, Ha, Dc], lse [rows, Ha])."""
    qa = np.ascontiguousarray(qa_bits, dtype=np.uint16)
    kv = np.ascontiguousarray(kv_bits, dtype=np.uint16)
    ix = np.ascontiguousarray(idx, dtype=np.int32)
    sc = None if sel_score is None else np.ascontiguousarray(sel_score, dtype=np.float32)
    n_q = qa.size // (Ha * Dc)
    n_kv = kv.size // Dc
    top_k = ix.size // max(n_q, 1) if n_q else 1
    r = np.arange(n_q, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((r.size, Ha, Dc), dtype=np.float64)
    lse = np.empty((r.size, Ha), dtype=np.float64)
    rc = _load().lid_oracle_sparse_attn(_ptr(qa), _ptr(kv), _ptr(ix), _ptr(sc), n_q, n_kv, Ha, Dc, top_k,
                                        int(dtype == "f16"), float(scale), _ptr(r), r.size, _ptr(out), _ptr(lse))
    if rc:
        raise RuntimeError(f"lid_oracle_sparse_attn failed with code {rc}")
    return out, lse


def decode_bf16(b: int) -> float:
    return _load().lid_oracle_decode_bf16(b)


def decode_f16(b: int) -> float:
    return _load().lid_oracle_decode_f16(b)


def decode_e4m3(b: int) -> float:
    return _load().lid_oracle_decode_e4m3(b)


def threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    return _load().lid_oracle_threads()
