"""GB300 (sm_103a) lightning-indexer top-k: Python binding of the C ABI.

The library (`liblid.so`, built in-tree from `csrc/` by `build()`) computes,
for every query t, the top_k keys of

    I[t,s] = sum_h w[t,h] * relu(q[t,h,:] . k[s,:]) + mask[t,s]

(DeepSeek-V4-Flash lightning indexer: llama.cpp issue 25468, root-cause
comment; fairydreaming/llama.cpp PR 2, API-change note) without forming the
n_q x n_kv score matrix. This module only marshals arguments: every step of
the computation runs in the CUDA kernels behind `include/lid.h`. PyTorch
provides device memory and streams. There is no fallback: if the library is
missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
LIB_PATH = os.path.join(_HERE, "_lib", "liblid.so")
SOURCES = ["lid_api.cu", "lid_attn.cu"]
HEADERS = ["lid_kernels.cuh", "lid_ptx.cuh", "lid_select.cuh", "lid_stream.cuh", "lid_attn.cuh", "lid_attn_tc.cuh",
           "lid_internal.h"]

(LID_OK, LID_ERR_INVALID_ARG, LID_ERR_UNSUPPORTED, LID_ERR_OOM, LID_ERR_CUDA, LID_ERR_DEVICE_TIMEOUT,
 LID_ERR_SCRATCH_TOO_SMALL) = range(7)
DTYPE_BF16, DTYPE_F16, DTYPE_E4M3 = 0, 1, 2

# symbols include/lid.h declares
EXPORTS = ("lid_topk", "lid_topk_f16", "lid_topk_ex", "lid_topk_ranges", "lid_topk_e4m3", "lid_topk_host",
           "lid_topk_host_async", "lid_topk_ws", "lid_topk_static", "lid_plan", "lid_sparse_attn", "lid_sparse_attn_plan",
           "lid_device_error", "lid_last_cuda_error", "lid_status_string")


def _nvcc() -> str:
    nvcc = os.environ.get("NVCC", "nvcc")
    if os.path.exists("/usr/local/cuda/bin/nvcc") and nvcc == "nvcc":
        nvcc = "/usr/local/cuda/bin/nvcc"
    return nvcc


def nvcc_commands(out_path: str = LIB_PATH):
    """(compile commands, one per translation unit, run in parallel; link command)."""
    flags = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-I", _INCLUDE]
    objs = [out_path + "." + os.path.splitext(s)[0] + ".o" for s in SOURCES]
    compiles = [[_nvcc()] + flags + ["-c", os.path.join(_CSRC, s), "-o", o] for s, o in zip(SOURCES, objs)]
    link = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", out_path] + objs
    return compiles, link, objs


def _stale(out_path: str) -> bool:
    if not os.path.exists(out_path):
        return True
    t = os.path.getmtime(out_path)
    deps = [os.path.join(_CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(_INCLUDE, "lid.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/ for sm_103a into _lib/liblid.so (in-tree). Returns its path."""
    if force or _stale(LIB_PATH):
        os.makedirs(os.path.dirname(LIB_PATH), exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        compiles, link, objs = nvcc_commands(tmp)
        procs = []
        for cmd in compiles:
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((cmd, subprocess.Popen(cmd)))
        failed = [cmd for cmd, pr in procs if pr.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        if verbose:
            print(" ".join(link), file=sys.stderr)
        subprocess.check_call(link)
        for o in objs:
            os.remove(o)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


class LidError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = ""
        if status == LID_ERR_CUDA and _lib is not None:
            detail = f" [{_lib.lid_last_cuda_error().decode()}]"
        super().__init__(f"{what}: {status_string(status)} (status {status}){detail}")


class Options(ctypes.Structure):
    """lid_options: tuning / test overrides (zeros = planned defaults)."""
    _fields_ = [("force_splits", ctypes.c_int), ("force_qg", ctypes.c_int), ("force_kstages", ctypes.c_int),
                ("fault_inject", ctypes.c_int), ("ev_score_begin", ctypes.c_void_p),
                ("ev_score_end", ctypes.c_void_p), ("path", ctypes.c_int), ("early_tiles", ctypes.c_int),
                ("plan_ranges", ctypes.c_int), ("reserved", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("qg", ctypes.c_int), ("n_groups", ctypes.c_int), ("splits", ctypes.c_int),
                ("tiles_per_split", ctypes.c_int), ("kstages", ctypes.c_int), ("acc_stages", ctypes.c_int),
                ("cap", ctypes.c_int), ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("fused", ctypes.c_int), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class AttnOptions(ctypes.Structure):
    """lid_attn_options: test overrides of lid_sparse_attn (zeros = planned)."""
    _fields_ = [("force_splits", ctypes.c_int), ("force_head_groups", ctypes.c_int), ("path", ctypes.c_int),
                ("reserved", ctypes.c_int)]


class AttnPlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("head_groups", ctypes.c_int), ("splits", ctypes.c_int),
                ("keys_per_split", ctypes.c_int), ("ctas", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None


def load(path: str = LIB_PATH):
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing; call "
                           "sparse_attention_lightning_lid_gb300.build() first")
    lib = ctypes.CDLL(path)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    args = [P, P, P, P, I64, I64, I, I, I, P, P, P]
    lib.lid_topk.argtypes = args
    lib.lid_topk_f16.argtypes = args
    lib.lid_topk_ex.argtypes = args + [I, ctypes.POINTER(Options)]
    lib.lid_topk_ranges.argtypes = [P, P, P, P, P, I64, I64, I, I, I, P, P, P, I, ctypes.POINTER(Options)]
    lib.lid_topk_e4m3.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I, I, I, P, P, P, ctypes.POINTER(Options)]
    lib.lid_topk_host.argtypes = args + [I]
    lib.lid_topk_host_async.argtypes = args + [I]
    lib.lid_topk_ws.argtypes = [P, P, P, P, P, P, P, P, I64, I64, I, I, I, P, P, P, I64, P, I, ctypes.POINTER(Options)]
    lib.lid_topk_static.argtypes = args + [I]
    lib.lid_plan.argtypes = [I64, I64, I, I, I, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]
    lib.lid_sparse_attn.argtypes = [P, P, P, P, I64, I64, I, I, I, ctypes.c_float, P, P, P, I64, P, I,
                                    ctypes.POINTER(AttnOptions)]
    lib.lid_sparse_attn_plan.argtypes = [I64, I64, I, I, I, ctypes.POINTER(AttnOptions),
                                         ctypes.POINTER(AttnPlanInfo)]
    lib.lid_device_error.argtypes = [I]
    lib.lid_status_string.argtypes = [I]
    lib.lid_status_string.restype = ctypes.c_char_p
    lib.lid_last_cuda_error.argtypes = []
    lib.lid_last_cuda_error.restype = ctypes.c_char_p
    for f in ("lid_topk", "lid_topk_f16", "lid_topk_ex", "lid_topk_ranges", "lid_topk_e4m3", "lid_topk_host",
              "lid_topk_host_async", "lid_topk_ws", "lid_topk_static", "lid_plan", "lid_sparse_attn", "lid_sparse_attn_plan",
              "lid_device_error"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().lid_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float16:
        return DTYPE_F16
    raise TypeError(f"q and k must be bfloat16 or float16, got {t.dtype}")


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def topk(q, k, w, mask, top_k: int, out_idx=None, out_score=None, stream=None, options: Options | None = None):
    """Top-k of the lightning-indexer score on the GPU.

    q [n_q, H, D] and k [n_kv, D]: bf16 or f16 CUDA tensors of one dtype;
    w [n_q, H] float32; mask [n_q, n_kv] float16 (or int16 f16 bits) or None.
    Returns (out_idx int32 [n_q, top_k], out_score float32 [n_q, top_k]),
    rows sorted by score descending then index ascending. Asynchronous on
    `stream` (default: the current torch stream).
    """
    import torch
    if q.dim() != 3 or k.dim() != 2 or w.dim() != 2:
        raise ValueError("expected q [n_q, H, D], k [n_kv, D], w [n_q, H]")
    n_q, H, D = q.shape
    n_kv = k.shape[0]
    if k.shape[1] != D or tuple(w.shape) != (n_q, H) or k.dtype != q.dtype:
        raise ValueError("shape or dtype mismatch between q, k and w")
    if w.dtype != torch.float32:
        raise TypeError("w must be float32")
    for name, t in (("q", q), ("k", k), ("w", w)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if mask is not None:
        if tuple(mask.shape) != (n_q, n_kv) or mask.element_size() != 2 or not mask.is_cuda or \
                not mask.is_contiguous():
            raise ValueError("mask must be a contiguous [n_q, n_kv] CUDA tensor of f16 values or bits")
    dev = q.device
    if out_idx is None:
        out_idx = torch.empty((n_q, top_k), dtype=torch.int32, device=dev)
    if out_score is None:
        out_score = torch.empty((n_q, top_k), dtype=torch.float32, device=dev)
    opt = ctypes.byref(options) if options is not None else None
    rc = load().lid_topk_ex(q.data_ptr(), k.data_ptr(), w.data_ptr(),
                            None if mask is None else mask.data_ptr(), n_q, n_kv, H, D, top_k,
                            out_idx.data_ptr(), out_score.data_ptr(), _stream_ptr(stream), _dtype_code(q), opt)
    if rc != LID_OK:
        raise LidError(rc, "lid_topk_ex")
    return out_idx, out_score


def topk_ranges(q, k, w, row_lo, row_hi, top_k: int, out_idx=None, out_score=None, stream=None,
                options: Options | None = None):
    """topk() with one visible key range per query instead of a mask: row t
    sees keys row_lo[t] <= s < row_hi[t] (int32 CUDA tensors [n_q]); every
    other key scores -inf."""
    import torch
    if q.dim() != 3 or k.dim() != 2 or w.dim() != 2:
        raise ValueError("expected q [n_q, H, D], k [n_kv, D], w [n_q, H]")
    n_q, H, D = q.shape
    n_kv = k.shape[0]
    if k.shape[1] != D or tuple(w.shape) != (n_q, H) or k.dtype != q.dtype or w.dtype != torch.float32:
        raise ValueError("shape or dtype mismatch between q, k and w")
    for name, t in (("q", q), ("k", k), ("w", w), ("row_lo", row_lo), ("row_hi", row_hi)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if row_lo.dtype != torch.int32 or row_hi.dtype != torch.int32 or row_lo.numel() != n_q or \
            row_hi.numel() != n_q:
        raise ValueError("row_lo and row_hi must be int32 tensors of n_q entries")
    if out_idx is None:
        out_idx = torch.empty((n_q, top_k), dtype=torch.int32, device=q.device)
    if out_score is None:
        out_score = torch.empty((n_q, top_k), dtype=torch.float32, device=q.device)
    opt = ctypes.byref(options) if options is not None else None
    rc = load().lid_topk_ranges(q.data_ptr(), k.data_ptr(), w.data_ptr(), row_lo.data_ptr(), row_hi.data_ptr(),
                                n_q, n_kv, H, D, top_k, out_idx.data_ptr(), out_score.data_ptr(),
                                _stream_ptr(stream), _dtype_code(q), opt)
    if rc != LID_OK:
        raise LidError(rc, "lid_topk_ranges")
    return out_idx, out_score


def topk_e4m3(q8, q_scale, k8, k_scale, w, mask, top_k: int, row_lo=None, row_hi=None, out_idx=None,
              out_score=None, stream=None, options: Options | None = None):
    """topk() with quantised operands (lid_topk_e4m3): q8 [n_q, H, D] and
    k8 [n_kv, D] E4M3 codes (uint8 or torch.float8_e4m3fn CUDA tensors),
    q_scale [n_q, H] and k_scale [n_kv] float32 (finite, >= 0); element values
    are scale * code value. D must be 128. Either mask ([n_q, n_kv] f16 or
    None) or row_lo/row_hi (int32 [n_q] visible ranges, mask None)."""
    import torch
    if q8.dim() != 3 or k8.dim() != 2 or w.dim() != 2:
        raise ValueError("expected q8 [n_q, H, D], k8 [n_kv, D], w [n_q, H]")
    n_q, H, D = q8.shape
    n_kv = k8.shape[0]
    if k8.shape[1] != D or tuple(w.shape) != (n_q, H) or tuple(q_scale.shape) != (n_q, H) or \
            tuple(k_scale.shape) != (n_kv,):
        raise ValueError("shape mismatch between q8, q_scale, k8, k_scale and w")
    if q8.element_size() != 1 or k8.element_size() != 1:
        raise TypeError("q8 and k8 must hold 8-bit codes")
    if w.dtype != torch.float32 or q_scale.dtype != torch.float32 or k_scale.dtype != torch.float32:
        raise TypeError("w, q_scale and k_scale must be float32")
    named = [("q8", q8), ("q_scale", q_scale), ("k8", k8), ("k_scale", k_scale), ("w", w)]
    if mask is not None:
        if tuple(mask.shape) != (n_q, n_kv) or mask.element_size() != 2:
            raise ValueError("mask must be [n_q, n_kv] f16 values or bits")
        named.append(("mask", mask))
    if (row_lo is None) != (row_hi is None):
        raise ValueError("row_lo and row_hi go together")
    if row_lo is not None:
        if row_lo.dtype != torch.int32 or row_hi.dtype != torch.int32 or row_lo.numel() != n_q or \
                row_hi.numel() != n_q:
            raise ValueError("row_lo and row_hi must be int32 tensors of n_q entries")
        named += [("row_lo", row_lo), ("row_hi", row_hi)]
    for name, t in named:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out_idx is None:
        out_idx = torch.empty((n_q, top_k), dtype=torch.int32, device=q8.device)
    if out_score is None:
        out_score = torch.empty((n_q, top_k), dtype=torch.float32, device=q8.device)
    opt = ctypes.byref(options) if options is not None else None
    def ptr(t):
        return None if t is None else t.data_ptr()

    rc = load().lid_topk_e4m3(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(), w.data_ptr(),
                              ptr(mask), ptr(row_lo), ptr(row_hi), n_q, n_kv, H, D, top_k, out_idx.data_ptr(),
                              out_score.data_ptr(), _stream_ptr(stream), opt)
    if rc != LID_OK:
        raise LidError(rc, "lid_topk_e4m3")
    return out_idx, out_score


def workspace(n_q: int, n_kv: int, H: int, D: int, top_k: int, options: Options | None = None, device="cuda"):
    """A zeroed workspace for topk_ws() of this shape (None when the shape needs
    none). Zero once; every call leaves its counter area zero again."""
    import torch
    nbytes = plan(n_q, n_kv, H, D, top_k, options)["workspace_bytes"]
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes > 0 else None


def topk_ws(q, k, w, top_k: int, ws, mask=None, row_lo=None, row_hi=None, q_scale=None, k_scale=None,
            out_idx=None, out_score=None, stream=None, options: Options | None = None):
    """topk() / topk_ranges() / topk_e4m3() with a caller-owned workspace
    (lid_topk_ws): `ws` is a CUDA uint8 tensor of at least lid_plan's
    workspace_bytes whose first 1024 bytes are zero before its first use (see
    workspace()); the call allocates nothing. q / k are bf16 or f16, or E4M3
    codes (uint8 / float8_e4m3fn) with q_scale and k_scale."""
    import torch
    if q.dim() != 3 or k.dim() != 2 or w.dim() != 2:
        raise ValueError("expected q [n_q, H, D], k [n_kv, D], w [n_q, H]")
    n_q, H, D = q.shape
    n_kv = k.shape[0]
    e4m3 = q.element_size() == 1
    if e4m3:
        dtype = DTYPE_E4M3
        if q_scale is None or k_scale is None:
            raise ValueError("E4M3 operands need q_scale and k_scale")
        if tuple(q_scale.shape) != (n_q, H) or tuple(k_scale.shape) != (n_kv,):
            raise ValueError("q_scale must be [n_q, H] and k_scale [n_kv]")
    else:
        dtype = _dtype_code(q)
    if k.shape[1] != D or tuple(w.shape) != (n_q, H) or k.element_size() != q.element_size() or \
            w.dtype != torch.float32:
        raise ValueError("shape or dtype mismatch between q, k and w")
    if (row_lo is None) != (row_hi is None):
        raise ValueError("row_lo and row_hi go together")
    named = [("q", q), ("k", k), ("w", w)]
    for name, t in (("mask", mask), ("row_lo", row_lo), ("row_hi", row_hi), ("q_scale", q_scale),
                    ("k_scale", k_scale), ("ws", ws)):
        if t is not None:
            named.append((name, t))
    for name, t in named:
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out_idx is None:
        out_idx = torch.empty((n_q, top_k), dtype=torch.int32, device=q.device)
    if out_score is None:
        out_score = torch.empty((n_q, top_k), dtype=torch.float32, device=q.device)

    def ptr(t):
        return None if t is None else t.data_ptr()

    opt = ctypes.byref(options) if options is not None else None
    rc = load().lid_topk_ws(q.data_ptr(), ptr(q_scale), k.data_ptr(), ptr(k_scale), w.data_ptr(), ptr(mask),
                            ptr(row_lo), ptr(row_hi), n_q, n_kv, H, D, top_k, out_idx.data_ptr(),
                            out_score.data_ptr(), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                            _stream_ptr(stream), dtype, opt)
    if rc != LID_OK:
        raise LidError(rc, "lid_topk_ws")
    return out_idx, out_score


def _host_call(fn: str, q_bits, k_bits, w, mask_bits, H: int, D: int, top_k: int, dtype: str, out_idx, out_score,
               stream):
    import numpy as np
    import torch

    def ptr(a):
        if a is None:
            return None
        return a.data_ptr() if isinstance(a, torch.Tensor) else a.ctypes.data

    n_q = (q_bits.numel() if isinstance(q_bits, torch.Tensor) else q_bits.size) // (H * D)
    n_kv = (k_bits.numel() if isinstance(k_bits, torch.Tensor) else k_bits.size) // D
    if out_idx is None:
        out_idx = np.empty((n_q, top_k), np.int32)
    if out_score is None:
        out_score = np.empty((n_q, top_k), np.float32)
    rc = getattr(load(), fn)(ptr(q_bits), ptr(k_bits), ptr(w), ptr(mask_bits), n_q, n_kv, H, D, top_k,
                             ptr(out_idx), ptr(out_score), _stream_ptr(stream),
                             DTYPE_F16 if dtype == "f16" else DTYPE_BF16)
    if rc != LID_OK:
        raise LidError(rc, fn)
    return out_idx, out_score


def topk_host(q_bits, k_bits, w, mask_bits, H: int, D: int, top_k: int, dtype: str = "bf16",
              out_idx=None, out_score=None, stream=None):
    """Host-buffer form (lid_topk_host): numpy or pinned CPU torch buffers in,
    host buffers out; copies and the kernels run on `stream` and the call
    returns after they finish. q_bits/k_bits hold bf16 or f16 bit patterns."""
    return _host_call("lid_topk_host", q_bits, k_bits, w, mask_bits, H, D, top_k, dtype, out_idx, out_score,
                      stream)


def topk_host_async(q_bits, k_bits, w, mask_bits, H: int, D: int, top_k: int, out_idx, out_score,
                    dtype: str = "bf16", stream=None):
    """lid_topk_host_async: as topk_host, but the call returns once the copies
    and kernels are enqueued on `stream`. out_idx / out_score are the caller's
    host buffers (pinned CPU tensors for the copies to be asynchronous); they
    hold the result, and the inputs must stay alive and unchanged, until the
    stream is synchronised."""
    return _host_call("lid_topk_host_async", q_bits, k_bits, w, mask_bits, H, D, top_k, dtype, out_idx,
                      out_score, stream)


def plan(n_q: int, n_kv: int, H: int, D: int, top_k: int, options: Options | None = None) -> dict:
    """The launch plan lid_topk_ex would use on the current device."""
    info = PlanInfo()
    rc = load().lid_plan(n_q, n_kv, H, D, top_k, ctypes.byref(options) if options is not None else None,
                         ctypes.byref(info))
    if rc != LID_OK:
        raise LidError(rc, "lid_plan")
    return info.as_dict()


def sparse_attn(qa, kv, idx, scale: float, sel_score=None, out=None, lse=None, ws=None, stream=None,
                options: AttnOptions | None = None):
    """Sparse attention over the selected latent rows (lid_sparse_attn): qa
    [n_q, Ha, Dc] and kv [n_kv, Dc] bf16/f16 CUDA tensors, idx [n_q, top_k]
    int32 (e.g. topk()'s indices), sel_score [n_q, top_k] f32 or None (e.g.
    topk()'s scores: -inf drops a selection). Returns (out [n_q, Ha, Dc] f32,
    lse [n_q, Ha] f32). `ws`: optional caller-owned uint8 workspace of
    attn_plan()'s workspace_bytes (else the library allocates it on the stream)."""
    import torch
    if qa.dim() != 3 or kv.dim() != 2 or idx.dim() != 2:
        raise ValueError("expected qa [n_q, Ha, Dc], kv [n_kv, Dc], idx [n_q, top_k]")
    n_q, Ha, Dc = qa.shape
    n_kv = kv.shape[0]
    top_k = idx.shape[1]
    if kv.shape[1] != Dc or kv.dtype != qa.dtype or idx.shape[0] != n_q or idx.dtype != torch.int32:
        raise ValueError("shape or dtype mismatch between qa, kv and idx")
    if sel_score is not None and (tuple(sel_score.shape) != tuple(idx.shape) or sel_score.dtype != torch.float32):
        raise ValueError("sel_score must be f32 of idx's shape")
    for name, t in (("qa", qa), ("kv", kv), ("idx", idx), ("sel_score", sel_score), ("ws", ws)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty((n_q, Ha, Dc), dtype=torch.float32, device=qa.device)
    if lse is None:
        lse = torch.empty((n_q, Ha), dtype=torch.float32, device=qa.device)
    rc = load().lid_sparse_attn(qa.data_ptr(), kv.data_ptr() if n_kv else None, idx.data_ptr(),
                                None if sel_score is None else sel_score.data_ptr(), n_q, n_kv, Ha, Dc, top_k,
                                float(scale), out.data_ptr(), lse.data_ptr(), None if ws is None else ws.data_ptr(),
                                0 if ws is None else ws.numel() * ws.element_size(), _stream_ptr(stream),
                                _dtype_code(qa), ctypes.byref(options) if options is not None else None)
    if rc != LID_OK:
        raise LidError(rc, "lid_sparse_attn")
    return out, lse


def attn_plan(n_q: int, n_kv: int, Ha: int, Dc: int, top_k: int, options: AttnOptions | None = None) -> dict:
    """The launch plan lid_sparse_attn would use on the current device."""
    info = AttnPlanInfo()
    rc = load().lid_sparse_attn_plan(n_q, n_kv, Ha, Dc, top_k,
                                     ctypes.byref(options) if options is not None else None, ctypes.byref(info))
    if rc != LID_OK:
        raise LidError(rc, "lid_sparse_attn_plan")
    return info.as_dict()


def device_error(reset: bool = False) -> int:
    """First device-side wait timeout code recorded (0 = none). Synchronises."""
    return load().lid_device_error(1 if reset else 0)
