"""Shared helpers of the GPU parity tests: moving seeded inputs to the GPU,
running the CUDA path through the C ABI, and comparing it with the oracle.

Comparison rules:
  * exact (integer-valued inputs): indices and scores identical to the
    oracle's, slot by slot (every intermediate is an integer below 2^24, so
    fp32 and fp64 agree exactly);
  * tolerance (float inputs), per row, with o_k the oracle's k-th score:
      - every returned index is valid and unique, padding only past n_kv;
      - each returned score is within 1e-3 * max(|o_s|, |o_k|) of the
        oracle's full-row value o_s of that index;
      - the returned and the oracle index sets differ only in keys whose
        oracle score is within 1e-3 * |o_k| of o_k;
      - slot j's score is within the same tolerance of the oracle's slot j;
      - the row is sorted by score descending.
"""
import numpy as np
import torch

import oracle
import sparse_attention_lightning_lid_gb300 as lid

REL = 1e-3


def to_device(inp, device="cuda"):
    """(q, k, w, mask) on the device; E4M3 codes as uint8 tensors."""
    if inp.dtype == "e4m3":
        q = torch.from_numpy(np.ascontiguousarray(inp.q_bits)).to(device)
        k = torch.from_numpy(np.ascontiguousarray(inp.k_bits)).to(device)
        w = torch.from_numpy(np.ascontiguousarray(inp.w)).to(device)
        m = None
        if inp.mask is not None:
            m = torch.from_numpy(np.ascontiguousarray(inp.mask).view(np.int16)).to(device).view(torch.float16)
        return q, k, w, m
    tdt = torch.float16 if inp.dtype == "f16" else torch.bfloat16
    q = torch.from_numpy(np.ascontiguousarray(inp.q_bits).view(np.int16)).to(device).view(tdt)
    k = torch.from_numpy(np.ascontiguousarray(inp.k_bits).view(np.int16)).to(device).view(tdt)
    w = torch.from_numpy(np.ascontiguousarray(inp.w)).to(device)
    m = None
    if inp.mask is not None:
        m = torch.from_numpy(np.ascontiguousarray(inp.mask).view(np.int16)).to(device).view(torch.float16)
    return q, k, w, m


def scales_to_device(inp, device="cuda"):
    return (torch.from_numpy(np.ascontiguousarray(inp.q_scale)).to(device),
            torch.from_numpy(np.ascontiguousarray(inp.k_scale)).to(device))


def run_gpu(inp, options=None, stream=None, ranges=None):
    """The CUDA path on `inp` (lid_topk_ex, or lid_topk_e4m3 for E4M3 inputs;
    `ranges` = (lo, hi) int32 arrays for the E4M3 form's visible ranges)."""
    q, k, w, m = to_device(inp)
    if inp.dtype == "e4m3":
        qs, ks = scales_to_device(inp)
        lo = hi = None
        if ranges is not None:
            lo, hi = (torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda() for a in ranges)
            m = None
        idx, sc = lid.topk_e4m3(q, qs, k, ks, w, m, inp.top_k, row_lo=lo, row_hi=hi, options=options,
                                stream=stream)
    else:
        idx, sc = lid.topk(q, k, w, m, inp.top_k, options=options, stream=stream)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


def check_exact(g_idx, g_sc, inp, rows=None):
    o_idx, o_sc = oracle.topk_inputs(inp, rows)
    gi = g_idx if rows is None else g_idx[rows]
    gs = g_sc if rows is None else g_sc[rows]
    bad = np.argwhere(gi != o_idx)
    assert bad.size == 0, f"index mismatch at {bad[:5].tolist()}: gpu {gi[tuple(bad[0])]} oracle {o_idx[tuple(bad[0])]}"
    assert np.array_equal(gs.astype(np.float64), o_sc), "score mismatch"


def check_tolerance(g_idx, g_sc, inp, rows):
    """Returns the worst ratio of a score error to its tolerance over the rows."""
    rows = np.asarray(rows, dtype=np.int64)
    worst = 0.0
    o_idx, o_sc = oracle.topk_inputs(inp, rows)
    full = oracle.scores_inputs(inp, rows)
    k = inp.top_k
    nv = min(k, inp.n_kv)
    for r, t in enumerate(rows):
        gi = g_idx[t].astype(np.int64)
        gs = g_sc[t].astype(np.float64)
        assert np.all(gi[nv:] == -1) and np.all(gs[nv:] == -np.inf), f"row {t}: bad padding"
        gv = gi[:nv]
        assert np.all((gv >= 0) & (gv < inp.n_kv)), f"row {t}: index out of range"
        assert np.unique(gv).size == nv, f"row {t}: duplicate indices"
        ok = full[r][gv]
        ref_k = o_sc[r][nv - 1]
        fin = np.isfinite(ok)
        assert np.array_equal(fin, np.isfinite(gs[:nv])), f"row {t}: -inf pattern differs"
        scale = np.maximum(np.abs(ok[fin]), abs(ref_k) if np.isfinite(ref_k) else 0.0)
        err = np.abs(gs[:nv][fin] - ok[fin])
        assert np.all(err <= REL * scale), f"row {t}: score error {err.max()} > tol"
        if err.size:
            worst = max(worst, float(np.max(err / np.maximum(REL * scale, 1e-300))))
        G, O = set(gv.tolist()), set(o_idx[r][:nv].tolist())
        if np.isfinite(ref_k):
            for s in G ^ O:
                assert abs(full[r][s] - ref_k) <= REL * abs(ref_k), \
                    f"row {t}: key {s} (oracle {full[r][s]}) differs from the oracle set beyond tolerance (k-th {ref_k})"
        else:
            assert G == O, f"row {t}: index sets differ with masked keys in the top-k"
        pos_scale = np.maximum(np.abs(o_sc[r][:nv]), abs(ref_k) if np.isfinite(ref_k) else 0.0)
        pf = np.isfinite(o_sc[r][:nv])
        assert np.all(np.abs(gs[:nv][pf] - o_sc[r][:nv][pf]) <= REL * pos_scale[pf]), f"row {t}: slot scores differ"
        d = np.diff(gs[:nv])
        assert np.all((d <= 0) | np.isnan(d)), f"row {t}: not sorted descending"
    return worst
