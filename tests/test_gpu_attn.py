"""Parity of lid_sparse_attn (sparse attention over the selected latent rows,
the consumer of the top-k) with the fp64 oracle, through the C ABI.

Tolerance, from the kernel's arithmetic: products of 16-bit inputs are exact in
fp32; the scores are fp32 sums of Dc = 512 products; each softmax weight p_j
is computed in fp32, summed unrounded into the normaliser, and rounded to the
input type (relative error delta_j <= 2^-9 for bf16) for the weighted sum of
the rows. The output is then sum_j w_j (1 + delta_j) v_j with sum_j w_j = 1,
so it is within 2^-9 * max_j |v_j| of the exact result, plus the effect of the
scores' fp32 rounding (below 5e-4 relative on these inputs). The test allows

    |out - oracle| <= 3e-3 * max |kv row selected by the query| + 1e-6
    |lse - oracle| <= 1e-3 + 1e-5 * |oracle lse|

element by element, over every row it runs.
"""
import numpy as np
import pytest
import torch

import lid_inputs as li
import oracle
import sparse_attention_lightning_lid_gb300 as lid

pytestmark = pytest.mark.gpu

OUT_REL = 3e-3
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lid.load()
    yield


def _tdt(dtype):
    return torch.float16 if dtype == "f16" else torch.bfloat16


def _dev(a):
    qa = torch.from_numpy(np.ascontiguousarray(a.qa_bits).view(np.int16)).cuda().view(_tdt(a.dtype))
    kv = torch.from_numpy(np.ascontiguousarray(a.kv_bits).view(np.int16)).cuda().view(_tdt(a.dtype))
    idx = torch.from_numpy(np.ascontiguousarray(a.idx)).cuda()
    sc = None if a.sel_score is None else torch.from_numpy(np.ascontiguousarray(a.sel_score)).cuda()
    return qa, kv, idx, sc


def _vmax(a, rows):
    """max |kv| over each row's valid selections (0 when there are none)."""
    if a.dtype == "bf16":
        kv = np.abs((a.kv_bits.astype(np.uint32) << 16).view(np.float32))
    else:
        kv = np.abs(a.kv_bits.view(np.float16).astype(np.float32))
    row_max = kv.max(axis=1) if kv.size else np.zeros(0, np.float32)
    out = np.zeros(len(rows))
    for i, t in enumerate(rows):
        sel = a.idx[t]
        ok = (sel >= 0) & (sel < a.n_kv)
        if a.sel_score is not None:
            ok &= a.sel_score[t] != -np.inf
        out[i] = row_max[sel[ok]].max() if ok.any() else 0.0
    return out


def _check(a, out, lse, rows=None):
    rows = np.arange(a.n_q) if rows is None else np.asarray(rows)
    o_out, o_lse = oracle.sparse_attn(a.qa_bits, a.kv_bits, a.idx, a.sel_score, a.Ha, a.Dc, a.scale,
                                      dtype=a.dtype, rows=rows)
    g_out = out.cpu().numpy()[rows].astype(np.float64)
    g_lse = lse.cpu().numpy()[rows].astype(np.float64)
    vmax = _vmax(a, rows)
    err = np.abs(g_out - o_out).max(axis=(1, 2))
    tol = OUT_REL * vmax + 1e-6
    assert np.all(err <= tol), (rows[err > tol][:5], err[err > tol][:5], tol[err > tol][:5])
    empty = np.isneginf(o_lse)
    assert np.array_equal(np.isneginf(g_lse), empty)
    fin = ~empty
    lerr = np.abs(g_lse[fin] - o_lse[fin])
    assert np.all(lerr <= LSE_ABS + 1e-5 * np.abs(o_lse[fin])), lerr.max()
    assert np.all(g_out[empty] == 0.0)
    return float((err / tol).max()) if len(rows) else 0.0


def _run(a, options=None, ws=None):
    qa, kv, idx, sc = _dev(a)
    out, lse = lid.sparse_attn(qa, kv, idx, a.scale, sel_score=sc, ws=ws, options=options)
    torch.cuda.synchronize()
    return out, lse


SMALL = [
    # n_q, n_kv, Ha, top_k, n_invalid, splits, head groups, dtype
    (3, 700, 16, 200, 5, 0, 0, "bf16"),       # ragged last chunk (200 = 3 * 64 + 8)
    (5, 2000, 32, 130, 7, 2, 0, "bf16"),
    (2, 900, 64, 64, 0, 1, 4, "f16"),
    (4, 3000, 64, 512, 9, 3, 2, "bf16"),
    (2, 500, 128, 257, 3, 0, 0, "bf16"),      # two head blocks
    (1, 1000, 64, 1, 0, 0, 0, "bf16"),        # one selection
    (3, 4096, 64, 2048, 11, 0, 0, "f16"),     # the largest top_k
    (40, 1500, 64, 300, 4, 0, 0, "bf16"),     # several queries per planned wave
    (200, 1024, 64, 96, 2, 0, 0, "bf16"),     # all heads per CTA, one split
]


@pytest.mark.parametrize("n_q,n_kv,Ha,top_k,n_inv,splits,G,dtype", SMALL)
def test_sparse_attn_matches_oracle(n_q, n_kv, Ha, top_k, n_inv, splits, G, dtype):
    """The warp-level MMA kernel (path 1)."""
    a = li.attn_inputs("s", n_q, n_kv, Ha, 512, top_k, seed=n_q * 7 + top_k, n_invalid=n_inv, dtype=dtype)
    opt = lid.AttnOptions()
    opt.force_splits, opt.force_head_groups, opt.path = splits, G, 1
    assert lid.attn_plan(n_q, n_kv, Ha, 512, top_k, opt)["path"] == 1
    out, lse = _run(a, opt)
    _check(a, out, lse)


@pytest.mark.parametrize("n_q,n_kv,Ha,top_k,n_inv,splits,G,dtype", [c for c in SMALL if c[2] % 64 == 0])
def test_tensor_core_kernel_matches_oracle(n_q, n_kv, Ha, top_k, n_inv, splits, G, dtype):
    """The tcgen05 kernel (path 2): 64 heads per CTA, chunks of 128 keys."""
    a = li.attn_inputs("s", n_q, n_kv, Ha, 512, top_k, seed=n_q * 7 + top_k, n_invalid=n_inv, dtype=dtype)
    opt = lid.AttnOptions()
    opt.force_splits, opt.path = splits, 2
    p = lid.attn_plan(n_q, n_kv, Ha, 512, top_k, opt)
    assert p["path"] == 2 and p["keys_per_split"] % 128 == 0
    out, lse = _run(a, opt)
    _check(a, out, lse)


def test_every_split_and_head_grouping_agrees():
    a = li.attn_inputs("s", 3, 5000, 64, 512, 450, seed=91, n_invalid=6)
    for G in (1, 2, 4):
        for S in (1, 2, 3, 8):
            opt = lid.AttnOptions()
            opt.force_splits, opt.force_head_groups, opt.path = S, G, 1
            p = lid.attn_plan(3, 5000, 64, 512, 450, opt)
            assert p["head_groups"] == G and p["splits"] == min(S, 8)
            out, lse = _run(a, opt)
            _check(a, out, lse)
    for S in (1, 2, 3, 4):
        opt = lid.AttnOptions()
        opt.force_splits, opt.path = S, 2
        p = lid.attn_plan(3, 5000, 64, 512, 450, opt)
        kps = -(-4 // S) * 128  # 450 selections = 4 chunks of 128, split as evenly as whole chunks allow
        assert p["keys_per_split"] == kps and p["splits"] == -(-450 // kps)
        out, lse = _run(a, opt)
        _check(a, out, lse)


@pytest.mark.parametrize("path", [1, 2])
def test_running_maximum_that_moves_late(path):
    """Selections ordered from small-norm to large-norm rows: the logits of the
    later chunks exceed the first chunk's maximum by far more than 2^8 in the
    exponent, so the tensor-core kernel must move its running maxima and
    rescale the output accumulated so far (and the other kernel its usual
    online rescaling)."""
    n_q, n_kv, Ha, top_k = 3, 3000, 64, 512
    a = li.attn_inputs("m", n_q, n_kv, Ha, 512, top_k, seed=77)
    kv = (a.kv_bits.astype(np.uint32) << 16).view(np.float32).copy()
    big = np.zeros(n_kv, bool)
    for t in range(n_q):
        big[a.idx[t, 256:]] = True  # the last two chunks of 128
    big[np.concatenate([a.idx[t, :256] for t in range(n_q)])] = False
    kv[big] *= 4.0
    kv[~big] *= 0.25
    a.kv_bits[:] = li.f32_to_bf16_bits(kv)
    opt = lid.AttnOptions()
    opt.path = path
    out, lse = _run(a, opt)
    _check(a, out, lse)


def test_results_are_deterministic():
    a = li.attn_inputs("s", 4, 3000, 64, 512, 512, seed=5)
    o1, l1 = _run(a)
    o2, l2 = _run(a)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_no_selection_rows_and_empty_kv():
    a = li.attn_inputs("s", 4, 800, 64, 512, 128, seed=12, n_invalid=3)
    a.idx[1] = -1
    a.sel_score[2] = -np.inf
    a.idx[3, :64] = 10_000  # past n_kv: not a selection
    for splits in (0, 2):
        opt = lid.AttnOptions()
        opt.force_splits = splits
        out, lse = _run(a, opt)
        _check(a, out, lse)
        o, l_ = out.cpu().numpy(), lse.cpu().numpy()
        assert np.all(o[1] == 0) and np.all(np.isneginf(l_[1]))
        assert np.all(o[2] == 0) and np.all(np.isneginf(l_[2]))
    # no rows at all
    qa = torch.randn(2, 64, 512, device="cuda").to(torch.bfloat16)
    kv = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(2, 16, dtype=torch.int32, device="cuda")
    out, lse = lid.sparse_attn(qa, kv, idx, 0.1)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    # no queries: nothing to do
    out, lse = lid.sparse_attn(qa[:0], kv, idx[:0], 0.1)
    assert out.shape == (0, 64, 512)


def test_without_selection_scores():
    a = li.attn_inputs("s", 3, 1200, 32, 512, 192, seed=14, n_invalid=4)
    a2 = li.AttnInputs(a.name, a.n_q, a.n_kv, a.Ha, a.Dc, a.top_k, a.qa_bits, a.kv_bits, a.idx, None, a.scale)
    out, lse = _run(a2)
    _check(a2, out, lse)


def test_caller_workspace_and_graph_capture():
    a = li.attn_inputs("s", 2, 4000, 64, 512, 512, seed=21, n_invalid=5)
    opt = lid.AttnOptions()
    opt.force_splits = 4
    p = lid.attn_plan(2, 4000, 64, 512, 512, opt)
    assert p["splits"] == 4 and p["workspace_bytes"] == 2 * 4 * 64 * (512 * 4 + 8)
    qa, kv, idx, sc = _dev(a)
    ws = torch.empty(p["workspace_bytes"], dtype=torch.uint8, device="cuda")
    out = torch.empty(2, 64, 512, device="cuda")
    lse = torch.empty(2, 64, device="cuda")
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        lid.sparse_attn(qa, kv, idx, a.scale, sel_score=sc, out=out, lse=lse, ws=ws, options=opt)
    st.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    _check(a, out, lse)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        lid.sparse_attn(qa, kv, idx, a.scale, sel_score=sc, out=out, lse=lse, ws=ws, options=opt, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


def test_errors_leave_outputs_untouched():
    qa = torch.zeros(2, 64, 512, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(100, 512, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(2, 128, dtype=torch.int32, device="cuda")
    out = torch.full((2, 64, 512), 7.0, device="cuda")
    lse = torch.full((2, 64), 7.0, device="cuda")
    L = lid.load()

    def call(qa_p=qa.data_ptr(), Ha=64, Dc=512, top_k=128, scale=0.1, ws=None, ws_bytes=0, dtype=lid.DTYPE_BF16,
             opt=None):
        return L.lid_sparse_attn(qa_p, kv.data_ptr(), idx.data_ptr(), None, 2, 100, Ha, Dc, top_k, scale,
                                 out.data_ptr(), lse.data_ptr(), ws, ws_bytes,
                                 torch.cuda.current_stream().cuda_stream, dtype, opt)

    assert call(Ha=48) == lid.LID_ERR_UNSUPPORTED
    assert call(Dc=256) == lid.LID_ERR_UNSUPPORTED
    assert call(top_k=0) == lid.LID_ERR_UNSUPPORTED
    assert call(top_k=4096) == lid.LID_ERR_UNSUPPORTED
    assert call(qa_p=qa.data_ptr() + 2) == lid.LID_ERR_INVALID_ARG
    assert call(scale=float("nan")) == lid.LID_ERR_INVALID_ARG
    assert call(dtype=lid.DTYPE_E4M3) == lid.LID_ERR_INVALID_ARG
    opt = lid.AttnOptions()
    opt.force_head_groups = 3
    assert call(opt=ctypes_ref(opt)) == lid.LID_ERR_INVALID_ARG
    opt = lid.AttnOptions()
    opt.force_splits = 2
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert call(ws=small.data_ptr(), ws_bytes=1024, opt=ctypes_ref(opt)) == lid.LID_ERR_SCRATCH_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)
    with pytest.raises(ValueError):
        lid.sparse_attn(qa, kv.to(torch.float16), idx, 0.1)


def ctypes_ref(o):
    import ctypes
    return ctypes.byref(o)


@pytest.mark.parametrize("name", ["attn_decode", "attn_prefill"])
@pytest.mark.parametrize("path", [0, 1, 2])
def test_full_size_workloads_every_row(name, path):
    """The bench's two workloads at full size (planned launch, and each kernel
    forced), every query row against the oracle."""
    a = li.attn_workload(name)
    opt = lid.AttnOptions()
    opt.path = path
    out, lse = _run(a, opt)
    ratio = _check(a, out, lse)
    print(f"{name} path {path}: worst error / tolerance = {ratio:.3f}")


def test_consumes_the_indexer_top_k():
    """The chain the pages describe: the indexer's top-k (lid_topk) feeds the
    attention (lid_sparse_attn) its indices and scores; the oracle side runs
    the oracle's top-k and the oracle's attention. Integer indexer inputs make
    both top-k lists identical, and the causal mask leaves the first queries
    fewer visible keys than top_k, so their lists end in (-1, -inf) padding or
    -inf selections that the attention must drop."""
    n_q, n_kv, H, D, top_k = 6, 1024, 64, 128, 256
    pos0 = 100
    mask = li.causal_mask(n_q, n_kv, pos0)
    ix = li.int_inputs("c", n_q, n_kv, H, D, top_k, seed=33, mask=mask, dtype="bf16", w_range=(-3, 3))
    att = li.attn_inputs("c", n_q, n_kv, 64, 512, top_k, seed=34)
    # the oracle chain
    o_idx, o_sc = oracle.topk_inputs(ix)
    chain = li.AttnInputs("c", n_q, n_kv, 64, 512, top_k, att.qa_bits, att.kv_bits, o_idx.astype(np.int32),
                          o_sc.astype(np.float32), att.scale)
    # the GPU chain
    from tests.parity import to_device
    q, k, w, m = to_device(ix)
    g_idx, g_sc = lid.topk(q, k, w, m, top_k)
    qa, kv, _, _ = _dev(att)
    out, lse = lid.sparse_attn(qa, kv, g_idx, att.scale, sel_score=g_sc)
    torch.cuda.synchronize()
    assert np.array_equal(g_idx.cpu().numpy(), o_idx)
    assert np.isneginf(o_sc[0]).any()  # the first query sees fewer than top_k keys
    _check(chain, out, lse)
