"""Host-side arithmetic of bench.py (no GPU): the algorithmic work per call
that the roofline fractions divide by, and the kernel-code hash that decides
whether a recorded ncu traffic figure still applies."""

import numpy as np

import bench
import lid_inputs as li


def test_algorithmic_work_dense_and_ranges_agree_on_keys_and_flops():
    # multiseq at reduced size: four disjoint ranges, every key visible to one row
    inp = li.float_inputs("m", 4, 8192, 64, 128, 512, seed=1, mask=li.range_mask(4, 8192, 2048))
    lo, hi = li.block_ranges(4, 2048)
    b_dense, f_dense, v_dense = bench.algorithmic_work(inp)
    b_rng, f_rng, v_rng = bench.algorithmic_work(inp, (lo, hi))
    assert v_dense == v_rng == 8192
    assert f_dense == f_rng == 2.0 * 64 * 128 * 8192
    # the ranges form reads no mask: the dense form's bytes less the mask, plus 8 bytes a row
    assert b_dense - b_rng == inp.mask.nbytes - 8 * inp.n_q
    # causal ranges: visible pairs and touched keys as the dense causal mask counts them
    inp = li.float_inputs("c", 5, 300, 8, 64, 16, seed=2, mask=li.causal_mask(5, 300, 200))
    lo, hi = li.causal_ranges(5, 200)
    _, f1, v1 = bench.algorithmic_work(inp)
    _, f2, v2 = bench.algorithmic_work(inp, (lo, hi))
    assert v1 == v2 == sum(201 + t for t in range(5)) and f1 == f2


def test_algorithmic_work_counts_each_visible_key_row_once():
    inp = li.float_inputs("o", 3, 1000, 8, 64, 16, seed=3, mask=None)
    lo = np.array([0, 100, 900], np.int32)
    hi = np.array([200, 300, 2000], np.int32)  # overlapping, and past the end
    nbytes, _, visible = bench.algorithmic_work(inp, (lo, hi))
    assert visible == 200 + 200 + 100
    k_rows = 300 + 100  # [0, 300) and [900, 1000)
    assert nbytes == k_rows * 64 * 2 + 8 * 3 + inp.q_bits.nbytes + inp.w.nbytes + 3 * 16 * 8


def test_source_hash_ignores_comments_and_layout(tmp_path, monkeypatch):
    csrc = tmp_path / "sparse_attention_lightning_lid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cuh").write_text("int f() { return 1; } // one\n")
    (csrc / "b.cuh").write_text("int g() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "SOURCE_GROUPS", {"indexer": ("a.cuh",), "attention": ("b.cuh",)})
    h1 = bench.source_hash()
    a1 = bench.source_hash("attention")
    (csrc / "a.cuh").write_text("/* a comment */\nint f()  {\n  return 1;\n}\n")
    assert bench.source_hash() == h1
    (csrc / "a.cuh").write_text("int f() { return 2; }\n")
    assert bench.source_hash() != h1
    assert bench.source_hash("attention") == a1  # another family's change leaves it alone


def test_algorithmic_work_of_e4m3_operands_counts_codes_and_scales():
    inp = li.e4m3_inputs("e", 2, 1000, 8, 128, 16, seed=2, mask=None)
    nbytes, flops, visible = bench.algorithmic_work(inp)
    assert visible == 2000 and flops == 2.0 * 8 * 128 * 2000
    # a key row is 128 one-byte codes and a 4-byte scale; q carries one scale per (t, h)
    assert nbytes == 1000 * (128 + 4) + 2 * 8 * 128 + 2 * 8 * 4 + inp.w.nbytes + 2 * 16 * 8
    lo, hi = np.array([0, 500], np.int32), np.array([300, 1000], np.int32)
    nb_r, _, vis_r = bench.algorithmic_work(inp, (lo, hi))
    assert vis_r == 800 and nb_r == 800 * 132 + 8 * 2 + 2 * 8 * 132 + inp.w.nbytes + 2 * 16 * 8
