"""Mutation check of the oracle's pins.

Each case plants one plausible slip in a copy of oracle/lid_oracle.c, builds
it with gcc into a temporary directory, points the oracle module at it, and
requires that at least one pin of test_oracle_pins.py, test_oracle_e4m3.py or
test_oracle_attn.py fails. This shows the
pins can tell a wrong oracle from the right one. Nothing here runs on a GPU.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_attn as pins_attn
from tests import test_oracle_e4m3 as pins_e4m3
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lid_oracle.c")

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "relu_as_abs": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot > 0.0 ? dot : -dot;"),
    "relu_negated": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot < 0.0 ? dot : 0.0;"),
    "weight_wrong_head": ("I += (double)w[t * H + h] * relu;", "I += (double)w[t * H + (H - 1 - h)] * relu;"),
    "weight_dropped": ("I += (double)w[t * H + h] * relu;", "I += relu;"),
    "query_head_fixed": ("const double *qh = qd + (r * H + h) * D;", "const double *qh = qd + (r * H + 0) * D;"),
    "key_features_reversed": ("return decode(o->k[s * D + d], o->is_f16);",
                              "return decode(o->k[s * D + (D - 1 - d)], o->is_f16);"),
    "last_feature_dropped": ("for (int d = 0; d < D; ++d) dot += qh[d] * krow[d];",
                             "for (int d = 0; d < D - 1; ++d) dot += qh[d] * krow[d];"),
    "mask_dropped": ("out[r * n_kv + s] = I + m;", "out[r * n_kv + s] = I;"),
    "mask_subtracted": ("out[r * n_kv + s] = I + m;", "out[r * n_kv + s] = I - m;"),
    "mask_as_bf16": ("double m = mask ? f16_to_double(mask[", "double m = mask ? bf16_to_double(mask["),
    "ties_reversed": ("return (x->idx < y->idx) ? -1 : (x->idx > y->idx);",
                      "return (x->idx > y->idx) ? -1 : (x->idx < y->idx);"),
    "sort_ascending": ("if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;",
                       "if (x->score > y->score) return 1;\n    if (x->score < y->score) return -1;"),
    "padding_index_zero": ("out_idx[o + j] = -1;", "out_idx[o + j] = 0;"),
    "padding_score_zero": ("out_score[o + j] = -INFINITY;", "out_score[o + j] = 0.0;"),
    "f16_exponent_off": ("e - 25); /* (1 + m/1024)", "e - 24); /* (1 + m/1024)"),
    "f16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "bf16_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    # the quantised (E4M3) form
    "e4m3_exponent_off": ("v = ldexp((double)(m + 8), e - 10);", "v = ldexp((double)(m + 8), e - 9);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "e4m3_sign_dropped": ("int sign = (b >> 7) & 1;", "int sign = 0;"),
    "e4m3_q_scale_wrong_row": ("o->q_scale[t * H + i / D]", "o->q_scale[t * H + i % H]"),
    "e4m3_k_scale_dropped": ("return (double)o->k_scale[s] * e4m3_to_double(o->k8[s * D + d]);",
                             "return e4m3_to_double(o->k8[s * D + d]);"),
    "e4m3_key_features_reversed": ("e4m3_to_double(o->k8[s * D + d]);",
                                   "e4m3_to_double(o->k8[s * D + (D - 1 - d)]);"),
    # the consumer: sparse attention over the selected latent rows
    "attn_scale_dropped": ("e[j] = scale * sj;", "e[j] = sj;"),
    "attn_keys_not_gathered": ("const uint16_t *krow = kv + sel[j] * (int64_t)Dc;",
                               "const uint16_t *krow = kv + (int64_t)j * Dc;"),
    "attn_values_from_next_row": ("const uint16_t *vrow = kv + sel[j] * (int64_t)Dc;",
                                  "const uint16_t *vrow = kv + ((sel[j] + 1) % n_kv) * (int64_t)Dc;"),
    "attn_uniform_weights": ("const double pj = e[j] / z;", "const double pj = 1.0 / nj;"),
    "attn_normaliser_dropped": ("const double pj = e[j] / z;", "const double pj = e[j];"),
    "attn_minus_inf_kept": ("if (sel_score && sel_score[t * top_k + j] == -INFINITY) continue;", ""),
    "attn_lse_without_max": ("lse[r * Ha + h] = m + log(z);", "lse[r * Ha + h] = log(z);"),
    "attn_query_head_fixed": ("const uint16_t *qrow = qa + (t * Ha + h) * (int64_t)Dc;",
                              "const uint16_t *qrow = qa + (t * Ha + 0) * (int64_t)Dc;"),
}


def _pin_calls():
    calls = []
    for seed in range(6):
        for dtype in ("f16", "bf16"):
            for kind in ("int", "float"):
                calls.append(lambda s=seed, d=dtype, k=kind: pins.test_oracle_matches_exact_brute_force(s, d, k))
    for name in dir(pins):
        fn = getattr(pins, name)
        if name.startswith("test_") and callable(fn) and name != "test_oracle_matches_exact_brute_force":
            calls.append(fn)
    for seed in range(5):
        calls.append(lambda s=seed: pins_e4m3.test_e4m3_oracle_matches_exact_brute_force(s))
    for name in dir(pins_e4m3):
        fn = getattr(pins_e4m3, name)
        if name.startswith("test_") and callable(fn) and name != "test_e4m3_oracle_matches_exact_brute_force":
            calls.append(fn)
    for name in dir(pins_attn):
        fn = getattr(pins_attn, name)
        if name.startswith("test_") and callable(fn):
            calls.append(fn)
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    mut = tmp_path / "lid_oracle_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(so), str(mut), "-lm"])
    prev = oracle.use_library(str(so))
    caught = 0
    try:
        for call in _pin_calls():
            try:
                call()
            except (AssertionError, RuntimeError, ValueError, IndexError):
                caught += 1
                break
    finally:
        oracle.use_library(None)
        oracle._lib = prev
    assert caught, f"no pin fails when the oracle has mistake {name!r}"
