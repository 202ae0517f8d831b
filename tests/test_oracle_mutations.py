"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies attn_oracle.c, plants one plausible mistake by a textual
edit, compiles the mutant with gcc into a temporary directory, points the
oracle wrapper at it and runs every pin in test_oracle_pins.py.  At least one
pin must fail for every mutant; the committed oracle itself is never touched.
"""
import ctypes
import inspect
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "causal_excludes_diagonal": ("if (j > i) { s[j] = -INFINITY; continue; }",
                                 "if (j >= i) { s[j] = -INFINITY; continue; }"),
    "gqa_interleaved": ("const uint32_t kvh = h / heads_per_kv;",
                        "const uint32_t kvh = h % num_kv_heads;"),
    "decode_gqa_interleaved": ("const uint32_t kvh = h / repeat;",
                               "const uint32_t kvh = h % kv_heads;"),
    "prefill_scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "decode_scale_dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
    "window_start_off_by_one": ("total_seq - window : 0;", "total_seq - window + 1 : 0;"),
    "mask_added_not_replaced": ("if (t < ws) s[t] = -1.0e4;", "if (t < ws) s[t] += -1.0e4;"),
    "key_row_transposed": ("const float *kj = k + (size_t)j * kv_stride",
                           "const float *kj = k + (size_t)i * kv_stride"),
    "value_row_reversed": ("const float *vr = v + j * v_row_pitch;",
                           "const float *vr = v + (n - 1 - j) * v_row_pitch;"),
    "not_normalised": ("for (size_t j = 0; j < n; ++j) scores[j] /= l;", ""),
    "exp_base_two": ("exp(scores[j] - m)", "exp2(scores[j] - m)"),
    "append_wrong_row": ("+ position) * d + e;\n            k_cache[dst] = k_src[src];",
                         "+ position - (position > 0)) * d + e;\n            k_cache[dst] = k_src[src];"),
    "rope_sign_flipped": ("y[i] = x[i] * c - x[i + h] * sn;", "y[i] = x[i] * c + x[i + h] * sn;"),
    "rope_adjacent_pairs": ("y[i + h] = x[i] * sn + x[i + h] * c;",
                            "y[i + h] = x[i] * sn + x[i + 1 - (i + 1 == h)] * c;"),
    "rope_query_not_rotated": ("if (rope_cos) rope(tmp, rope_cos, rope_sin, d, qd + (size_t)h * d);",
                               "if (0) rope(tmp, rope_cos, rope_sin, d, qd + (size_t)h * d);"),
    "fused_value_not_appended": ("v_cache[dst] = v_new[(size_t)g * d + e];", "(void)dst;"),
    # Each mutant below stays inside the buffers it reads (the pins run it
    # in this process).
    "causal_mask_dropped": ("if (j > i) { s[j] = -INFINITY; continue; }", ""),
    "value_gqa_interleaved": ("softmax_weighted_sum(s, m, v + (size_t)kvh * d, kv_stride, d, out);",
                              "softmax_weighted_sum(s, m, v + (size_t)(h % num_kv_heads) * d, kv_stride, d, out);"),
    "query_head_is_kv_head": ("const float *qi = q + (size_t)i * q_stride + (size_t)h * d;",
                              "const float *qi = q + (size_t)i * q_stride + (size_t)kvh * d;"),
    "decode_newest_row_dropped": ("softmax_weighted_sum(s, total_seq, vb, d, d, out + (size_t)h * d);",
                                  "softmax_weighted_sum(s, total_seq - 1, vb, d, d, out + (size_t)h * d);"),
    "window_mask_minus_infinity": ("if (t < ws) s[t] = -1.0e4;", "if (t < ws) s[t] = -INFINITY;"),
    "cache_head_pitch_total_seq": ("const float *kb = k_cache + (size_t)kvh * max_seq * d;",
                                   "const float *kb = k_cache + (size_t)kvh * total_seq * d;"),
    "rope_cos_sin_swapped": ("const double c = (double)cosv[i], sn = (double)sinv[i];",
                             "const double c = (double)sinv[i], sn = (double)cosv[i];"),
    "append_value_from_key": ("if (v_cache) v_cache[dst] = v_src[src];",
                              "if (v_cache) v_cache[dst] = k_src[src];"),
    "fused_key_not_rotated": ("if (rope_cos) rope(tmp, rope_cos, rope_sin, d, tmp + d);",
                              "if (0) rope(tmp, rope_cos, rope_sin, d, tmp + d);"),
    "prefill_scale_squared": ("s[j] = scale * dot;", "s[j] = scale * scale * dot;"),
    "window_start_from_max_seq": ("total_seq - window : 0;", "max_seq - window : 0;"),
    "decode_query_is_kv_head": ("const double *qh = qd + (size_t)h * d;",
                                "const double *qh = qd + (size_t)kvh * d;"),
    "decode_value_from_key_cache": ("const float *vb = v_cache + (size_t)kvh * max_seq * d;",
                                    "const float *vb = k_cache + (size_t)kvh * max_seq * d;"),
    "window_masks_newest_rows": ("if (t < ws) s[t] = -1.0e4;",
                                 "if (t >= total_seq - ws) s[t] = -1.0e4;"),
}


def _pin_functions():
    return [f for n, f in inspect.getmembers(pins, inspect.isfunction)
            if n.startswith("test_")]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut_src = tmp_path / "attn_oracle_mut.c"
    mut_src.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    str(mut_src), "-o", str(so), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_LIB_PATH", str(so))
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    monkeypatch.setattr(oracle, "_lib", None)
    caught = []
    for f in _pin_functions():
        try:
            f()
        except (AssertionError, ValueError, FloatingPointError) as e:
            caught.append(f.__name__)
    monkeypatch.setattr(oracle, "_lib", None)
    assert caught, f"no pin caught the planted mistake {name}"
