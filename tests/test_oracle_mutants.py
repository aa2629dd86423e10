"""The oracle's pins must have teeth: plant plausible mistakes in a copy of the
oracle (dropped terms, wrong signs, off-by-one masks, wrong GQA mapping,
transposed or swapped operands) and check that the pins reject every one.

The mistakes are planted only in temporary copies compiled here on the CPU;
the oracle source itself is never modified.
"""
import math
import os

import numpy as np
import pytest

import oracle
from test_oracle_pins import GOLDEN_CASES, LIB_CASES, torch_reference

MUTANTS = [
    ("dq_drops_scale", "dqi[d] += scale * ds * kj[d];", "dqi[d] += ds * kj[d];"),
    ("ds_sign_flipped_dq", "const double ds = pij * (dot(doi, vj, D) - Di);",
     "const double ds = pij * (Di - dot(doi, vj, D));"),
    ("ds_sign_flipped_dk", "(dot(doi, vj, D) - Dv[", "(-dot(doi, vj, D) + Dv["),
    ("window_off_by_one", "i - j >= window) return 0;", "i - j > window) return 0;"),
    ("causal_masks_diagonal", "if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    ("gqa_interleaved", "g = h / reps;", "g = h % Hkv;"),
    ("gqa_interleaved_dkv", "for (int h = g * reps; h < (g + 1) * reps; ++h)",
     "for (int h = g; h < Hq; h += Hkv)"),
    ("dk_wrong_operand", "dkj[d] += scale * ds * qi[d];", "dkj[d] += scale * ds * doi[d];"),
    ("dv_uses_ds", "dvj[d] += pij * doi[d];", "dvj[d] += ds * doi[d];"),
    ("lse_drops_max", "const double lse = m + log(sum);", "const double lse = log(sum);"),
    ("dvec_wrong_operand", "const double Di = dot(dout + row * D, orow, D);",
     "const double Di = dot(dout + row * D, q + row * D, D);"),
    ("scores_drop_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("bwd_scores_drop_scale", "exp(scale * dot(qi, kj, D) - Li)", "exp(dot(qi, kj, D) - Li)"),
    ("o_reads_keys", "o_row[d] += s[j] * vj[d];", "o_row[d] += s[j] * kg[(int64_t)j * D + d];"),
    ("dp_reads_keys", "dot(doi, vj, D)", "dot(doi, kj, D)"),
]


def _close(a, b, tol):
    a, b = np.asarray(a), np.asarray(b)
    if a.shape != b.shape:
        return False
    same_inf = np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    return same_inf and not np.isnan(a[fin]).any() and np.allclose(a[fin], b[fin], atol=tol, rtol=0)


def pins_pass(lib) -> bool:
    """The value pins of test_oracle_pins, run against another oracle build."""
    for c in GOLDEN_CASES:
        B, Hq, Hkv, Tq, Tkv, D = c["dims"]
        args = (c["q"].reshape(B, Hq, Tq, D), c["k"].reshape(B, Hkv, Tkv, D),
                c["v"].reshape(B, Hkv, Tkv, D))
        do = c["do"].reshape(B, Hq, Tq, D)
        o, lse = oracle.attn_fwd(*args, c["scale"], c["causal"], c["window"], lib=lib)
        g = oracle.attn_bwd(*args, do, c["scale"], c["causal"], c["window"], lib=lib)
        for got, want in ((o, c["o"]), (lse, c["lse"]), (g["dq"], c["dq"]),
                          (g["dk"], c["dk"]), (g["dv"], c["dv"])):
            if not _close(got.ravel(), want, 1e-12):
                return False
    for (B, Hq, Hkv, Tq, Tkv, D, causal, window) in LIB_CASES:
        rng = np.random.default_rng(B * 1000 + Tq * 10 + Tkv)
        q = rng.standard_normal((B, Hq, Tq, D))
        k = rng.standard_normal((B, Hkv, Tkv, D))
        v = rng.standard_normal((B, Hkv, Tkv, D))
        do = rng.standard_normal((B, Hq, Tq, D))
        s = 1 / math.sqrt(D)
        o_t, lse_t, dq_t, dk_t, dv_t = torch_reference(q, k, v, do, s, causal, window)
        o, lse = oracle.attn_fwd(q, k, v, s, causal, window, lib=lib)
        g = oracle.attn_bwd(q, k, v, do, s, causal, window, lib=lib)
        for got, want in ((o, o_t), (lse, lse_t), (g["dq"], np.nan_to_num(dq_t)),
                          (g["dk"], dk_t), (g["dv"], dv_t)):
            if not _close(got, want, 1e-10):
                return False
    return True


def test_unmodified_copy_passes(tmp_path):
    src = open(oracle.SOURCE).read()
    path = tmp_path / "same.c"
    path.write_text(src)
    lib = oracle.load_library(oracle.compile_source(str(path), str(tmp_path / "same.so")))
    assert pins_pass(lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load_library(oracle.compile_source(str(path), str(tmp_path / f"{name}.so")))
    assert not pins_pass(lib), f"pins did not catch planted mistake {name}"
