"""The pins are strong enough: each plausible mistake, planted into a copy of
the C oracle's source and compiled on the CPU, makes at least one pin fail.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import _build

import test_oracle_pins as pins

SRC = _build.SRC

# (name, text in la_oracle.c, replacement)
MUTANTS = [
    ("state transposed (v k^T)",
     "Si[j] = a[i] * Si[j] + kf[i] * (double)vt[j];",
     "Si[j] = a[i] * Si[j] + kf[j % dk] * (double)vt[i % dv];"),
    ("read before the update",
     "for (int i = 0; i < dk; ++i) num += qf[i] * S[(size_t)i * dv + j];",
     "for (int i = 0; i < dk; ++i) num += qf[i] * (S[(size_t)i * dv + j] - kf[i] * (double)vt[j]);"),
    ("denominator dropped",
     "ot[j] = norm ? num / den : num;",
     "ot[j] = num;"),
    ("elu without the +1",
     "return x > 0.0 ? x + 1.0 : exp(x);",
     "return x > 0.0 ? x : exp(x);"),
    ("retention gate ignored",
     "a[i] = gamma;",
     "a[i] = 1.0;"),
    ("decay applied after the add",
     "Si[j] = a[i] * Si[j] + kf[i] * (double)vt[j];",
     "Si[j] = a[i] * (Si[j] + kf[i] * (double)vt[j]);"),
    ("logsigmoid sign flipped",
     "return x - log1p(exp(x));",
     "return x + log1p(exp(x));"),
    ("normaliser not decayed",
     "if (norm) z[i] = a[i] * z[i] + kf[i];",
     "if (norm) z[i] = z[i] + kf[i];"),
    ("query feature map skipped",
     "qf[i] = or_phi((double)qt[i], elu1);",
     "qf[i] = (double)qt[i];"),
    ("gate read from the wrong step",
     "a[i] = exp(or_log_sigmoid((double)g[(size_t)t * dk + i]) / 16.0);",
     "a[i] = exp(or_log_sigmoid((double)g[(size_t)(t > 0 ? t - 1 : 0) * dk + i]) / 16.0);"),
]

PIN_TESTS = [
    pins.test_worked_example_two_tokens,
    pins.test_worked_example_three_tokens,
    lambda: pins.test_phi_values_through_c(1.0, 2.0),
    pins.test_gamma_zero_sees_only_itself,
    pins.test_gamma_one_identity_is_masked_matmul,
    pins.test_retention_unrolled_state,
    pins.test_unit_gate_final_state_is_KtV,
    pins.test_channel_gate_reduces_to_linear_and_to_retention,
] + [
    (lambda m=m: pins.test_recurrent_equals_parallel_and_chunkwise(*m)) for m in pins.MODES
]


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new)
    c = tmp_path / "mut.c"
    c.write_text(mutated)
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-std=c99", str(c),
                    "-o", str(so), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    so = _compile(tmp_path, name, old, new)
    good = oracle._load()
    lib = ctypes.CDLL(so)
    for fn in ("oracle_forward", "oracle_decode_step", "oracle_max_threads"):
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
        getattr(lib, fn).restype = getattr(good, fn).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = 0
    for t in PIN_TESTS:
        try:
            with np.errstate(all="ignore"):
                t()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the mutant '%s'" % name


def test_unmutated_source_passes_every_pin():
    for t in PIN_TESTS:
        t()
