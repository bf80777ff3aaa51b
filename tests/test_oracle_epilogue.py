"""Pins of the RetNet output epilogue of the oracle (``oracle.group_norm_swish``:
GroupNorm with one group per head, then the swish output gate; learnllm m22,
"Retention") against what the mathematics and independent library routines
fix, and planted mistakes in copies of its C source that the pins must catch."""
import ctypes
import math
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import _build


def _rand(B, H, L, dv, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, H, L, dv)) * 3.0 + rng.standard_normal((B, H, L, 1))
    og = rng.standard_normal((B, H, L, dv)).astype(np.float32) * 2
    w = (1.0 + 0.5 * rng.standard_normal((H, dv))).astype(np.float32)
    b = (0.3 * rng.standard_normal((H, dv))).astype(np.float32)
    return x, og, w, b


def test_matches_torch_group_norm_times_silu():
    """torch's GroupNorm over [tokens, H*dv] with H groups, times torch's SiLU
    (= swish), both in fp64: an independent implementation of the same thing."""
    B, H, L, dv = 2, 3, 5, 8
    x, og, w, b = _rand(B, H, L, dv, seed=1)
    for eps in (1e-5, 0.3):
        got = oracle.group_norm_swish(x, og, w, b, eps=eps)
        xt = torch.from_numpy(x).permute(0, 2, 1, 3).reshape(B * L, H * dv)
        y = torch.nn.functional.group_norm(xt, H, torch.from_numpy(w.astype(np.float64)).reshape(-1),
                                           torch.from_numpy(b.astype(np.float64)).reshape(-1), eps)
        y = y.reshape(B, L, H, dv).permute(0, 2, 1, 3)
        ref = torch.nn.functional.silu(torch.from_numpy(og.astype(np.float64))) * y
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


def test_worked_row():
    """x = (1, 2, 3, 4): mean 5/2, biased variance 5/4, so with eps = 0 the
    normalised row is (-3, -1, 1, 3) / sqrt(5); a gate of 40 passes it times
    40 sigmoid(40)."""
    x = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 1, 4)
    got = oracle.group_norm_swish(x, np.full((1, 1, 1, 4), 40.0, np.float32), eps=0.0)
    gate = 40.0 / (1.0 + math.exp(-40.0))
    np.testing.assert_allclose(got.ravel(), np.array([-3, -1, 1, 3]) / math.sqrt(5) * gate, rtol=1e-15, atol=0)


def test_swish_values():
    """swish(0) = 0, swish(1) = 1 / (1 + 1/e), swish(-1) = -1 / (1 + e), and
    swish(u) - swish(-u) = u."""
    x = np.array([-1.0, 1.0]).reshape(1, 1, 1, 2)  # normalises to (-1, 1) with eps = 0
    for u, want in ((0.0, 0.0), (1.0, 1.0 / (1.0 + math.exp(-1.0))), (-1.0, -1.0 / (1.0 + math.e)),
                    (30.0, 30.0 / (1.0 + math.exp(-30.0))), (-30.0, -30.0 * math.exp(-30.0) / (1 + math.exp(-30.0)))):
        got = oracle.group_norm_swish(x, np.full((1, 1, 1, 2), u, np.float32), eps=0.0)
        np.testing.assert_allclose(got.ravel(), [-want, want], rtol=1e-14, atol=1e-300)
    u = np.linspace(-6, 6, 16).astype(np.float32).reshape(1, 1, 1, 16)
    ones = np.tile(np.array([-1.0, 1.0]), 8).reshape(1, 1, 1, 16)
    pos = oracle.group_norm_swish(ones, u, eps=0.0) * ones
    neg = oracle.group_norm_swish(ones, -u, eps=0.0) * ones
    np.testing.assert_allclose(pos - neg, u.astype(np.float64), rtol=0, atol=1e-14)


def test_rows_are_standardised():
    """Without the affine part and with a gate of 40 (swish(40) = 40 to
    rounding) every row comes out with mean 0 and variance var / (var + eps)."""
    x, _, _, _ = _rand(2, 2, 6, 16, seed=2)
    eps = 0.05
    out = oracle.group_norm_swish(x, np.full(x.shape, 40.0, np.float32), eps=eps) / 40.0
    var = x.var(axis=-1)
    np.testing.assert_allclose(out.mean(axis=-1), 0.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out.var(axis=-1), var / (var + eps), rtol=1e-12, atol=0)


def test_shift_and_scale():
    """With eps = 0 the norm forgets a shift and a positive scale of the row and
    flips sign with a negative one."""
    x, og, w, b = _rand(1, 2, 4, 8, seed=3)
    base = oracle.group_norm_swish(x, og, w, eps=0.0)
    np.testing.assert_allclose(oracle.group_norm_swish(2.5 * x - 7.0, og, w, eps=0.0), base, rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.group_norm_swish(-x, og, w, eps=0.0), -base, rtol=0, atol=1e-12)


def test_constant_row_gives_the_bias():
    """A row with no spread normalises to zero, leaving bias * swish(og)."""
    H, dv = 2, 4
    x = np.ones((1, H, 3, dv)) * 5.0
    og = np.full((1, H, 3, dv), 1.5, np.float32)
    b = np.arange(H * dv, dtype=np.float32).reshape(H, dv)
    got = oracle.group_norm_swish(x, og, np.full((H, dv), 3.0, np.float32), b, eps=1e-5)
    sw = 1.5 / (1.0 + math.exp(-1.5))
    np.testing.assert_allclose(got, np.broadcast_to(b.astype(np.float64)[None, :, None, :] * sw, got.shape), rtol=1e-14, atol=0)


def test_affine_belongs_to_the_head():
    """Rows of head h take weight[h] and bias[h], whatever their token or batch."""
    B, H, L, dv = 2, 3, 4, 8
    x, og, w, b = _rand(B, H, L, dv, seed=4)
    full = oracle.group_norm_swish(x, og, w, b, eps=1e-5)
    plain = oracle.group_norm_swish(x, np.full(x.shape, 40.0, np.float32), eps=1e-5) / 40.0
    sw = og.astype(np.float64) / (1.0 + np.exp(-og.astype(np.float64)))
    want = (plain * w[None, :, None, :] + b[None, :, None, :]) * sw
    np.testing.assert_allclose(full, want, rtol=0, atol=1e-12)


PINS = [test_matches_torch_group_norm_times_silu, test_worked_row, test_swish_values, test_rows_are_standardised,
        test_shift_and_scale, test_constant_row_gives_the_bias, test_affine_belongs_to_the_head]

MUTANTS = [
    ("unbiased variance", "        var /= dv;\n", "        var /= (dv - 1);\n"),
    ("eps outside the root", "const double rstd = 1.0 / sqrt(var + eps);",
     "const double rstd = 1.0 / (sqrt(var) + eps);"),
    ("mean not subtracted", "double y = (xr[i] - mean) * rstd;", "double y = xr[i] * rstd;"),
    ("gate is the sigmoid alone", "if (u >= 0.0) return u / (1.0 + exp(-u));",
     "if (u >= 0.0) return 1.0 / (1.0 + exp(-u));"),
    ("affine indexed by token", "const int h = (int)((r / L) % H);", "const int h = (int)((r % L) % H);"),
    ("bias inside the gate", "orow[i] = or_swish((double)gr[i]) * y;",
     "orow[i] = or_swish((double)gr[i]) * y + (bias ? (double)bias[(size_t)h * dv + i] : 0.0);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    src = open(_build.SRC).read()
    assert src.count(old) == 1, name
    c = tmp_path / "mut.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-std=c99", str(c), "-o", str(so), "-lm"],
                   check=True)
    good = oracle._load()
    lib = ctypes.CDLL(str(so))
    for fn in ("oracle_forward", "oracle_decode_step", "oracle_delta_forward", "oracle_group_norm_swish",
               "oracle_max_threads"):
        getattr(lib, fn).argtypes = getattr(good, fn).argtypes
        getattr(lib, fn).restype = getattr(good, fn).restype
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = 0
    for t in PINS:
        try:
            with np.errstate(all="ignore"):
                t()
        except AssertionError:
            failed += 1
    assert failed > 0, "no pin caught the mutant '%s'" % name
