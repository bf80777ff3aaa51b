"""Pins of the delta-rule oracle (``oracle.delta_forward``: S <- S (I - beta k
k^T) + beta v k^T, out_t = S q_t; linear_sparse_attention.py,
"delta_rule_recurrent") against what the page and the mathematics fix, and
planted mistakes in copies of its C source that the pins must catch."""
import ctypes
import subprocess

import numpy as np
import pytest

import oracle
from oracle import _build, forms


def _rand(B, H, L, dk, dv, seed, unit=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, L, dk))
    k = rng.standard_normal((B, H, L, dk))
    if unit:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, L))))
    return [a.astype(np.float32) for a in (q, k, v, beta)]


def test_matches_the_matrix_form():
    """The C loops against the page's matrix form S @ (I - b k k^T) + b outer(v, k)."""
    q, k, v, beta = _rand(2, 3, 13, 6, 5, seed=1)
    out, st = oracle.delta_forward(q, k, v, beta)
    for b in range(2):
        for h in range(3):
            states, o = forms.delta_recurrent(k[b, h], v[b, h], beta[b, h], Q=q[b, h])
            np.testing.assert_allclose(st[b, h], states[-1].ravel(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(out[b, h], o, rtol=0, atol=1e-12)


def test_single_token():
    """From zero, one token leaves S = beta v k^T and reads out beta v (k . q)."""
    q, k, v, beta = _rand(1, 1, 1, 4, 3, seed=2)
    out, st = oracle.delta_forward(q, k, v, beta)
    b, kk, vv, qq = float(beta[0, 0, 0]), k[0, 0, 0].astype(np.float64), v[0, 0, 0].astype(np.float64), q[0, 0, 0]
    np.testing.assert_allclose(st[0, 0].reshape(3, 4), b * np.outer(vv, kk), rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[0, 0, 0], b * vv * float(kk @ qq), rtol=0, atol=1e-12)


def test_orthonormal_keys_with_unit_beta_are_additive():
    """The page's check [e]: with orthonormal keys and beta = 1 nothing is erased,
    so S_t = sum_{s<=t} v_s k_s^T."""
    rng = np.random.default_rng(3)
    d = 8
    Ko = np.linalg.qr(rng.standard_normal((d, d)))[0].T.astype(np.float32)
    V = rng.standard_normal((d, 5)).astype(np.float32)
    Q = rng.standard_normal((d, d)).astype(np.float32)
    out, st = oracle.delta_forward(Q[None, None], Ko[None, None], V[None, None], np.ones((1, 1, d), np.float32))
    Kd, Vd = Ko.astype(np.float64), V.astype(np.float64)
    np.testing.assert_allclose(st[0, 0].reshape(5, d), Vd.T @ Kd, rtol=0, atol=1e-6)
    for t in range(d):
        np.testing.assert_allclose(out[0, 0, t], (Vd[:t + 1].T @ Kd[:t + 1]) @ Q[t].astype(np.float64),
                                   rtol=0, atol=1e-5)


def test_overlapping_keys_are_not_additive():
    """The page's check [e], first half: with keys that overlap, the erase term
    changes the state."""
    q, k, v, _ = _rand(1, 1, 12, 6, 6, seed=4)
    beta = np.ones((1, 1, 12), np.float32)
    _, st = oracle.delta_forward(q, k, v, beta)
    additive = v[0, 0].astype(np.float64).T @ k[0, 0].astype(np.float64)
    assert np.linalg.norm(st[0, 0].reshape(6, 6) - additive) > 1e-3


def test_page_check_d_no_erase_and_unit_beta_is_additive():
    """The page's check [d] on the matrix form: without the erase term and with
    beta = 1 the rule is plain S += v k^T."""
    _, k, v, _ = _rand(1, 1, 9, 5, 5, seed=5)
    states, _ = forms.delta_recurrent(k[0, 0], v[0, 0], np.ones(9), use_delta=False)
    np.testing.assert_allclose(states[-1], v[0, 0].astype(np.float64).T @ k[0, 0].astype(np.float64),
                               rtol=0, atol=1e-6)


def test_same_key_twice_overwrites():
    """A unit key written twice with beta = 1 keeps only the second value."""
    rng = np.random.default_rng(6)
    kk = rng.standard_normal(4)
    kk /= np.linalg.norm(kk)
    k = np.stack([kk, kk]).astype(np.float32)[None, None]
    v = rng.standard_normal((1, 1, 2, 3)).astype(np.float32)
    q = rng.standard_normal((1, 1, 2, 4)).astype(np.float32)
    out, st = oracle.delta_forward(q, k, v, np.ones((1, 1, 2), np.float32))
    k64 = k[0, 0, 0].astype(np.float64)
    np.testing.assert_allclose(st[0, 0].reshape(3, 4), np.outer(v[0, 0, 1], k64), rtol=0, atol=1e-6)
    np.testing.assert_allclose(out[0, 0, 1], v[0, 0, 1] * float(k64 @ q[0, 0, 1]), rtol=0, atol=1e-6)


def test_reading_with_the_key_returns_the_value_just_written():
    """With unit keys and beta = 1, S_t k_t = v_t exactly (erase, then write):
    queries equal to the keys read back every value."""
    _, k, v, _ = _rand(2, 2, 10, 8, 6, seed=7)
    out, _ = oracle.delta_forward(k, k, v, np.ones((2, 2, 10), np.float32))
    np.testing.assert_allclose(out, v.astype(np.float64), rtol=0, atol=1e-6)


def test_zero_beta_keeps_the_state():
    q, k, v, _ = _rand(1, 2, 5, 4, 3, seed=8)
    S0 = np.random.default_rng(9).standard_normal((1, 2, 12))
    out, st = oracle.delta_forward(q, k, v, np.zeros((1, 2, 5), np.float32), state_in=S0)
    np.testing.assert_allclose(st, S0, rtol=0, atol=0)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], q[0, h].astype(np.float64) @ S0[0, h].reshape(3, 4).T,
                                   rtol=0, atol=1e-12)


def test_continuing_from_a_state_equals_one_run():
    q, k, v, beta = _rand(2, 2, 20, 6, 4, seed=10)
    out, st = oracle.delta_forward(q, k, v, beta)
    _, st1 = oracle.delta_forward(q[:, :, :7], k[:, :, :7], v[:, :, :7], beta[:, :, :7])
    out2, st2 = oracle.delta_forward(q[:, :, 7:], k[:, :, 7:], v[:, :, 7:], beta[:, :, 7:], state_in=st1)
    np.testing.assert_allclose(out2, out[:, :, 7:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(st2, st, rtol=0, atol=1e-12)


@pytest.mark.parametrize("C", [1, 4, 7, 16, 64])
def test_chunkwise_form_equals_the_recurrence(C):
    """The chunked (triangular-solve) form restated in numpy against the page's
    recurrence, on a ragged length, from a state."""
    q, k, v, beta = _rand(1, 2, 37, 8, 6, seed=11)
    S0 = np.random.default_rng(12).standard_normal((6, 8))
    for h in range(2):
        states, o = forms.delta_recurrent(k[0, h], v[0, h], beta[0, h], Q=q[0, h], S0=S0)
        out, S = forms.delta_chunkwise(k[0, h], v[0, h], beta[0, h], q[0, h], C, S0=S0)
        np.testing.assert_allclose(out, o, rtol=0, atol=1e-11)
        np.testing.assert_allclose(S, states[-1], rtol=0, atol=1e-11)


PINS = [test_matches_the_matrix_form, test_single_token, test_orthonormal_keys_with_unit_beta_are_additive,
        test_overlapping_keys_are_not_additive, test_same_key_twice_overwrites,
        test_reading_with_the_key_returns_the_value_just_written, test_zero_beta_keeps_the_state,
        test_continuing_from_a_state_equals_one_run]

MUTANTS = [
    ("erase added instead of subtracted",
     "for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] -= b * Sk[i] * kt[j];",
     "for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += b * Sk[i] * kt[j];"),
    ("erase skipped",
     "for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] -= b * Sk[i] * kt[j];",
     "for (int j = 0; j < dk; ++j) (void)Sk[i];"),
    ("beta missing on the write",
     "for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += b * vi * kt[j];",
     "for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += vi * kt[j];"),
    ("output read with the key",
     "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];",
     "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kt[j];"),
    ("erase projects on the query",
     "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kt[j];\n                Sk[i] = acc;",
     "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];\n                Sk[i] = acc;"),
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
    for fn in ("oracle_forward", "oracle_decode_step", "oracle_delta_forward", "oracle_max_threads"):
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
