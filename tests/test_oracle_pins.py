"""Pins for the oracle: each test ties the fp64 recurrent definition (C) to
something other than itself -- the pages' worked example, an independent
formula (parallel masked matmul, brute-force double sum, chunkwise), a closed
form, or an invariant the mathematics fixes. CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")

ELU1, NORM, GHEAD, GCHAN = oracle.PHI_ELU1, oracle.NORMALIZE, oracle.GATE_HEAD, oracle.GATE_CHANNEL


def _seq(L, dk, dv, seed, scale=1.0, gate_scale=1.0):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((L, dk)) * scale).astype(np.float32)
    k = (rng.standard_normal((L, dk)) * scale).astype(np.float32)
    v = (rng.standard_normal((L, dv)) * scale).astype(np.float32)
    g = (rng.standard_normal((L, dk)) * gate_scale).astype(np.float32)
    return q, k, v, g


def _c_forward_seq(q, k, v, mode, gamma=None, g=None, state_in=None):
    """Run the C oracle on one (1,1,L,d) sequence."""
    L, dk = q.shape
    dv = v.shape[1]
    gate = None
    if mode & GHEAD:
        gate = np.array([gamma], dtype=np.float32)
    if mode & GCHAN:
        gate = g.reshape(1, 1, L, dk)
    out, st = oracle.forward(q.reshape(1, 1, L, dk), k.reshape(1, 1, L, dk),
                             v.reshape(1, 1, L, dv), gate, mode, state_in=state_in)
    S = st[0, 0, :dk * dv].reshape(dk, dv)
    z = st[0, 0, dk * dv:] if mode & NORM else None
    return out[0, 0], S, z


def _gates(mode, L, dk, gamma=None, g=None):
    if mode & GCHAN:
        return forms.step_gates(L, dk, g=g)
    if mode & GHEAD:
        # the gate is a float32 array at the interface
        return forms.step_gates(L, dk, gamma=float(np.float32(gamma)))
    return forms.step_gates(L, dk)


def _rel(a, b):
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b))) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------
# 1. The worked example (insideout lesson 16, Example 1.1 and "Your turn")
# --------------------------------------------------------------------------

def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_worked_example_two_tokens():
    gd = _golden()
    q = np.array(gd["queries"][:2], np.float32)
    k = np.array(gd["keys"][:2], np.float32)
    v = np.array(gd["values"][:2], np.float32)
    out, S, z = _c_forward_seq(q, k, v, NORM)
    e = gd["after_two_tokens"]
    np.testing.assert_array_equal(S, np.array(e["state_S"], float))
    np.testing.assert_array_equal(z, np.array(e["state_z"], float))
    np.testing.assert_allclose(out[1], e["out"], rtol=0, atol=1e-15)
    # the same read without the divide is q^T S
    out_u, _, _ = _c_forward_seq(q, k, v, 0)
    np.testing.assert_array_equal(out_u[1], np.array(e["unnormalised_qS"], float))


def test_worked_example_three_tokens():
    gd = _golden()
    q = np.array(gd["queries"], np.float32)
    k = np.array(gd["keys"], np.float32)
    v = np.array(gd["values"], np.float32)
    out, S, z = _c_forward_seq(q, k, v, NORM)
    e = gd["after_three_tokens"]
    np.testing.assert_array_equal(S, np.array(e["state_S"], float))
    np.testing.assert_array_equal(z, np.array(e["state_z"], float))
    np.testing.assert_allclose(out[2], e["out"], rtol=0, atol=1e-15)
    out_u, _, _ = _c_forward_seq(q, k, v, 0)
    np.testing.assert_array_equal(out_u[2], np.array(e["unnormalised_qS"], float))
    # the distractor the page names: dividing by the z from before the third key
    stale_z = np.array(gd["after_two_tokens"]["state_z"], float)
    distractor = out_u[2] / (q[2].astype(float) @ stale_z)
    np.testing.assert_allclose(distractor, e["distractor_stale_z"], rtol=1e-15)
    assert not np.allclose(out[2], distractor)


def test_worked_example_orientation():
    """k v^T, not v k^T: the transposed state reads (2.5, 2) in step 1."""
    gd = _golden()
    k = np.array(gd["keys"][:2], float)
    v = np.array(gd["values"][:2], float)
    q = np.array(gd["queries"][1], float)
    S_t = sum(np.outer(v[j], k[j]) for j in range(2))
    wrong = (q @ S_t) / (q @ k.sum(0))
    np.testing.assert_allclose(wrong, [2.5, 2.0])
    out, _, _ = _c_forward_seq(np.array(gd["queries"][:2], np.float32),
                               np.array(gd["keys"][:2], np.float32),
                               np.array(gd["values"][:2], np.float32), NORM)
    assert not np.allclose(out[1], wrong)


# --------------------------------------------------------------------------
# 2. Feature map and closed forms at L = 1
# --------------------------------------------------------------------------

@pytest.mark.parametrize("x,expected", [(0.0, 1.0), (1.0, 2.0), (2.5, 3.5),
                                        (-1.0, math.exp(-1.0)), (-30.0, math.exp(-30.0))])
def test_phi_values_through_c(x, expected):
    """One token, d=1, unnormalised: out = phi(q) phi(k) v; q = 0 -> phi = 1."""
    q = np.array([[0.0]], np.float32)
    k = np.array([[x]], np.float32)
    v = np.array([[1.0]], np.float32)
    out, S, _ = _c_forward_seq(q, k, v, ELU1)
    assert out[0, 0] == pytest.approx(expected, rel=1e-15)
    assert S[0, 0] == pytest.approx(expected, rel=1e-15)
    assert forms.phi(np.array([x]), True)[0] == pytest.approx(expected, rel=1e-15)


def test_normalised_single_token_returns_its_value():
    q, k, v, _ = _seq(1, 8, 5, 3)
    for mode in (NORM | ELU1, NORM | ELU1 | GHEAD):
        out, _, _ = _c_forward_seq(q, k, v, mode, gamma=0.7)
        np.testing.assert_allclose(out[0], v[0].astype(float), rtol=1e-14)


# --------------------------------------------------------------------------
# 3. Cross-form agreement (ragged L=13, dk != dv to expose transpositions)
# --------------------------------------------------------------------------

MODES = [
    ("linear, identity", 0, None),
    ("linear, elu+1, normalised", ELU1 | NORM, None),
    ("linear, elu+1", ELU1, None),
    ("retention gamma=0.9", GHEAD, 0.9),
    ("retention gamma=0.9, elu+1, normalised", GHEAD | ELU1 | NORM, 0.9),
    ("gated, elu+1", GCHAN | ELU1, None),
    ("gated, elu+1, normalised", GCHAN | ELU1 | NORM, None),
    ("gated, identity", GCHAN, None),
]


@pytest.mark.parametrize("name,mode,gamma", MODES, ids=[m[0] for m in MODES])
def test_recurrent_equals_parallel_and_chunkwise(name, mode, gamma):
    L, dk, dv = 13, 6, 5
    q, k, v, g = _seq(L, dk, dv, 11, gate_scale=3.0)
    elu1, norm = bool(mode & ELU1), bool(mode & NORM)
    a = _gates(mode, L, dk, gamma, g)
    out_c, S_c, z_c = _c_forward_seq(q, k, v, mode, gamma, g)
    out_np, S_np, z_np = forms.recurrent(q, k, v, a, elu1, norm)
    assert _rel(out_c, out_np) < 1e-13
    assert _rel(S_c, S_np) < 1e-13
    out_par = forms.parallel(q, k, v, a, elu1, norm)
    assert _rel(out_c, out_par) < 1e-12
    for C in (1, 4, 7, L):
        out_ch, R, zR = forms.chunkwise(q, k, v, a, C, elu1, norm)
        assert _rel(out_c, out_ch) < 1e-12, C
        assert _rel(S_c, R) < 1e-12, C
        if norm:
            assert _rel(z_c, zR) < 1e-12


@pytest.mark.parametrize("name,mode,gamma", MODES[:2] + MODES[3:4] + MODES[5:7],
                         ids=[m[0] for m in MODES[:2] + MODES[3:4] + MODES[5:7]])
def test_recurrent_equals_brute_force(name, mode, gamma):
    L, dk, dv = 9, 4, 3
    q, k, v, g = _seq(L, dk, dv, 5, gate_scale=2.0)
    a = _gates(mode, L, dk, gamma, g)
    out_c, _, _ = _c_forward_seq(q, k, v, mode, gamma, g)
    out_bf = forms.brute_force(q, k, v, a, bool(mode & ELU1), bool(mode & NORM))
    assert _rel(out_c, out_bf) < 1e-12


def test_chunk_size_invariance():
    """linear_sparse_attention.py check [b]: every C gives the same output."""
    L, dk, dv = 13, 6, 6
    q, k, v, g = _seq(L, dk, dv, 2)
    a = forms.step_gates(L, dk, g=g)
    outs = [forms.chunkwise(q, k, v, a, C, True, False)[0] for C in (1, 4, 7, L)]
    for o in outs[1:]:
        assert _rel(o, outs[0]) < 1e-12


# --------------------------------------------------------------------------
# 4. Special cases that reduce to a textbook expression
# --------------------------------------------------------------------------

def test_gamma_one_identity_is_masked_matmul():
    """learnllm m22 Exercise 2: gamma = 1 with identity phi is (QK^T * tril) V."""
    L, dk, dv = 17, 5, 7
    q, k, v, _ = _seq(L, dk, dv, 9)
    out, _, _ = _c_forward_seq(q, k, v, GHEAD, gamma=1.0)
    qd, kd, vd = q.astype(float), k.astype(float), v.astype(float)
    expect = (np.tril(qd @ kd.T)) @ vd
    assert _rel(out, expect) < 1e-13


def test_gamma_zero_sees_only_itself():
    """learnllm m22 "Try It" 2: gamma = 0 keeps only the diagonal (0^0 = 1)."""
    L, dk, dv = 11, 4, 3
    q, k, v, _ = _seq(L, dk, dv, 4)
    out, _, _ = _c_forward_seq(q, k, v, GHEAD, gamma=0.0)
    qd, kd, vd = q.astype(float), k.astype(float), v.astype(float)
    expect = np.sum(qd * kd, axis=1, keepdims=True) * vd
    assert _rel(out, expect) < 1e-14


def test_unit_gate_final_state_is_KtV():
    L, dk, dv = 40, 6, 9
    q, k, v, _ = _seq(L, dk, dv, 8)
    _, S, z = _c_forward_seq(q, k, v, ELU1 | NORM)
    kf = forms.phi(k, True)
    assert _rel(S, kf.T @ v.astype(float)) < 1e-13
    assert _rel(z, kf.sum(axis=0)) < 1e-13
    _, S0, _ = _c_forward_seq(q, k, v, 0)
    assert _rel(S0, k.astype(float).T @ v.astype(float)) < 1e-13


def test_retention_unrolled_state():
    """S_n = sum_m gamma^(n-m) k_m^T v_m (learnllm m22, "Retention")."""
    L, dk, dv = 30, 4, 6
    q, k, v, _ = _seq(L, dk, dv, 12)
    gamma = float(np.float32(0.93))
    _, S, _ = _c_forward_seq(q, k, v, GHEAD, gamma=gamma)
    w = gamma ** (L - 1 - np.arange(L))
    expect = (k.astype(float) * w[:, None]).T @ v.astype(float)
    assert _rel(S, expect) < 1e-13


def test_channel_gate_reduces_to_linear_and_to_retention():
    """The per-channel gate at alpha = 1 is linear attention; at alpha = gamma
    it is retention (learnllm m22, the gate table of the unified recurrence)."""
    L, dk, dv = 20, 5, 4
    q, k, v, _ = _seq(L, dk, dv, 21)
    big = np.full((L, dk), 80.0, np.float32)        # logsigmoid(80) ~ -1.8e-35
    out_g, S_g, _ = _c_forward_seq(q, k, v, GCHAN | ELU1 | NORM, g=big)
    out_l, S_l, _ = _c_forward_seq(q, k, v, ELU1 | NORM)
    assert _rel(out_g, out_l) < 1e-14 and _rel(S_g, S_l) < 1e-14
    gamma = 0.9
    g_eq = np.float32(math.log(gamma ** 16 / (1.0 - gamma ** 16)))   # logit(gamma^16)
    g = np.full((L, dk), g_eq, np.float32)
    gamma_eff = math.exp(-math.log1p(math.exp(-float(g_eq))) / 16.0)
    out_g, S_g, _ = _c_forward_seq(q, k, v, GCHAN, g=g)
    out_r, S_r, _ = _c_forward_seq(q, k, v, GHEAD, gamma=np.float32(gamma_eff))
    assert abs(gamma_eff - gamma) < 1e-7
    assert _rel(out_g, out_r) < 1e-6 and _rel(S_g, S_r) < 1e-6


def test_multiscale_heads_use_their_own_gamma():
    L, dk, dv, H = 10, 4, 4, 4
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, H, L, dk)).astype(np.float32)
    k = rng.standard_normal((1, H, L, dk)).astype(np.float32)
    v = rng.standard_normal((1, H, L, dv)).astype(np.float32)
    gam = np.array([1 - 2.0 ** (-5 - h) for h in range(H)], np.float32)
    out, _ = oracle.forward(q, k, v, gam, GHEAD)
    for h in range(H):
        o1, _, _ = _c_forward_seq(q[0, h], k[0, h], v[0, h], GHEAD, gamma=gam[h])
        np.testing.assert_array_equal(out[0, h], o1)


def test_multiscale_decays_printed_values():
    """learnllm m22 prints per-head gamma [0.9688, 0.9844, 0.9922, 0.9961]."""
    from retention_gb300.workloads import retention_gammas
    g = retention_gammas(4, step=1.0).numpy()
    np.testing.assert_allclose(np.round(g, 4), [0.9688, 0.9844, 0.9922, 0.9961])


# --------------------------------------------------------------------------
# 5. Invariants
# --------------------------------------------------------------------------

def test_normalised_outputs_are_convex_combinations():
    L, dk, dv = 50, 8, 6
    q, k, v, _ = _seq(L, dk, dv, 31, scale=2.0)
    out, _, _ = _c_forward_seq(q, k, v, ELU1 | NORM)
    vd = v.astype(float)
    for t in range(L):
        lo = vd[:t + 1].min(axis=0) - 1e-12
        hi = vd[:t + 1].max(axis=0) + 1e-12
        assert np.all(out[t] >= lo) and np.all(out[t] <= hi)


def test_state_size_independent_of_length():
    """linear_sparse_attention.py check [c]."""
    dk, dv = 6, 6
    sizes = set()
    for L in (1, 5, 50, 300):
        q, k, v, _ = _seq(L, dk, dv, L)
        _, st = oracle.forward(q[None, None], k[None, None], v[None, None], None, ELU1 | NORM)
        sizes.add(st.shape)
    assert sizes == {(1, 1, dk * dv + dk)}


@pytest.mark.parametrize("mode,gamma", [(ELU1 | NORM, None), (GHEAD, 0.95), (GCHAN | ELU1, None)])
def test_prefill_then_decode_equals_longer_forward(mode, gamma):
    """learnllm m22 cell 4: the incremental state object equals the full
    recompute. Forward over L tokens, then n decode steps, matches a forward
    over L+n tokens, outputs and state."""
    B, H, L, n, dk, dv = 2, 3, 12, 5, 6, 7
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, H, L + n, dk)).astype(np.float32)
    k = rng.standard_normal((B, H, L + n, dk)).astype(np.float32)
    v = rng.standard_normal((B, H, L + n, dv)).astype(np.float32)
    g = rng.standard_normal((B, H, L + n, dk)).astype(np.float32)
    gate_full = None
    if mode & GHEAD:
        gate_full = np.full(H, gamma, np.float32)
    if mode & GCHAN:
        gate_full = g
    out_full, st_full = oracle.forward(q, k, v, gate_full, mode)
    gate_pre = gate_full[:, :, :L] if mode & GCHAN else gate_full
    out_pre, st = oracle.forward(q[:, :, :L], k[:, :, :L], v[:, :, :L], gate_pre, mode)
    assert _rel(out_pre, out_full[:, :, :L]) < 1e-15
    for s in range(n):
        t = L + s
        gs = g[:, :, t] if mode & GCHAN else gate_full
        o = oracle.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], st, gs, mode)
        assert _rel(o, out_full[:, :, t]) < 1e-13
    assert _rel(st, st_full) < 1e-13


def test_forward_from_state_continues_the_sequence():
    B, H, L1, L2, dk, dv = 1, 2, 9, 14, 5, 4
    rng = np.random.default_rng(17)
    q = rng.standard_normal((B, H, L1 + L2, dk)).astype(np.float32)
    k = rng.standard_normal((B, H, L1 + L2, dk)).astype(np.float32)
    v = rng.standard_normal((B, H, L1 + L2, dv)).astype(np.float32)
    g = rng.standard_normal((B, H, L1 + L2, dk)).astype(np.float32)
    mode = GCHAN | ELU1 | NORM
    out_full, st_full = oracle.forward(q, k, v, g, mode)
    _, st1 = oracle.forward(q[:, :, :L1], k[:, :, :L1], v[:, :, :L1], g[:, :, :L1], mode)
    out2, st2 = oracle.forward(q[:, :, L1:], k[:, :, L1:], v[:, :, L1:], g[:, :, L1:], mode,
                               state_in=st1)
    assert _rel(out2, out_full[:, :, L1:]) < 1e-13
    assert _rel(st2, st_full) < 1e-13


def test_oracle_rejects_bad_arguments():
    q = np.zeros((1, 1, 4, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.forward(q, q, q, None, GHEAD)            # gate mode without a gate
    with pytest.raises(ValueError):
        oracle.forward(q, q, q, np.ones(1, np.float32), GHEAD | GCHAN)
