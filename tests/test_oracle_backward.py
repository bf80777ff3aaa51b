"""Pins of the backward oracle (``oracle.backward``: gradients of the forward
recurrence with respect to q, k, v and the per-channel gate) against what the
mathematics fixes: central finite differences of the independent fp64 numpy
parallel form, autograd through a plain torch fp64 recurrence written here,
the closed form of the ungated identity case, and linearity in the output
gradient; plus planted mistakes in copies of its C source."""
import ctypes
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import _build, forms

MODES = {
    "la": oracle.PHI_ELU1 | oracle.NORMALIZE,
    "la-unnorm": oracle.PHI_ELU1,
    "identity": 0,
    "retention": oracle.GATE_HEAD,
    "retention-norm-elu": oracle.GATE_HEAD | oracle.NORMALIZE | oracle.PHI_ELU1,
    "gla": oracle.PHI_ELU1 | oracle.GATE_CHANNEL,
    "gla-norm": oracle.PHI_ELU1 | oracle.GATE_CHANNEL | oracle.NORMALIZE,
    "gla-identity": oracle.GATE_CHANNEL,
}


def _inputs(B, H, L, dk, dv, mode, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, L, dk)).astype(np.float32)
    k = rng.standard_normal((B, H, L, dk)).astype(np.float32)
    v = rng.standard_normal((B, H, L, dv)).astype(np.float32)
    do = rng.standard_normal((B, H, L, dv)).astype(np.float32)
    gate = None
    if mode & oracle.GATE_HEAD:
        gate = np.linspace(0.6, 0.95, H).astype(np.float32)
    elif mode & oracle.GATE_CHANNEL:
        gate = (2.0 * rng.standard_normal((B, H, L, dk))).astype(np.float32)
    return q, k, v, do, gate


def _loss(q, k, v, g, gamma, mode, do):
    """sum(dout * out) for one head, in fp64 through the parallel form."""
    L, dk = q.shape
    a = forms.step_gates(L, dk, gamma=gamma, g=g)
    out = forms.parallel(q, k, v, a, elu1=bool(mode & oracle.PHI_ELU1), normalize=bool(mode & oracle.NORMALIZE))
    return float(np.sum(out * do))


@pytest.mark.parametrize("name", list(MODES))
def test_matches_finite_differences(name):
    mode = MODES[name]
    q, k, v, do, gate = _inputs(1, 2, 6, 3, 4, mode, seed=len(name))
    if mode & oracle.NORMALIZE and not mode & oracle.PHI_ELU1:
        pytest.skip("identity features can zero the normaliser")
    dq, dk, dv, dg = oracle.backward(q, k, v, do, gate, mode)
    h = 1e-6
    for hd in range(2):
        base = [x[0, hd].astype(np.float64) for x in (q, k, v)]
        g = gate[0, hd].astype(np.float64) if mode & oracle.GATE_CHANNEL else None
        gamma = float(gate[hd]) if mode & oracle.GATE_HEAD else None
        D = do[0, hd].astype(np.float64)
        targets = [(0, dq), (1, dk), (2, dv)] + ([(3, dg)] if g is not None else [])
        for which, grad in targets:
            arr = g if which == 3 else base[which]
            for idx in np.ndindex(arr.shape):
                plus, minus = [x.copy() for x in base], [x.copy() for x in base]
                gp, gm = (g.copy(), g.copy()) if g is not None else (None, None)
                if which == 3:
                    gp[idx] += h
                    gm[idx] -= h
                else:
                    plus[which][idx] += h
                    minus[which][idx] -= h
                fd = (_loss(*plus, gp, gamma, mode, D) - _loss(*minus, gm, gamma, mode, D)) / (2 * h)
                assert abs(fd - grad[0, hd][idx]) <= 1e-6 * (1.0 + abs(fd)), (name, which, idx, fd, grad[0, hd][idx])


def _torch_recurrence(q, k, v, gate, mode):
    """The forward recurrence in plain torch fp64 ops, one token at a time."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    phi = (lambda x: torch.where(x > 0, x + 1.0, torch.exp(x))) if mode & oracle.PHI_ELU1 else (lambda x: x)
    S = torch.zeros(B, H, dk, dv, dtype=torch.float64)
    z = torch.zeros(B, H, dk, dtype=torch.float64)
    outs = []
    for t in range(L):
        qf, kf = phi(q[:, :, t]), phi(k[:, :, t])
        if mode & oracle.GATE_CHANNEL:
            a = torch.exp(torch.nn.functional.logsigmoid(gate[:, :, t]) / 16.0)
        elif mode & oracle.GATE_HEAD:
            a = gate.view(1, H, 1).expand(B, H, dk)
        else:
            a = torch.ones(B, H, dk, dtype=torch.float64)
        S = a.unsqueeze(-1) * S + kf.unsqueeze(-1) * v[:, :, t].unsqueeze(-2)
        o = torch.einsum("bhi,bhij->bhj", qf, S)
        if mode & oracle.NORMALIZE:
            z = a * z + kf
            o = o / (qf * z).sum(-1, keepdim=True)
        outs.append(o)
    return torch.stack(outs, dim=2)


@pytest.mark.parametrize("name", ["la", "retention", "gla", "gla-norm", "la-unnorm"])
def test_matches_torch_autograd(name):
    mode = MODES[name]
    q, k, v, do, gate = _inputs(2, 2, 20, 8, 6, mode, seed=7)
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    tg = None
    if gate is not None:
        tg = torch.tensor(gate, dtype=torch.float64, requires_grad=bool(mode & oracle.GATE_CHANNEL))
    out = _torch_recurrence(tq, tk, tv, tg, mode)
    (out * torch.tensor(do, dtype=torch.float64)).sum().backward()
    dq, dk, dv, dg = oracle.backward(q, k, v, do, gate, mode)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-10)
    if mode & oracle.GATE_CHANNEL:
        np.testing.assert_allclose(dg, tg.grad.numpy(), rtol=1e-9, atol=1e-10)


def test_ungated_identity_closed_form():
    """A = 1, identity features, no normaliser: out = tril(Q K^T) V, so
    dV = tril(Q K^T)^T dO, dQ = tril(dO V^T) K, dK = tril(dO V^T)^T Q."""
    q, k, v, do, _ = _inputs(1, 1, 9, 5, 4, 0, seed=3)
    dq, dk, dv, _ = oracle.backward(q, k, v, do, None, 0)
    Q, K, V, D = (x[0, 0].astype(np.float64) for x in (q, k, v, do))
    M = np.tril(np.ones((9, 9)))
    G = M * (D @ V.T)
    np.testing.assert_allclose(dv[0, 0], (M * (Q @ K.T)).T @ D, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq[0, 0], G @ K, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk[0, 0], G.T @ Q, rtol=0, atol=1e-12)


@pytest.mark.parametrize("name", ["la", "gla"])
def test_linear_in_the_output_gradient(name):
    mode = MODES[name]
    q, k, v, do1, gate = _inputs(1, 2, 11, 4, 3, mode, seed=5)
    do2 = np.random.default_rng(6).standard_normal(do1.shape)
    # multiples of 2^-10: do1 + 2 do2 is exact in float32
    do1, do2 = (np.round(x.astype(np.float64) * 1024) / 1024 for x in (do1, do2))
    do1, do2 = do1.astype(np.float32), do2.astype(np.float32)
    g1 = oracle.backward(q, k, v, do1, gate, mode)
    g2 = oracle.backward(q, k, v, do2, gate, mode)
    g12 = oracle.backward(q, k, v, (do1.astype(np.float64) + 2 * do2).astype(np.float32), gate, mode)
    for a, b, c in zip(g1, g2, g12):
        if a is not None:
            np.testing.assert_allclose(c, a + 2 * b, rtol=1e-12, atol=1e-12)


PINS = [lambda: test_matches_finite_differences("la"), lambda: test_matches_finite_differences("gla"),
        lambda: test_matches_finite_differences("retention"), lambda: test_matches_torch_autograd("gla-norm"),
        test_ungated_identity_closed_form]

MUTANTS = [
    ("reverse sweep decays with the token's own gate",
     "const double *an = t + 1 < L ? a + (size_t)(t + 1) * dk : NULL;",
     "const double *an = t + 1 < L ? a + (size_t)t * dk : NULL;"),
    ("feature-map derivative dropped",
     "if (elu1 && (double)qb[x] <= 0.0) dQ[x] *= exp((double)qb[x]);", "(void)0;"),
    ("key term of the gate gradient with the wrong sign",
     "c += qf[x] * dQ[x] - kf[x] * dK[x];", "c += qf[x] * dQ[x] + kf[x] * dK[x];"),
    ("value gradient contracted with the queries",
     "for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * kt[i];",
     "for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * qt[i];"),
    ("normaliser term left out of dQ",
     "dQ[(size_t)t * dk + i] = acc + z[i] * e[t];", "dQ[(size_t)t * dk + i] = acc;"),
    ("sigmoid(g) for sigmoid(-g)",
     "const double sm = gx >= 0.0 ? exp(-gx) / (1.0 + exp(-gx)) : 1.0 / (1.0 + exp(gx));",
     "const double sm = gx >= 0.0 ? 1.0 / (1.0 + exp(-gx)) : exp(gx) / (1.0 + exp(gx));"),
    ("denominator gradient with the wrong sign", "e[t] = -dot / den;", "e[t] = dot / den;"),
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
               "oracle_backward", "oracle_max_threads"):
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
