"""GPU parity of la_chunk_bwd (gradients of the chunk forward with respect to
q, k, v and the per-channel gate) against the fp64 backward oracle on the same
seeded inputs: every mode, fp32 and bf16, several head dims, ragged lengths,
a full-size sample and the edge cases."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, oracle_mode, to_dev
from retention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MODES = [
    dict(phi="elu1", normalize=True, gate=None),
    dict(phi="elu1", normalize=False, gate=None),
    dict(phi="identity", normalize=False, gate=None),
    dict(phi="identity", normalize=False, gate="head"),
    dict(phi="elu1", normalize=True, gate="head"),
    dict(phi="elu1", normalize=False, gate="channel"),
    dict(phi="elu1", normalize=True, gate="channel"),
    dict(phi="identity", normalize=False, gate="channel"),
    dict(phi="identity", normalize=True, gate=None),
]
MID = lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"])


def _host(t):
    return None if t is None else t.float().numpy()


def _check(cfg, seed=0, heads=None, tol=None, simt=False):
    """GPU gradients against the oracle's; ``heads`` limits the oracle to the
    first few heads of every batch row (the GPU computes all of them)."""
    from retention_gb300 import la
    inp = W.chunk_inputs(cfg, seed)
    if cfg["phi"] == "identity" and cfg["normalize"]:
        # with the identity map the normaliser needs features that are already
        # positive: den_t = q_t . z_t then stays away from zero (signed inputs
        # let it cross zero, where the form has no precision left to compare)
        inp = dict(inp, q=inp["q"].abs(), k=inp["k"].abs())
    dout = W.bwd_inputs(cfg, seed)
    x = to_dev(inp)
    d = dout.cuda()
    nan = lambda t: torch.full_like(t, float("nan"))
    dq, dk, dv = nan(x["q"]), nan(x["k"]), nan(x["v"])
    dg = nan(x["q"]) if cfg["gate"] == "channel" else None
    n0 = la.kernel_launches()
    la.chunk_bwd(x["q"], x["k"], x["v"], d, x["gate"], phi=cfg["phi"], normalize=cfg["normalize"],
                 gate_kind=cfg["gate"], dq=dq, dk=dk, dv=dv, dgate=dg, simt=simt)
    torch.cuda.synchronize()
    launches = la.kernel_launches() - n0
    hs = slice(None) if heads is None else slice(0, heads)
    gate = inp["gate"]
    if gate is not None:
        gate = gate[hs] if cfg["gate"] == "head" else gate[:, hs]
    ref = oracle.backward(_host(inp["q"][:, hs]), _host(inp["k"][:, hs]), _host(inp["v"][:, hs]),
                          _host(dout[:, hs]), _host(gate), oracle_mode(cfg))
    tol = tol or TOL[cfg["dtype"]]
    # max|gpu - oracle| over the larger of max|oracle| and the largest gradient
    # of the call: a gradient that is zero by cancellation (one normalised
    # token, whose output is its value whatever q and k; a gate with no state
    # to decay) has no scale of its own, and the rounding of the terms that
    # cancel is set by the other gradients' scale
    scale = max(float(np.max(np.abs(r))) for r in ref if r is not None)
    errs = []
    for name, g, r in zip(("dq", "dk", "dv", "dg"), [dq, dk, dv, dg], ref):
        if r is None:
            continue
        gg = g[:, hs].float().cpu().numpy()
        assert np.all(np.isfinite(gg)), name
        errs.append((name, float(np.max(np.abs(gg - r))) / max(float(np.max(np.abs(r))), scale, 1e-300)))
    assert all(e <= tol for _, e in errs), errs
    return launches


@pytest.mark.parametrize("m", MODES, ids=MID)
@pytest.mark.parametrize("L", [1, 13, 77])
def test_fp32_modes_ragged(m, L):
    cfg = W.workload("tiny", B=2, H=3, L=L, dk=32, dv=16, gamma_step=1.0, **m)
    _check(cfg, seed=L)


@pytest.mark.parametrize("dk,dv", [(16, 128), (128, 16), (64, 64), (128, 128), (16, 16)])
def test_fp32_head_dims(dk, dv):
    cfg = W.workload("tiny", B=1, H=2, L=70, dk=dk, dv=dv, gate="channel", normalize=True)
    _check(cfg, seed=dk + dv)


@pytest.mark.parametrize("m", MODES, ids=MID)
@pytest.mark.parametrize("simt", [False, True], ids=["default", "simt"])
def test_bf16_modes(m, simt):
    """Every mode; except the per-channel gate with the normaliser the default
    route is the tensor-core one: three forwards, two of them anti-causal
    (scalar gate, identity feature map), with phi = elu + 1 a pass before them
    for phi(q), phi(k) and one after for phi'; with the normaliser and no
    gate the backward-prep forward and three more, with the head gate three
    preps, six forwards and a post; with the per-channel gate three
    forwards (two anti-causal, two with the gate on the value side), one pass
    after them and the gate gradient's scan (carries, dg)."""
    cfg = W.workload("la", B=2, H=3, L=333, **m)
    launches = _check(cfg, seed=3, simt=simt)
    tc = not simt and not (m["normalize"] and m["gate"] == "channel")
    # a forward is three launches when the short batch is split into segments
    if tc and m["gate"] == "channel":
        # three forwards (two anti-causal), the post pass, the dg carries and dg
        assert launches in (6, 12), launches
    elif tc and m["normalize"]:
        assert launches in ((10, 22) if m["gate"] == "head" else (4, 12)), launches
    elif tc:
        assert launches in ((5, 11) if m["phi"] == "elu1" else (3, 9)), launches
    else:
        assert launches == (4 if m["normalize"] else 3), launches


@pytest.mark.parametrize("m", [MODES[0], MODES[1], MODES[3], MODES[4], MODES[5], MODES[7], MODES[8]], ids=MID)
@pytest.mark.parametrize("B,H,L", [(1, 2, 1000), (2, 40, 200), (1, 1, 1), (1, 3, 65)])
def test_bf16_tensor_core_route_shapes(m, B, H, L):
    """Split and unsplit sequences, one token, a ragged chunk."""
    _check(W.workload("la", B=B, H=H, L=L, **m), seed=B + H + L)


@pytest.mark.parametrize("m", [MODES[0], MODES[8]], ids=MID)
def test_bf16_normalised_split_segments_of_several_chunks(m):
    """The normalised route on a short batch whose segments hold two chunks
    each (79 chunks over 40 segments): the carried sums of the bias instances
    run inside a segment and across the segment scan."""
    launches = _check(W.workload("la", B=1, H=2, L=5000, **m), seed=9)
    assert launches == 12, launches


def test_bf16_gated_long_sequence():
    cfg = W.workload("gla", B=1, H=2, L=4096)
    _check(cfg, seed=4)


def test_bf16_gated_more_chunks_than_scan_threads():
    """313 chunks: the gate gradient's carry scan gives each of its 256 threads
    a run of two chunks (and some none), with a ragged last chunk."""
    cfg = W.workload("gla", B=1, H=2, L=20000)
    _check(cfg, seed=6, heads=1)


@pytest.mark.parametrize("name", ["retention", "la"])
def test_full_size_sampled_heads(name):
    """The full workload shapes on the GPU, the oracle on two heads of every
    batch row."""
    cfg = W.workload(name)
    launches = _check(cfg, seed=0, heads=2)
    # retention: three tensor-core forwards (two anti-causal); la (normalised, one CTA per
    # sequence): the backward-prep forward (w, e), the biased dQ and dK forwards (phi' in
    # their store), dv
    assert launches == (4 if cfg["normalize"] else 3)


def test_without_the_gate_gradient():
    from retention_gb300 import la
    cfg = W.workload("gla", B=1, H=2, L=100)
    x = to_dev(W.chunk_inputs(cfg, 5))
    d = W.bwd_inputs(cfg, 5).cuda()
    dq, dk, dv, dg = la.chunk_bwd(x["q"], x["k"], x["v"], d, x["gate"], phi="elu1", gate_kind="channel",
                                  want_dgate=False)
    assert dg is None
    torch.cuda.synchronize()
    dq2, dk2, dv2, _ = la.chunk_bwd(x["q"], x["k"], x["v"], d, x["gate"], phi="elu1", gate_kind="channel")
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_empty_and_invalid():
    from retention_gb300 import la
    lib = la.load()
    s = la._stream(None)
    z = torch.zeros(1, 1, 4, 16, device="cuda")
    vp = lambda t: la._dev(t, "t")
    f32 = la.LA_DTYPE_F32
    # L = 0 and an empty batch are no-ops
    assert lib.la_chunk_bwd(None, None, None, None, None, None, None, None, None, 1, 1, 0, 16, 16, f32, s) == 0
    assert lib.la_chunk_bwd(None, None, None, None, None, None, None, None, None, 0, 1, 4, 16, 16, f32, s) == 0
    # a gate mode without the gate, a missing gradient buffer, an unsupported head dim
    assert lib.la_chunk_bwd(vp(z), vp(z), vp(z), None, vp(z), vp(z), vp(z), vp(z), None,
                            1, 1, 4, 16, 16, f32 | la.LA_GATE_HEAD, s) == -1
    assert lib.la_chunk_bwd(vp(z), vp(z), vp(z), None, vp(z), None, vp(z), vp(z), None,
                            1, 1, 4, 16, 16, f32, s) == -1
    assert lib.la_chunk_bwd(vp(z), vp(z), vp(z), None, vp(z), vp(z), vp(z), vp(z), None,
                            1, 1, 4, 48, 16, f32, s) == -2
