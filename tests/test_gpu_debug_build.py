"""The small parity cases on the bounds-checking build of the library.

The library built with LA_DEBUG checks every shared-memory range, TMA
coordinate, TMEM address (including that a warp touches only its own lane
quarter) and global index of the tensor-core forward and the decode step
against its extent before using it; a failed check skips the access and makes
la_device_status return LA_ERR_INTERNAL. Here that build runs the forward in
every mode (split and unsplit, ragged), the anti-causal form, the fused RetNet
epilogue, the forward from a state, the decode step and the backward's
instances, each matched against the oracle, and no check may fail. It stands in for a memory checker, which is
not available on these GPUs.
"""
import pytest
import torch

import oracle
from parity import TOL, rel_err, run_gpu, run_oracle, to_dev
from retention_gb300 import build as la_build, la, workloads as W
from test_gpu_chunk import FP32_MODES

pytestmark = pytest.mark.gpu

MODE_IDS = lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"])


@pytest.fixture(scope="module")
def checked():
    path = la_build.build(debug=True)
    with la.library(path) as lib:
        assert la.device_status() == 0
        yield lib


def _parity(out, st, out_ref, st_ref):
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)
    assert la.device_status() == 0  # no bounds check failed


@pytest.mark.parametrize("m", FP32_MODES, ids=MODE_IDS)
@pytest.mark.parametrize("B,H,L", [(1, 2, 1000), (2, 40, 200)], ids=["split", "unsplit"])
def test_forward_modes(checked, m, B, H, L):
    cfg = W.workload("la", B=B, H=H, L=L, **m)
    inp = W.chunk_inputs(cfg, seed=41)
    out, st = run_gpu(inp, cfg)
    _parity(out, st, *run_oracle(inp, cfg))


@pytest.mark.parametrize("B,H,L", [(1, 4, 1000), (2, 40, 333)], ids=["split", "unsplit"])
def test_anti_causal_form(checked, B, H, L):
    cfg = W.workload("retention", B=B, H=H, L=L)
    inp = W.chunk_inputs(cfg, seed=42)
    flip = {n: (t.flip(2) if (t is not None and t.dim() == 4) else t) for n, t in inp.items()}
    out_ref, st_ref = run_oracle(flip, cfg)
    out, st = run_gpu(inp, cfg, reverse=True)
    _parity(out, st, out_ref[:, :, ::-1], st_ref)


@pytest.mark.parametrize("B,H,L", [(1, 4, 1000), (2, 40, 333)], ids=["split", "unsplit"])
def test_from_a_state(checked, B, H, L):
    cfg = W.workload("retention", B=B, H=H, L=L)
    inp = W.chunk_inputs(cfg, seed=43)
    s0 = W.decode_state(dict(cfg, state_std=0.1), 43)
    out, st = run_gpu(inp, cfg, initial_state=s0)
    _parity(out, st, *run_oracle(inp, cfg, state_in=s0.numpy()))


@pytest.mark.parametrize("B,H,L", [(1, 4, 1000), (2, 40, 333)], ids=["split", "unsplit"])
def test_fused_epilogue(checked, B, H, L):
    cfg = W.workload("retnet", B=B, H=H, L=L)
    inp = W.chunk_inputs(cfg, seed=44)
    ep = W.epilogue_inputs(cfg, seed=44)
    o_ref, st_ref = run_oracle(inp, cfg)
    ref = oracle.group_norm_swish(o_ref, ep["og"].float().numpy(), ep["weight"].numpy(), ep["bias"].numpy(),
                                  eps=cfg["gn_eps"])
    x, e = to_dev(inp), to_dev(ep)
    out, st = la.chunk_fwd_gn_swish(x["q"], x["k"], x["v"], e["og"], x["gate"], gn_weight=e["weight"],
                                    gn_bias=e["bias"], gn_eps=cfg["gn_eps"], phi="identity", gate_kind="head")
    torch.cuda.synchronize()
    _parity(out.float().cpu().numpy(), st.cpu().numpy(), ref, st_ref)


@pytest.mark.parametrize("m", [dict(phi="elu1", normalize=True, gate=None),
                               dict(phi="identity", normalize=False, gate="head"),
                               dict(phi="elu1", normalize=False, gate="channel")], ids=MODE_IDS)
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32)])
def test_decode_step(checked, m, dk, dv):
    cfg = W.workload("decode", B=4, H=8, dk=dk, dv=dv, **m)
    st0 = W.decode_state(cfg, 45)
    tok = W.decode_tokens(cfg, 0, 45)
    ref_state = st0.double().numpy().copy()
    mode = (oracle.PHI_ELU1 if m["phi"] == "elu1" else 0) | (oracle.NORMALIZE if m["normalize"] else 0)
    mode |= oracle.GATE_HEAD if m["gate"] == "head" else oracle.GATE_CHANNEL if m["gate"] == "channel" else 0
    f = lambda t: None if t is None else t.float().numpy()
    ref = oracle.decode_step(f(tok["q"]), f(tok["k"]), f(tok["v"]), ref_state, f(tok["gate"]), mode)
    state = st0.cuda()
    d = to_dev(tok)
    out = la.decode_step(d["q"], d["k"], d["v"], state, d["gate"], phi=m["phi"], normalize=m["normalize"],
                         gate_kind=m["gate"])
    torch.cuda.synchronize()
    _parity(out.float().cpu().numpy(), state.cpu().numpy(), ref, ref_state)


@pytest.mark.parametrize("name,B,H,L", [("la", 2, 40, 333), ("la", 1, 2, 5000), ("gla", 1, 2, 1000),
                                        ("gla", 2, 40, 200), ("retention", 1, 4, 1000)],
                         ids=["normalised-unsplit", "normalised-split", "gated-split", "gated-unsplit",
                              "retention-split"])
def test_backward(checked, name, B, H, L):
    """The backward's forward instances: the backward-prep and bias instances
    (normalised), the anti-causal gated and value-side instances (gated), the
    anti-causal scalar-decay instance (retention)."""
    from test_gpu_bwd import _check
    _check(W.workload(name, B=B, H=H, L=L), seed=45)
    assert la.device_status() == 0  # no bounds check failed
