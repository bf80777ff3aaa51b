"""GPU parity of la_chunk_fwd_from_state: the chunk forward continuing from a
given state instead of zero (a prefill's final state, or any state), against
the fp64 oracle started from the same state; chaining a prefill into a
continuation equals one forward over the whole sequence."""
import ctypes

import numpy as np
import pytest
import torch

from parity import TOL, rel_err, run_gpu, run_oracle, to_dev
from retention_gb300 import la, workloads as W
from test_gpu_chunk import FP32_MODES

pytestmark = pytest.mark.gpu

MODE_IDS = lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"])


def _state(cfg, seed):
    return W.decode_state(dict(cfg, state_std=0.1), seed)


def _check(cfg, seed, simt=False, chunk=None):
    inp = W.chunk_inputs(cfg, seed)
    s0 = _state(cfg, seed + 100)
    out_ref, st_ref = run_oracle(inp, cfg, state_in=s0.numpy())
    out, st = run_gpu(inp, cfg, chunk=chunk, simt=simt, initial_state=s0)
    tol = TOL[cfg["dtype"]]
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= tol and e_st <= tol, (e_out, e_st)


@pytest.mark.parametrize("m", FP32_MODES, ids=MODE_IDS)
@pytest.mark.parametrize("B,H,L", [(1, 2, 1000), (2, 40, 200)], ids=["split", "unsplit"])
def test_bf16_tensor_cores_from_state(m, B, H, L):
    """Every mode through the tensor-core kernel, with the sequences cut into
    segments (the scan starts from the given state) and with one CTA per
    sequence (segment 0 starts from it)."""
    cfg = W.workload("la", B=B, H=H, L=L, **m)
    assert la.chunk_fwd_path(B, H, L, 128, 128, la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"]), 64) == 1
    _check(cfg, seed=11)


@pytest.mark.parametrize("m", FP32_MODES, ids=MODE_IDS)
@pytest.mark.parametrize("chunk", [7, 64])
def test_fp32_general_kernel_from_state(m, chunk):
    cfg = W.workload("tiny", B=2, H=3, L=77, dk=32, dv=16, gamma_step=1.0, **m)
    _check(cfg, seed=12, chunk=chunk)


@pytest.mark.parametrize("name,B,H,L1,L2", [("la", 2, 3, 200, 333), ("retention", 2, 16, 128, 100),
                                            ("gla", 1, 3, 1000, 777)])
def test_prefill_then_continue_equals_one_forward(name, B, H, L1, L2):
    """forward(first L1 tokens) -> final state -> forward_from_state(next L2
    tokens) gives the outputs and final state of one forward over L1 + L2."""
    cfg = W.workload(name, B=B, H=H, L=L1 + L2)
    inp = W.chunk_inputs(cfg, seed=13)
    out_ref, st_ref = run_oracle(inp, cfg)
    x = to_dev(inp)
    part = lambda t, a, b: None if t is None else (t if t.dim() == 1 else t[:, :, a:b].contiguous())
    kw = dict(phi=cfg["phi"], normalize=cfg["normalize"], gate_kind=cfg["gate"], chunk=cfg["chunk"])
    _, st1 = la.chunk_fwd(part(x["q"], 0, L1), part(x["k"], 0, L1), part(x["v"], 0, L1),
                          part(x["gate"], 0, L1), **kw)
    out2, st2 = la.chunk_fwd(part(x["q"], L1, L1 + L2), part(x["k"], L1, L1 + L2), part(x["v"], L1, L1 + L2),
                             part(x["gate"], L1, L1 + L2), initial_state=st1, **kw)
    torch.cuda.synchronize()
    tol = TOL[cfg["dtype"]]
    assert rel_err(out2.float().cpu().numpy(), out_ref[:, :, L1:]) <= tol
    assert rel_err(st2.cpu().numpy(), st_ref) <= tol


def test_empty_sequence_returns_the_initial_state():
    cfg = W.workload("la", B=2, H=3, L=0)
    s0 = _state(cfg, 7).cuda()
    st = torch.full_like(s0, float("nan"))
    q = torch.empty(2, 3, 0, 128, dtype=torch.bfloat16, device="cuda")
    la.chunk_fwd(q, q, q, None, phi="elu1", normalize=True, out=torch.empty_like(q), final_state=st,
                 initial_state=s0)
    torch.cuda.synchronize()
    assert torch.equal(st, s0)


def test_null_initial_state_is_la_chunk_fwd():
    cfg = W.workload("gla", B=1, H=3, L=500)
    x = to_dev(W.chunk_inputs(cfg, seed=14))
    B, H, L, d = x["q"].shape
    mode = la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"])
    outs, sts = [], []
    for fn in ("la_chunk_fwd", "la_chunk_fwd_from_state"):
        out = torch.empty_like(x["v"])
        st = torch.empty(B, H, d * d, device="cuda")
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())
        args = [ptr(x["q"]), ptr(x["k"]), ptr(x["v"]), ptr(x["gate"])]
        if fn == "la_chunk_fwd_from_state":
            args.append(ctypes.c_void_p(None))
        args += [ptr(out), ptr(st), B, H, L, d, d, mode, 64, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)]
        assert getattr(la.load(), fn)(*args) == 0
        torch.cuda.synchronize()
        outs.append(out)
        sts.append(st)
    assert torch.equal(outs[0], outs[1]) and torch.equal(sts[0], sts[1])


def test_misaligned_initial_state_is_rejected():
    cfg = W.workload("la", B=1, H=2, L=64)
    x = to_dev(W.chunk_inputs(cfg, seed=15))
    s0 = torch.zeros(1 * 2 * (128 * 128 + 128) + 4, device="cuda")
    with pytest.raises(la.LAError) as e:
        la.chunk_fwd(x["q"], x["k"], x["v"], None, phi="elu1", normalize=True,
                     initial_state=s0[1:1 + 2 * (128 * 128 + 128)].view(1, 2, -1))
    assert e.value.status == -3  # LA_ERR_MISALIGNED


@pytest.mark.parametrize("B,H,L", [(1, 8, 6100), (2, 40, 1300)], ids=["split", "unsplit"])
def test_retention_window_ends_from_state(B, H, L):
    """Retention from a given state with decays whose rescale windows close
    after 1 to 625 chunks (see test_gpu_chunk.WINDOW_GAMMAS), split and
    unsplit: the carried state enters each window's bookkeeping."""
    from test_gpu_chunk import window_inputs
    cfg = W.workload("retention", B=B, H=H, L=L)
    inp = window_inputs(cfg, seed=22)
    s0 = _state(cfg, 122)
    out_ref, st_ref = run_oracle(inp, cfg, state_in=s0.numpy())
    out, st = run_gpu(inp, cfg, initial_state=s0)
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)
