"""la_chunk_fwd_noalloc against la_chunk_fwd, through the C ABI.

Some callers cannot let a library allocate device memory while they run: a
server that plans all of its device memory up front, or code running while
another allocator owns the device's memory pool. la_chunk_fwd_noalloc serves
them. Where la_chunk_fwd takes stream-ordered scratch (the tensor-core path
cutting a short batch into sequence segments), it uses a fixed device array
inside the library instead. These tests check that it returns what
la_chunk_fwd returns, on two calls in a row: the second call reuses the array
exactly as the first one left it. The file is named to be collected last, so
that a run stopping at the first failure has already run every other test.
"""
import pytest
import torch

from parity import TOL, rel_err
from retention_gb300 import la, workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    # 8 sequences: split into segments, scratch from the fixed array
    "gated-split": (W.workload("gla", B=1, H=8, L=8192), 3),
    # normalised, 8 sequences, ragged length: split, z carried through the scratch
    "normalised-split": (W.workload("la", B=2, H=4, L=2000), 3),
    # 128 sequences: one CTA per sequence, no scratch at all
    "retention-unsplit": (W.workload("retention", B=8, H=16, L=512), 1),
}


def _device_inputs(cfg, seed):
    x = W.chunk_inputs(cfg, seed)
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def _poisoned(cfg, like):
    B, H, L, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dv"]
    out = torch.full((B, H, L, dv), float("nan"), dtype=like.dtype, device="cuda")
    st = torch.full((B, H, la.state_block(cfg["dk"], dv, cfg["normalize"])), float("nan"),
                    dtype=torch.float32, device="cuda")
    return out, st


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_chunk_fwd_on_two_calls(name):
    cfg, launches_per_call = CASES[name]
    kw = dict(phi=cfg["phi"], normalize=cfg["normalize"], gate_kind=cfg["gate"], chunk=cfg["chunk"])
    x = _device_inputs(cfg, seed=11)
    ref_out, ref_st = la.chunk_fwd(x["q"], x["k"], x["v"], x["gate"], **kw)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_st = ref_st.cpu().numpy()
    for call in range(2):
        out, st = _poisoned(cfg, x["q"])
        n0 = la.kernel_launches()
        la.chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["gate"], out=out, final_state=st, **kw)
        torch.cuda.synchronize()
        assert la.kernel_launches() - n0 == launches_per_call
        e_out = rel_err(out.float().cpu().numpy(), ref_out)
        e_st = rel_err(st.cpu().numpy(), ref_st)
        assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (call, e_out, e_st)


def test_noalloc_second_call_after_a_different_shape():
    """The array keeps whatever the previous call left; a call with other sizes
    right after must not read any of it."""
    a_cfg, _ = CASES["normalised-split"]
    b_cfg, _ = CASES["gated-split"]
    for cfg in (a_cfg, b_cfg, a_cfg):
        kw = dict(phi=cfg["phi"], normalize=cfg["normalize"], gate_kind=cfg["gate"], chunk=cfg["chunk"])
        x = _device_inputs(cfg, seed=5)
        ref_out, ref_st = la.chunk_fwd(x["q"], x["k"], x["v"], x["gate"], **kw)
        out, st = _poisoned(cfg, x["q"])
        la.chunk_fwd_noalloc(x["q"], x["k"], x["v"], x["gate"], out=out, final_state=st, **kw)
        torch.cuda.synchronize()
        assert rel_err(out.float().cpu().numpy(), ref_out.float().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(st.cpu().numpy(), ref_st.cpu().numpy()) <= TOL["bf16"]
