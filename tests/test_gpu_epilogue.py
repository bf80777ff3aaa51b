"""GPU parity of the RetNet output epilogue (swish(og) * GroupNorm_h(o)) against
the fp64 oracle on the same seeded inputs: la_group_norm_swish on its own, and
la_chunk_fwd_gn_swish, the chunk forward followed by it."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, rel_err, run_oracle, to_dev
from retention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _host(t):
    return None if t is None else t.float().numpy()


def _gn_ref(o_ref, ep, eps, affine):
    return oracle.group_norm_swish(o_ref, _host(ep["og"]), _host(ep["weight"]) if affine else None,
                                   _host(ep["bias"]) if affine else None, eps=eps)


# ------------------------------------------------------------------ la_group_norm_swish

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dv", [16, 32, 64, 128])
@pytest.mark.parametrize("affine", [True, False], ids=["affine", "plain"])
def test_group_norm_swish(dtype, dv, affine):
    """Ragged row count (B H L = 2 * 3 * 37), rows of every supported width."""
    from retention_gb300 import la
    cfg = W.workload("retnet", B=2, H=3, L=37, dv=dv, dtype=dtype)
    gen = torch.Generator("cpu").manual_seed(dv)
    x = (torch.randn(2, 3, 37, dv, generator=gen) * 0.3 + torch.randn(2, 3, 37, 1, generator=gen))
    x = x.to(W.TORCH_DTYPES[dtype])
    ep = W.epilogue_inputs(cfg, seed=dv)
    d = to_dev(dict(x=x, **ep))
    out = torch.full_like(d["x"], float("nan"))
    la.group_norm_swish(d["x"], d["og"], gn_weight=d["weight"] if affine else None,
                        gn_bias=d["bias"] if affine else None, gn_eps=1e-5, out=out)
    torch.cuda.synchronize()
    ref = _gn_ref(_host(x).astype(np.float64), ep, 1e-5, affine)
    assert rel_err(out.float().cpu().numpy(), ref) <= TOL[dtype]


def test_group_norm_swish_in_place_and_decode_shape():
    """out = x (in place) on a decode output [B, H, d_v]."""
    from retention_gb300 import la
    gen = torch.Generator("cpu").manual_seed(5)
    x = torch.randn(4, 16, 128, generator=gen).to(torch.bfloat16)
    og = torch.randn(4, 16, 128, generator=gen).to(torch.bfloat16)
    xd, ogd = x.cuda(), og.cuda()
    la.group_norm_swish(xd, ogd, gn_eps=1e-6, out=xd)
    torch.cuda.synchronize()
    ref = oracle.group_norm_swish(_host(x)[:, :, None].astype(np.float64), _host(og)[:, :, None], eps=1e-6)
    assert rel_err(xd.float().cpu().numpy(), ref[:, :, 0]) <= TOL["bf16"]


def test_group_norm_swish_rejects_bad_arguments():
    from retention_gb300 import la
    x = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16, device="cuda")
    lib = la.load()
    s = la._stream(None)
    vp = lambda t: la._dev(t, "t")
    assert lib.la_group_norm_swish(vp(x), vp(x), None, None, -1.0, vp(x), 1, 2, 4, 128, 0, s) == -1
    assert lib.la_group_norm_swish(vp(x), vp(x), None, None, float("nan"), vp(x), 1, 2, 4, 128, 0, s) == -1
    assert lib.la_group_norm_swish(vp(x), None, None, None, 1e-5, vp(x), 1, 2, 4, 128, 0, s) == -1
    assert lib.la_group_norm_swish(vp(x), vp(x), None, None, 1e-5, vp(x), 1, 2, 4, 48, 0, s) == -2
    odd = torch.zeros(300, device="cuda")
    import ctypes
    w_odd = ctypes.c_void_p(odd.data_ptr() + 4)
    assert lib.la_group_norm_swish(vp(x), vp(x), w_odd, None, 1e-5, vp(x), 1, 2, 4, 128, 0, s) == -3
    # an empty batch is a no-op
    assert lib.la_group_norm_swish(None, None, None, None, 1e-5, None, 0, 2, 4, 128, 0, s) == 0


# ------------------------------------------------------------------ la_chunk_fwd_gn_swish

def _check_fused(cfg, seed=0, simt=False, initial_state=None, affine=True):
    from retention_gb300 import la
    inp = W.chunk_inputs(cfg, seed)
    ep = W.epilogue_inputs(cfg, seed)
    eps = cfg.get("gn_eps", 1e-5)
    o_ref, st_ref = run_oracle(inp, cfg, state_in=None if initial_state is None else initial_state.numpy())
    ref = _gn_ref(o_ref, ep, eps, affine)
    x = to_dev(inp)
    e = to_dev(ep)
    B, H, L, dk = x["q"].shape
    dv = x["v"].shape[-1]
    out = torch.full((B, H, L, dv), float("nan"), dtype=x["q"].dtype, device="cuda")
    st = torch.full((B, H, la.state_block(dk, dv, cfg["normalize"])), float("nan"), device="cuda")
    n0 = la.kernel_launches()
    la.chunk_fwd_gn_swish(x["q"], x["k"], x["v"], e["og"], x["gate"], gn_weight=e["weight"] if affine else None,
                          gn_bias=e["bias"] if affine else None, gn_eps=eps, phi=cfg["phi"],
                          normalize=cfg["normalize"], gate_kind=cfg["gate"], chunk=cfg["chunk"], out=out,
                          final_state=st, simt=simt,
                          initial_state=None if initial_state is None else initial_state.cuda())
    torch.cuda.synchronize()
    launches = la.kernel_launches() - n0
    tol = TOL[cfg["dtype"]]
    e_out, e_st = rel_err(out.float().cpu().numpy(), ref), rel_err(st.cpu().numpy(), st_ref)
    assert e_out <= tol and e_st <= tol, (e_out, e_st)
    return launches


TC_FORMS = [
    dict(phi="identity", normalize=False, gate="head"),   # retention (RetNet)
    dict(phi="elu1", normalize=False, gate=None),
    dict(phi="identity", normalize=False, gate=None),
    dict(phi="elu1", normalize=True, gate="head"),
    dict(phi="elu1", normalize=True, gate=None),
    dict(phi="elu1", normalize=False, gate="channel"),
    dict(phi="elu1", normalize=True, gate="channel"),
]


def _fuses(m):
    # the epilogue goes into the tensor-core kernel's store without the
    # normaliser and the per-channel gate; otherwise it is a kernel of its own
    return not m["normalize"] and m["gate"] != "channel"


@pytest.mark.parametrize("m", TC_FORMS, ids=lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"]))
@pytest.mark.parametrize("B,H,L", [(2, 40, 200), (1, 2, 1000), (2, 3, 333), (2, 40, 1)],
                         ids=["unsplit", "split", "ragged", "one-token"])
def test_tensor_core_forms(m, B, H, L):
    """Every form through the tensor-core kernel (one launch, or three for
    split sequences): with the epilogue in its store (no normaliser, no
    per-channel gate), or followed by the epilogue kernel."""
    cfg = W.workload("retnet", B=B, H=H, L=L, **m)
    launches = _check_fused(cfg, seed=11)
    assert launches in ((1, 3) if _fuses(m) else (2, 4)), launches


@pytest.mark.parametrize("L", [64, 65, 4000], ids=["one-chunk", "chunk-and-a-token", "long"])
def test_fused_store_rows_and_window_ends(L):
    """The epilogue in the store on retention decays whose rescale windows
    close after 1 to 625 chunks, with a final chunk of every fill."""
    from test_gpu_chunk import window_inputs
    from retention_gb300 import la
    cfg = W.workload("retnet", B=2, H=40, L=L)
    inp = window_inputs(cfg, seed=L)
    ep = W.epilogue_inputs(cfg, seed=L)
    o_ref, st_ref = run_oracle(inp, cfg)
    ref = _gn_ref(o_ref, ep, cfg["gn_eps"], True)
    x, e = to_dev(inp), to_dev(ep)
    out = torch.full((2, 40, L, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    n0 = la.kernel_launches()
    _, st = la.chunk_fwd_gn_swish(x["q"], x["k"], x["v"], e["og"], x["gate"], gn_weight=e["weight"],
                                  gn_bias=e["bias"], gn_eps=cfg["gn_eps"], phi="identity", gate_kind="head",
                                  out=out)
    torch.cuda.synchronize()
    assert la.kernel_launches() - n0 == 1
    assert rel_err(out.float().cpu().numpy(), ref) <= TOL["bf16"]
    assert rel_err(st.cpu().numpy(), st_ref) <= TOL["bf16"]


@pytest.mark.parametrize("affine", [True, False], ids=["affine", "plain"])
def test_without_affine_and_from_a_state(affine):
    cfg = W.workload("retnet", B=2, H=4, L=300)
    gen = torch.Generator("cpu").manual_seed(21)
    S0 = torch.randn(2, 4, 128 * 128, generator=gen) * 0.1
    assert _check_fused(cfg, seed=13, affine=affine, initial_state=S0) == 3  # split, epilogue in the store


@pytest.mark.parametrize("dtype,dk,dv", [("f32", 32, 16), ("f32", 64, 64), ("bf16", 128, 128)])
def test_general_kernel_then_epilogue(dtype, dk, dv):
    cfg = W.workload("retnet", B=2, H=3, L=77, dk=dk, dv=dv, dtype=dtype, chunk=16)
    launches = _check_fused(cfg, seed=14, simt=True)
    assert launches == 2, launches


def test_full_size_retnet_workload():
    """The retnet workload (retention, B=8 H=16 L=4096 d=128) in the launch the
    benchmark times, element by element against the oracle."""
    launches = _check_fused(W.workload("retnet"), seed=0)
    assert launches == 1  # the epilogue runs in the forward kernel's store


def test_fused_call_requires_the_gate():
    from retention_gb300 import la
    x = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    vp = lambda t: la._dev(t, "t")
    rc = la.load().la_chunk_fwd_gn_swish(vp(x), vp(x), vp(x), None, None, None, None, None, 1e-5, vp(x), None,
                                         1, 1, 64, 128, 128, 0, 64, la._stream(None))
    assert rc == -1
