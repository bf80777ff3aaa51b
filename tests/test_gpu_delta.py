"""GPU parity of la_delta_fwd (the delta rule) against the fp64 recurrent
oracle on the same seeded inputs, for both kernels: the chunked tensor-core
one (bf16, d = 128, the default there) and the token-by-token one
(LA_KERNEL_SIMT, and every other case): bf16 and fp32, every head size,
ragged and tiny lengths, chunk boundaries, the full workload, and the
read-back property of unit keys."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, rel_err
from retention_gb300 import la, workloads as W

pytestmark = pytest.mark.gpu


def _run(cfg, seed, beta_one=False, q_is_k=False, simt=False):
    x = W.delta_inputs(cfg, seed)
    if beta_one:
        x["beta"] = torch.ones_like(x["beta"])
    if q_is_k:
        x["q"] = x["k"].clone()
    out_ref, st_ref = oracle.delta_forward(*(x[n].float().numpy() for n in ("q", "k", "v", "beta")))
    d = {n: t.cuda() for n, t in x.items()}
    B, H, L, dk = d["q"].shape
    dv = d["v"].shape[-1]
    out = torch.full((B, H, L, dv), float("nan"), dtype=d["q"].dtype, device="cuda")
    st = torch.full((B, H, dv * dk), float("nan"), dtype=torch.float32, device="cuda")
    la.delta_fwd(d["q"], d["k"], d["v"], d["beta"], out=out, final_state=st, simt=simt)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st.cpu().numpy(), out_ref, st_ref, x


def _check(cfg, seed=0, simt=False):
    out, st, out_ref, st_ref, _ = _run(cfg, seed, simt=simt)
    tol = TOL[cfg["dtype"]]
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= tol and e_st <= tol, (e_out, e_st)


@pytest.mark.parametrize("simt", [False, True], ids=["chunked", "recurrent"])
def test_bf16_small_ragged(simt):
    _check(W.workload("delta", B=2, H=3, L=333), seed=1, simt=simt)


@pytest.mark.parametrize("dk,dv", [(16, 128), (128, 16), (64, 64), (32, 32), (128, 128)])
def test_fp32_head_dims(dk, dv):
    _check(W.workload("delta", B=2, H=3, L=77, dk=dk, dv=dv, dtype="f32"), seed=2)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 129, 200])
@pytest.mark.parametrize("simt", [False, True], ids=["chunked", "recurrent"])
def test_block_boundaries(L, simt):
    """The recurrent kernel's 32-token blocks, the chunked kernel's 64-token
    chunks and its 16-row blocks of the triangular inverse."""
    _check(W.workload("delta", B=1, H=4, L=L), seed=L, simt=simt)


@pytest.mark.parametrize("simt", [False, True], ids=["chunked", "recurrent"])
def test_full_size_workload(simt):
    """The workload the benchmark times, element by element against the oracle."""
    _check(W.workload("delta"), seed=0, simt=simt)


def test_chunked_kernel_is_the_default_and_one_launch():
    """T of every chunk and the state recurrence in one kernel."""
    cfg = W.workload("delta", B=2, H=2, L=100)
    d = {n: t.cuda() for n, t in W.delta_inputs(cfg, 0).items()}
    n0 = la.kernel_launches()
    la.delta_fwd(d["q"], d["k"], d["v"], d["beta"])
    torch.cuda.synchronize()
    assert la.kernel_launches() - n0 == 1


@pytest.mark.parametrize("simt", [False, True], ids=["chunked", "recurrent"])
def test_unit_keys_read_back_their_values_bf16(simt):
    """beta = 1, queries = the unit keys: out_t = v_t (S_t k_t = v_t after the
    write), within the bf16 tolerance."""
    cfg = W.workload("delta", B=2, H=4, L=300)
    out, _, _, _, x = _run(cfg, seed=4, beta_one=True, q_is_k=True, simt=simt)
    v = x["v"].float().numpy()
    assert rel_err(out, v) <= TOL["bf16"]


def test_unit_keys_read_back_their_values():
    """With beta = 1 and queries equal to the (unit) keys, every output is the
    value just written (S_t k_t = v_t), up to the bf16 rounding of the inputs."""
    cfg = W.workload("delta", B=2, H=4, L=300, dtype="f32")
    out, _, _, _, x = _run(cfg, seed=3, beta_one=True, q_is_k=True)
    np.testing.assert_allclose(out, x["v"].numpy(), rtol=0, atol=2e-5)


def test_empty_sequence_gives_zero_state():
    q = torch.empty(2, 3, 0, 128, dtype=torch.bfloat16, device="cuda")
    beta = torch.empty(2, 3, 0, dtype=torch.bfloat16, device="cuda")
    st = torch.full((2, 3, 128 * 128), float("nan"), device="cuda")
    la.delta_fwd(q, q, q, beta, out=torch.empty_like(q), final_state=st)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st).item() == 0


def test_gate_or_feature_bits_are_rejected():
    cfg = W.workload("delta", B=1, H=1, L=8)
    d = {n: t.cuda() for n, t in W.delta_inputs(cfg, 0).items()}
    out = torch.empty_like(d["v"])
    st = torch.empty(1, 1, 128 * 128, device="cuda")
    rc = la.load().la_delta_fwd(*(la._dev(d[n], n) for n in ("q", "k", "v", "beta")), la._dev(out, "out"),
                                la._dev(st, "st"), 1, 1, 8, 128, 128, la.LA_PHI_ELU1, la._stream(None))
    assert rc == -1  # LA_ERR_INVALID_ARG
