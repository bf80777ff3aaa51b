"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded inputs and measure max|gpu - oracle| / max|oracle|."""
import numpy as np
import torch

import oracle

# tolerances: fp32 path and bf16 inputs with fp32 accumulation
TOL = {"f32": 1e-4, "bf16": 2e-2}


def oracle_mode(cfg):
    m = 0
    if cfg["phi"] == "elu1":
        m |= oracle.PHI_ELU1
    if cfg["normalize"]:
        m |= oracle.NORMALIZE
    if cfg["gate"] == "head":
        m |= oracle.GATE_HEAD
    elif cfg["gate"] == "channel":
        m |= oracle.GATE_CHANNEL
    return m


def host(t):
    return None if t is None else t.float().numpy()


def run_oracle(inp, cfg, state_in=None, nthreads=0):
    return oracle.forward(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["gate"]),
                          oracle_mode(cfg), state_in=state_in, nthreads=nthreads)


def to_dev(inp):
    d = torch.device("cuda")
    return {k: (None if v is None else v.to(d)) for k, v in inp.items()}


def run_gpu(inp, cfg, chunk=None, simt=False, initial_state=None, reverse=False):
    """la_chunk_fwd (la_chunk_fwd_from_state with ``initial_state``, a [B,H,block]
    float32 tensor) through the binding; outputs are NaN-poisoned first so that
    an element the kernel never writes fails the comparison."""
    from retention_gb300 import la
    x = to_dev(inp)
    B, H, L, dk = x["q"].shape
    dv = x["v"].shape[-1]
    out = torch.full((B, H, L, dv), float("nan"), dtype=x["q"].dtype, device="cuda")
    st = torch.full((B, H, la.state_block(dk, dv, cfg["normalize"])), float("nan"),
                    dtype=torch.float32, device="cuda")
    la.chunk_fwd(x["q"], x["k"], x["v"], x["gate"], phi=cfg["phi"], normalize=cfg["normalize"],
                 gate_kind=cfg["gate"], chunk=chunk or cfg["chunk"], out=out, final_state=st,
                 simt=simt, initial_state=None if initial_state is None else initial_state.cuda(),
                 reverse=reverse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st.cpu().numpy()


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite values in the GPU result"
    return float(np.max(np.abs(got - ref)) / max(float(np.max(np.abs(ref))), 1e-300))
