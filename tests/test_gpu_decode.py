"""GPU parity of la_decode_step against the oracle: the full decode batch
(256 sequences x 32 heads, the benchmark's launch configuration) for a few
steps, a 1000-step run on a subset of sequences, every gate mode, and the
prefill -> decode hand-off from la_chunk_fwd."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL, host, oracle_mode, rel_err, run_gpu, run_oracle, to_dev
from retention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _decode_run(cfg, steps, seed=0, batch=None):
    """Run `steps` decode steps on GPU and oracle from the same initial state.
    Returns (max rel err of outputs, rel err of final state)."""
    from retention_gb300 import la
    B = cfg["B"] if batch is None else len(batch)
    st0 = W.decode_state(cfg, seed)
    if batch is not None:
        st0 = st0[list(batch)].contiguous()
    st_ref = st0.double().numpy().copy()
    st_gpu = st0.cuda()
    mode = oracle_mode(cfg)
    outs_gpu, outs_ref = [], []
    for s in range(steps):
        tok = W.decode_tokens(cfg, s, seed, batch=batch)
        outs_ref.append(oracle.decode_step(host(tok["q"]), host(tok["k"]), host(tok["v"]), st_ref,
                                           host(tok["gate"]), mode))
        d = to_dev(tok)
        outs_gpu.append(la.decode_step(d["q"], d["k"], d["v"], st_gpu, d["gate"], phi=cfg["phi"],
                                       normalize=cfg["normalize"], gate_kind=cfg["gate"]))
    torch.cuda.synchronize()
    og = torch.stack(outs_gpu).float().cpu().numpy()
    return rel_err(og, np.stack(outs_ref)), rel_err(st_gpu.cpu().numpy(), st_ref)


def test_decode_full_batch_three_steps():
    cfg = W.workload("decode")
    e_out, e_st = _decode_run(cfg, 3)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


def test_decode_subset_thousand_steps():
    cfg = W.workload("decode")
    e_out, e_st = _decode_run(cfg, 1000, batch=range(8))
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


@pytest.mark.parametrize("m", [dict(gate="head", normalize=False, phi="identity"),
                               dict(gate="channel", normalize=False, phi="elu1"),
                               dict(gate="channel", normalize=True, phi="elu1"),
                               dict(gate=None, normalize=False, phi="elu1")],
                         ids=["retention", "gated", "gated-norm", "plain"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (16, 128)])
def test_decode_modes_and_dims(m, dk, dv):
    cfg = W.workload("decode", B=4, H=16, dk=dk, dv=dv, **m)
    e_out, e_st = _decode_run(cfg, 20)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


def test_decode_fp32_tokens():
    cfg = W.workload("decode", B=3, H=5, dtype="f32", gate="channel")
    e_out, e_st = _decode_run(cfg, 30)
    assert e_out <= TOL["f32"] and e_st <= TOL["f32"], (e_out, e_st)


@pytest.mark.parametrize("name", ["la", "retention", "gla"])
def test_prefill_then_decode(name):
    """learnllm m22 cell 4 (incremental == full recompute), across the ABI:
    la_chunk_fwd over L tokens, then n la_decode_step calls on its final
    state, equals the oracle over L + n tokens."""
    from retention_gb300 import la
    L, n = 150, 6
    cfg = W.workload(name, B=2, H=4, L=L + n)
    inp = W.chunk_inputs(cfg, 5)
    out_ref, st_ref = run_oracle(inp, cfg)
    pre = {k: (v if v is None or v.dim() == 1 else v[:, :, :L].contiguous()) for k, v in inp.items()}
    cfg_pre = dict(cfg, L=L)
    out_pre, st = run_gpu(pre, cfg_pre)
    assert rel_err(out_pre, out_ref[:, :, :L]) <= TOL["bf16"]
    state = torch.from_numpy(st).cuda()
    d = to_dev(inp)
    for s in range(n):
        t = L + s
        g = d["gate"]
        if cfg["gate"] == "channel":
            g = g[:, :, t].contiguous()
        o = la.decode_step(d["q"][:, :, t].contiguous(), d["k"][:, :, t].contiguous(),
                           d["v"][:, :, t].contiguous(), state, g, phi=cfg["phi"],
                           normalize=cfg["normalize"], gate_kind=cfg["gate"])
        torch.cuda.synchronize()
        assert rel_err(o.float().cpu().numpy(), out_ref[:, :, t]) <= TOL["bf16"]
    assert rel_err(state.cpu().numpy(), st_ref) <= TOL["bf16"]
