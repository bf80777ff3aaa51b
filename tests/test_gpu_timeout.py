"""The bounded waits of the tensor-core forward, made to run out on purpose.

Every wait of that kernel on an mbarrier gives up after a time limit (2 s in
ordinary calls). la_chunk_fwd_stall_test launches it with the TMA producer
issuing no tiles from a given chunk on and a limit of 20 ms: the roles left
waiting must leave their loops together (each group's decision to leave goes
through one barrier reduction), the CTA must drain what it issued and free its
tensor memory, and the kernel must return with its error word set. Nothing
faults or hangs: afterwards la_device_status reports LA_ERR_TIMEOUT once, a
second read is clean, and an ordinary call right after matches the oracle.
"""
import time

import pytest
import torch

from parity import TOL, rel_err, run_gpu, run_oracle
from retention_gb300 import la, workloads as W

pytestmark = pytest.mark.gpu


def _unsplit_heads():
    # enough (b, h) sequences that the forward runs one CTA per sequence (no split)
    return torch.cuda.get_device_properties(0).multi_processor_count // 2 + 4


@pytest.mark.parametrize("name", ["la", "retention", "gla"])
def test_bounded_wait_runs_out_and_the_context_stays_usable(name):
    assert la.device_status() == 0
    H = _unsplit_heads()
    cfg = W.workload(name, B=1, H=H, L=192)
    inp = W.chunk_inputs(cfg, seed=31)
    x = {n: (None if t is None else t.cuda()) for n, t in inp.items()}
    t0 = time.perf_counter()
    la.chunk_fwd_stall_test(x["q"], x["k"], x["v"], x["gate"], phi=cfg["phi"], normalize=cfg["normalize"],
                            gate_kind=cfg["gate"], stall_chunk=1, wait_ns=20_000_000)
    st = la.device_status()
    elapsed = time.perf_counter() - t0
    assert st == -5, st  # LA_ERR_TIMEOUT
    assert elapsed < 1.5, elapsed
    assert la.device_status() == 0
    # the same case through the ordinary call, right after
    out_ref, st_ref = run_oracle(inp, cfg)
    out, stt = run_gpu(inp, cfg)
    e_out, e_st = rel_err(out, out_ref), rel_err(stt, st_ref)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)
    assert la.device_status() == 0


def test_stall_past_the_last_chunk_is_an_ordinary_run():
    H = _unsplit_heads()
    cfg = W.workload("la", B=1, H=H, L=192)
    inp = W.chunk_inputs(cfg, seed=32)
    x = {n: (None if t is None else t.cuda()) for n, t in inp.items()}
    out = la.chunk_fwd_stall_test(x["q"], x["k"], x["v"], phi="elu1", normalize=True, stall_chunk=3,
                                  wait_ns=20_000_000)
    assert la.device_status() == 0
    out_ref, _ = run_oracle(inp, cfg)
    assert rel_err(out.float().cpu().numpy(), out_ref) <= TOL["bf16"]


def test_stall_arguments_are_checked():
    q = torch.zeros(1, 2, 64, 128, dtype=torch.bfloat16, device="cuda")
    for kw, status in ((dict(wait_ns=10), -1), (dict(stall_chunk=-1), -1)):
        with pytest.raises(la.LAError) as e:
            la.chunk_fwd_stall_test(q, q, q, **kw)
        assert e.value.status == status
    # two sequences of ten chunks would be split into segments: not this diagnostic's case
    q = torch.zeros(1, 2, 640, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(la.LAError) as e:
        la.chunk_fwd_stall_test(q, q, q)
    assert e.value.status == -2
