"""GPU parity of la_chunk_fwd against the fp64 oracle on the same seeded
inputs: the five workloads' chunk-forward shapes, the worked example, every
mode, ragged lengths, several chunk sizes and the edge cases."""
import json
import os

import numpy as np
import pytest
import torch

from parity import TOL, rel_err, run_gpu, run_oracle, to_dev
from retention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _check(cfg, seed=0, chunk=None, simt=False, tol=None):
    inp = W.chunk_inputs(cfg, seed)
    out_ref, st_ref = run_oracle(inp, cfg)
    out, st = run_gpu(inp, cfg, chunk=chunk, simt=simt)
    tol = tol or TOL[cfg["dtype"]]
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= tol and e_st <= tol, (e_out, e_st)
    return e_out, e_st


# ------------------------------------------------------------------ fp32 path

def test_tiny_workload():
    _check(W.workload("tiny"))


@pytest.mark.parametrize("chunk", [1, 2, 3, 16])
def test_worked_example_through_the_kernel(chunk):
    """insideout lesson 16, Example 1.1 and "Your turn", zero-padded to d = 16:
    (0.5, 3) after two tokens and (1.5, 2.5) after the third."""
    gd = json.load(open(GOLDEN))
    pad = lambda rows: torch.tensor([r + [0.0] * 14 for r in rows], dtype=torch.float32)[None, None]
    inp = dict(q=pad(gd["queries"]), k=pad(gd["keys"]), v=pad(gd["values"]), gate=None)
    cfg = W.workload("tiny", B=1, H=1, L=3, phi="identity", normalize=True)
    out, st = run_gpu(inp, cfg, chunk=chunk)
    np.testing.assert_allclose(out[0, 0, 1, :2], gd["after_two_tokens"]["out"], atol=1e-6)
    np.testing.assert_allclose(out[0, 0, 2, :2], gd["after_three_tokens"]["out"], atol=1e-6)
    S = st[0, 0, :256].reshape(16, 16)
    np.testing.assert_allclose(S[:2, :2], gd["after_three_tokens"]["state_S"], atol=1e-6)
    np.testing.assert_allclose(st[0, 0, 256:258], gd["after_three_tokens"]["state_z"], atol=1e-6)


FP32_MODES = [
    dict(phi="elu1", normalize=True, gate=None),
    dict(phi="elu1", normalize=False, gate=None),
    dict(phi="identity", normalize=False, gate=None),
    dict(phi="identity", normalize=False, gate="head"),
    dict(phi="elu1", normalize=True, gate="head"),
    dict(phi="elu1", normalize=False, gate="channel"),
    dict(phi="elu1", normalize=True, gate="channel"),
    dict(phi="identity", normalize=False, gate="channel"),
]


@pytest.mark.parametrize("m", FP32_MODES, ids=lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"]))
@pytest.mark.parametrize("L,chunk", [(13, 1), (13, 4), (13, 7), (13, 13), (77, 16), (77, 64), (200, 128)])
def test_fp32_modes_chunks_ragged(m, L, chunk):
    cfg = W.workload("tiny", B=2, H=3, L=L, dk=32, dv=16, gamma_step=1.0, **m)
    _check(cfg, seed=L + chunk)


@pytest.mark.parametrize("dk,dv", [(16, 128), (128, 16), (64, 64), (128, 128)])
def test_fp32_head_dims(dk, dv):
    cfg = W.workload("tiny", B=1, H=2, L=70, dk=dk, dv=dv, gate="channel", normalize=False)
    _check(cfg, seed=dk + dv, chunk=32)


# ------------------------------------------------------------------ bf16, small

BF16_SMALL = {
    "la": dict(B=2, H=3, L=333),
    "retention": dict(B=2, H=16, L=333),
    "gla": dict(B=1, H=3, L=1000),
}


@pytest.mark.parametrize("name", list(BF16_SMALL))
@pytest.mark.parametrize("simt", [False, True], ids=["default", "simt"])
def test_bf16_small_ragged(name, simt):
    cfg = W.workload(name, **BF16_SMALL[name])
    _check(cfg, seed=3, simt=simt)


@pytest.mark.parametrize("name", list(BF16_SMALL))
@pytest.mark.parametrize("L", [1, 63, 64, 65, 129])
def test_bf16_chunk_boundaries(name, L):
    cfg = W.workload(name, **dict(BF16_SMALL[name], L=L))
    _check(cfg, seed=L)


# ------------------------------------------------------------------ bf16, every mode on the tensor cores

@pytest.mark.parametrize("m", FP32_MODES, ids=lambda m: "%s-%s-%s" % (m["phi"], m["normalize"], m["gate"]))
@pytest.mark.parametrize("B,H,L", [(1, 2, 1000), (2, 40, 200)], ids=["split", "unsplit"])
def test_bf16_modes_tensor_cores(m, B, H, L):
    """Every feature-map / normaliser / gate combination through the
    tensor-core kernel, with few sequences (each cut into segments: state-only
    pass, scan, full pass) and with one CTA per sequence. The combinations have
    their own shared-memory layouts (stage count, shared ones block, gate ring)."""
    from retention_gb300 import la
    cfg = W.workload("la", B=B, H=H, L=L, **m)
    mode = la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"])
    assert la.chunk_fwd_path(B, H, L, cfg["dk"], cfg["dv"], mode, cfg["chunk"]) == 1
    _check(cfg, seed=7)


# ------------------------------------------------------------------ full size

@pytest.mark.parametrize("name", ["la", "retention", "gla"])
def test_full_size_workload(name):
    """The full workloads, in the launch configuration the benchmark times,
    compared element by element with the oracle."""
    _check(W.workload(name))


# ------------------------------------------------------------------ edges

def test_empty_sequence_gives_zero_state():
    from retention_gb300 import la
    q = torch.zeros(2, 3, 0, 16, device="cuda")
    st = torch.full((2, 3, 16 * 16 + 16), float("nan"), device="cuda")
    out = torch.empty(2, 3, 0, 16, device="cuda")
    la.chunk_fwd(q, q, torch.zeros(2, 3, 0, 16, device="cuda"), normalize=True, out=out,
                 final_state=st, chunk=16)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st).item() == 0


def test_misaligned_and_missing_gate_are_rejected():
    from retention_gb300 import la
    base = torch.zeros(1 * 1 * 9 * 16 + 1, device="cuda")
    q = base[1:].view(1, 1, 9, 16)             # 4-byte offset
    good = torch.zeros(1, 1, 9, 16, device="cuda")
    with pytest.raises(la.LAError) as e:
        la.chunk_fwd(q, good, good, chunk=4)
    assert e.value.status == -3
    with pytest.raises(la.LAError) as e:
        la.chunk_fwd(good, good, good, None, gate_kind="channel", chunk=4)
    assert e.value.status == -1


def test_launch_counter_advances():
    from retention_gb300 import la
    n0 = la.kernel_launches()
    cfg = W.workload("tiny", L=16)
    run_gpu(W.chunk_inputs(cfg), cfg)
    assert la.kernel_launches() >= n0 + 1


@pytest.mark.parametrize("name", ["la", "retention", "gla"])
def test_bf16_workloads_take_the_tensor_core_kernel(name):
    from retention_gb300 import la
    cfg = W.workload(name)
    mode = la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"])
    assert la.chunk_fwd_path(cfg["B"], cfg["H"], cfg["L"], 128, 128, mode, 64) == 1
    assert la.chunk_fwd_path(cfg["B"], cfg["H"], cfg["L"], 128, 128, mode | la.LA_KERNEL_SIMT, 64) == 0
    assert la.chunk_fwd_path(cfg["B"], cfg["H"], cfg["L"], 128, 128, mode, 32) == 0


def test_device_status_is_clean_after_the_bounded_wait_kernels():
    """la_device_status: none of the kernels with bounded waits (the
    tensor-core forward, the chunked delta rule) gave one up on ordinary
    inputs, and a second read finds the flags still clear."""
    from retention_gb300 import la
    assert la.device_status() == 0  # no earlier call in this process gave a wait up
    cfg = W.workload("la", B=1, H=2, L=300)
    x = {n: t.cuda() for n, t in W.chunk_inputs(cfg, 1).items() if t is not None}
    la.chunk_fwd(x["q"], x["k"], x["v"], phi="elu1", normalize=True, chunk=64)
    dcfg = W.workload("delta", B=1, H=2, L=300)
    d = {n: t.cuda() for n, t in W.delta_inputs(dcfg, 1).items()}
    la.delta_fwd(d["q"], d["k"], d["v"], d["beta"])
    assert la.device_status() == 0
    assert la.device_status() == 0
    assert la.load().la_status_string(-5).decode().startswith("LA_ERR_TIMEOUT")


# ------------------------------------------------------------------ retention windows

# Decays whose rescale windows of the tensor-core kernel (the accumulator holds
# S / gamma^(64 m) for m chunks, rescaled once per window) close after 1, 2, 5,
# 12, 20, 41, 62 and 625 chunks, so that short runs cross window ends.
WINDOW_GAMMAS = [0.5, 0.8, 0.9, 0.95, 0.97, 0.985, 0.99, 0.999]


def window_inputs(cfg, seed):
    inp = W.chunk_inputs(cfg, seed)
    inp["gate"] = torch.tensor([WINDOW_GAMMAS[h % len(WINDOW_GAMMAS)] for h in range(cfg["H"])],
                               dtype=torch.float32)
    return inp


@pytest.mark.parametrize("B,H,L", [(1, 8, 6100), (2, 40, 1300)], ids=["split", "unsplit"])
def test_retention_window_ends(B, H, L):
    """Retention through the tensor-core kernel with windows that end inside
    each CTA's run of chunks: split (8 sequences, segments of 6 chunks) and
    unsplit (80 sequences of 21 chunks), ragged lengths."""
    from retention_gb300 import la
    cfg = W.workload("retention", B=B, H=H, L=L)
    assert la.chunk_fwd_path(B, H, L, 128, 128, la.mode_bits("identity", False, "head"), 64) == 1
    inp = window_inputs(cfg, seed=21)
    out_ref, st_ref = run_oracle(inp, cfg)
    out, st = run_gpu(inp, cfg)
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


# ------------------------------------------------------------------ the anti-causal form (LA_REVERSE)

def _flip(inp):
    return {n: (t.flip(2) if (t is not None and t.dim() == 4) else t) for n, t in inp.items()}


def _reversed_inputs(inp, cfg):
    """The token-reversed sequence; with the per-channel gate, reversed token u
    decays by the gate of original token L - u, and reversed token 0 by none
    (a gate of 30: alpha = sigmoid(30)^(1/16), 1 to within 1e-14)."""
    flip = _flip(inp)
    if cfg["gate"] == "channel":
        g = flip["gate"]
        flip["gate"] = torch.cat([torch.full_like(g[:, :, :1], 30.0), g[:, :, :-1]], dim=2)
    return flip


def _check_reverse(cfg, inp, initial_state=None):
    """LA_REVERSE sums over the token and every later one; that is the causal
    recurrence of the token-reversed sequence (with the per-channel gate, of
    the gate shifted by a token), which the oracle computes (its final state is
    the state before token 0)."""
    s0 = None if initial_state is None else initial_state.numpy()
    out_ref, st_ref = run_oracle(_reversed_inputs(inp, cfg), cfg, state_in=s0)
    out_ref = out_ref[:, :, ::-1]
    out, st = run_gpu(inp, cfg, reverse=True, initial_state=initial_state)
    e_out, e_st = rel_err(out, out_ref), rel_err(st, st_ref)
    assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (e_out, e_st)


@pytest.mark.parametrize("phi,gate", [("identity", None), ("identity", "head"), ("elu1", None),
                                      ("identity", "channel"), ("elu1", "channel")])
@pytest.mark.parametrize("B,H,L", [(1, 4, 1000), (2, 40, 333), (2, 40, 129), (1, 80, 64), (1, 80, 1)],
                         ids=["split", "unsplit-ragged", "unsplit-129", "one-chunk", "one-token"])
def test_reverse_matches_the_reversed_causal_oracle(phi, gate, B, H, L):
    from retention_gb300 import la
    cfg = W.workload("gla" if gate == "channel" else "retention", B=B, H=H, L=L, gate=gate, phi=phi)
    mode = la.mode_bits(phi, False, gate, reverse=True)
    assert la.chunk_fwd_path(B, H, L, 128, 128, mode, 64) == 1
    _check_reverse(cfg, W.chunk_inputs(cfg, seed=L + H))


@pytest.mark.parametrize("B,H,L", [(1, 8, 6100), (2, 40, 1300)], ids=["split", "unsplit"])
def test_reverse_window_ends(B, H, L):
    """Decays whose rescale windows close after 1 to 625 chunks, on ragged
    lengths: the reverse form takes the ragged chunk first, and that chunk
    closes a window of its own."""
    cfg = W.workload("retention", B=B, H=H, L=L)
    _check_reverse(cfg, window_inputs(cfg, seed=23))


@pytest.mark.parametrize("name", ["retention", "gla"])
@pytest.mark.parametrize("B,H,L", [(1, 4, 1000), (2, 40, 333)], ids=["split", "unsplit"])
def test_reverse_from_a_state(name, B, H, L):
    """An initial state of the reverse form sits after the last token (with the
    per-channel gate it is decayed by the gates of tokens 1 .. L - 1 and by none
    for the last token's successor, as the reversed sequence's first token is)."""
    cfg = W.workload(name, B=B, H=H, L=L)
    s0 = W.decode_state(dict(cfg, state_std=0.1), 77)
    _check_reverse(cfg, W.chunk_inputs(cfg, seed=24), initial_state=s0)
