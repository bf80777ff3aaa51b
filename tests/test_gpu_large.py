"""Tensors past 2^31 elements: the forward and the backward over B=1, H=8,
L=2^21+37 (every [B,H,L,128] array holds 2.1e9 values, so the last heads'
offsets need 64-bit arithmetic) and a decode step on a 131168-head state
(2.2e9 floats).

With a strong decay the last outputs of a sequence depend on its last few
hundred tokens only: a token 256 places back weighs gamma^256 = 2^-256 with
gamma = 0.5 (retention), or e^-(over 70) with gates near -8 (gated), far below
bf16 resolution. So the oracle, run from a zero state on the last 448 tokens,
gives the exact last 192 outputs and the final state of the full sequence, and
the parity check runs on the heads whose data sit past 2^31 elements. The same
holds for the gradients of the last tokens: dq reads a decayed past, dk, dv
and the gate's gradient read only later tokens, all inside the suffix."""
import numpy as np
import pytest
import torch

import oracle
from parity import TOL

pytestmark = pytest.mark.gpu

L_BIG = (1 << 21) + 37  # 8 heads x L x 128 > 2^31 values per array
SUFFIX, CHECKED = 448, 192
HEADS = (0, 7)


def _rel(a, b):
    return float(np.max(np.abs(a - b))) / max(float(np.max(np.abs(b))), 1e-300)


def _host(t):
    return t.float().cpu().numpy()


def _check_suffix(q, k, v, gate, out, st, mode, channel_gate):
    for h in HEADS:
        sl = slice(L_BIG - SUFFIX, L_BIG)
        qs, ks, vs = (_host(x[:, h:h + 1, sl]) for x in (q, k, v))
        if channel_gate:
            gs = _host(gate[:, h:h + 1, sl])
        else:
            gs = _host(gate[h:h + 1])
        ref_out, ref_st = oracle.forward(qs, ks, vs, gs, mode)
        e_out = _rel(_host(out[:, h:h + 1, L_BIG - CHECKED:]), ref_out[:, :, SUFFIX - CHECKED:])
        e_st = _rel(st[:, h:h + 1].cpu().numpy(), ref_st)
        assert e_out <= TOL["bf16"] and e_st <= TOL["bf16"], (h, e_out, e_st)


def _inputs(gen, n, scale=128 ** -0.5):
    return [(torch.randn(1, 8, L_BIG, 128, generator=gen, device="cuda", dtype=torch.float32) * scale)
            .to(torch.bfloat16) for _ in range(n)]


def test_retention_beyond_2_31_elements():
    from retention_gb300 import la
    gen = torch.Generator(device="cuda").manual_seed(31)
    q, k, v = _inputs(gen, 3)
    gamma = torch.full((8,), 0.5, dtype=torch.float32, device="cuda")
    out, st = la.chunk_fwd(q, k, v, gamma, phi="identity", gate_kind="head")
    torch.cuda.synchronize()
    assert q.numel() > 2 ** 31  # the last head's rows sit past 2^31 values
    _check_suffix(q, k, v, gamma, out, st, oracle.GATE_HEAD, channel_gate=False)
    del q, k, v, out, st
    torch.cuda.empty_cache()


def test_gated_beyond_2_31_elements():
    from retention_gb300 import la
    gen = torch.Generator(device="cuda").manual_seed(32)
    q, k, v = _inputs(gen, 3)
    # gates near -8: each token's log decay is logsigmoid(g) / 16, about -0.5
    g = (torch.randn(1, 8, L_BIG, 128, generator=gen, device="cuda", dtype=torch.float32) - 8.0).to(torch.bfloat16)
    out, st = la.chunk_fwd(q, k, v, g, phi="elu1", gate_kind="channel")
    torch.cuda.synchronize()
    _check_suffix(q, k, v, g, out, st, oracle.PHI_ELU1 | oracle.GATE_CHANNEL, channel_gate=True)
    del q, k, v, g, out, st
    torch.cuda.empty_cache()


def test_decode_beyond_2_31_state_values():
    from retention_gb300 import la
    B, H, d = 4099, 32, 128  # 131168 heads x (128 x 128 + 128) floats
    gen = torch.Generator(device="cuda").manual_seed(33)
    blk = d * d + d
    state = torch.empty(B, H, blk, dtype=torch.float32, device="cuda")
    state[:, :, :d * d].normal_(0.0, 0.1, generator=gen)
    state[:, :, d * d:].uniform_(0.0, 1.0, generator=gen)
    assert state.numel() > 2 ** 31
    q, k, v = ((torch.randn(B, H, d, generator=gen, device="cuda") * d ** -0.5).to(torch.bfloat16) for _ in range(3))
    before = state[-1:, -2:].double().cpu().numpy()
    out = la.decode_step(q, k, v, state, phi="elu1", normalize=True)
    torch.cuda.synchronize()
    ref_state = before.copy()
    ref_out = oracle.decode_step(_host(q[-1:, -2:]), _host(k[-1:, -2:]), _host(v[-1:, -2:]), ref_state, None,
                                 oracle.PHI_ELU1 | oracle.NORMALIZE)
    assert _rel(_host(out[-1:, -2:]), ref_out) <= TOL["bf16"]
    assert _rel(state[-1:, -2:].cpu().numpy(), ref_state) <= TOL["bf16"]
    del state, q, k, v, out
    torch.cuda.empty_cache()


def _check_bwd_suffix(x, gate, grads, mode, channel_gate):
    tail = slice(SUFFIX - CHECKED, SUFFIX)
    for h in HEADS:
        sl = slice(L_BIG - SUFFIX, L_BIG)
        qs, ks, vs, ds = (_host(t[:, h:h + 1, sl]) for t in x)
        gs = _host(gate[:, h:h + 1, sl]) if channel_gate else _host(gate[h:h + 1])
        refs = [r[:, :, tail] for r in oracle.backward(qs, ks, vs, ds, gs, mode) if r is not None]
        gots = [_host(g[:, h:h + 1, L_BIG - CHECKED:]) for g in grads if g is not None]
        assert len(refs) == len(gots)
        # relative to the largest gradient, as in the other backward parity tests
        scale = max(float(np.max(np.abs(r))) for r in refs)
        errs = [float(np.max(np.abs(g - r))) / max(float(np.max(np.abs(r))), scale) for g, r in zip(gots, refs)]
        assert all(e <= TOL["bf16"] for e in errs), (h, errs)


def test_retention_backward_beyond_2_31_elements():
    from retention_gb300 import la
    gen = torch.Generator(device="cuda").manual_seed(34)
    q, k, v = _inputs(gen, 3)
    (dout,) = _inputs(gen, 1, scale=1.0)
    gamma = torch.full((8,), 0.5, dtype=torch.float32, device="cuda")
    dq, dk, dv, _ = la.chunk_bwd(q, k, v, dout, gamma, phi="identity", gate_kind="head")
    torch.cuda.synchronize()
    _check_bwd_suffix((q, k, v, dout), gamma, (dq, dk, dv), oracle.GATE_HEAD, channel_gate=False)
    del q, k, v, dout, dq, dk, dv
    torch.cuda.empty_cache()


def test_gated_backward_beyond_2_31_elements():
    from retention_gb300 import la
    gen = torch.Generator(device="cuda").manual_seed(35)
    q, k, v = _inputs(gen, 3)
    (dout,) = _inputs(gen, 1, scale=1.0)
    g = (torch.randn(1, 8, L_BIG, 128, generator=gen, device="cuda", dtype=torch.float32) - 8.0).to(torch.bfloat16)
    dq, dk, dv, dg = la.chunk_bwd(q, k, v, dout, g, phi="elu1", gate_kind="channel")
    torch.cuda.synchronize()
    _check_bwd_suffix((q, k, v, dout), g, (dq, dk, dv, dg), oracle.PHI_ELU1 | oracle.GATE_CHANNEL, channel_gate=True)
    del q, k, v, dout, g, dq, dk, dv, dg
    torch.cuda.empty_cache()
