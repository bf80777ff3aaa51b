"""Seeded synthetic inputs for the chunkwise forward and the decode step.

This module draws inputs and nothing else: it holds none of the method's
arithmetic, so both the CUDA path and the oracle can be fed from it. Every
tensor is drawn on the CPU from ``torch.Generator('cpu').manual_seed(seed)``
as float32 N(0,1) (or U(0,1)), in the order q, k, v, then the gate, then any
state; it is then scaled and rounded to the workload's dtype (round to
nearest even for bf16). The oracle reads those exact rounded values.

Workloads (shapes, feature map, normaliser, gate, chunk), as named:

* ``tiny``      B=1 H=1 L=64 d=16 fp32, N(0,1), elu+1, normalised, A=1, C=16
* ``la``        B=8 H=16 L=4096 d=128 bf16, N(0,1)/sqrt(128), elu+1,
                normalised, A=1, C=64
* ``retention`` same shapes, identity feature map, no normaliser,
                gamma_h = 1 - 2^(-5 - h/4), C=64
* ``gla``       B=1 H=8 L=131072 d=128 bf16, elu+1, no normaliser,
                g = bf16(N(0,1)) [B,H,L,d], C=64
* ``delta``     B=8 H=16 L=4096 d=128 bf16 for the delta rule: q, k rows
                of unit length, v N(0,1)/sqrt(128), beta = sigmoid(N(0,1))
                per token (``delta_inputs``)
* ``retnet``    the ``retention`` workload followed by the RetNet output
                epilogue: output gate og = bf16(N(0,1)) [B,H,L,d], GroupNorm
                weight N(1, 0.1^2) and bias N(0, 0.1^2) fp32 [H,d], eps 1e-5
                (``epilogue_inputs``)
* ``decode``    256 sequences x H=32, d=128; fp32 S ~ N(0, var 0.01),
                z ~ U(0,1); per step one bf16 token N(0,1)/sqrt(128) per
                sequence; elu+1, normalised; 1000 steps
"""
import math

import torch

WORKLOADS = {
    "tiny": dict(B=1, H=1, L=64, dk=16, dv=16, dtype="f32", phi="elu1",
                 normalize=True, gate=None, chunk=16, scale=1.0),
    "la": dict(B=8, H=16, L=4096, dk=128, dv=128, dtype="bf16", phi="elu1",
               normalize=True, gate=None, chunk=64, scale=1.0 / math.sqrt(128)),
    "retention": dict(B=8, H=16, L=4096, dk=128, dv=128, dtype="bf16", phi="identity",
                      normalize=False, gate="head", chunk=64, scale=1.0 / math.sqrt(128)),
    "gla": dict(B=1, H=8, L=131072, dk=128, dv=128, dtype="bf16", phi="elu1",
                normalize=False, gate="channel", chunk=64, scale=1.0 / math.sqrt(128)),
    "retnet": dict(B=8, H=16, L=4096, dk=128, dv=128, dtype="bf16", phi="identity",
                   normalize=False, gate="head", chunk=64, scale=1.0 / math.sqrt(128), gn_eps=1e-5),
    "delta": dict(B=8, H=16, L=4096, dk=128, dv=128, dtype="bf16", phi="identity",
                  normalize=False, gate=None, chunk=1, scale=1.0 / math.sqrt(128)),
    "decode": dict(B=256, H=32, dk=128, dv=128, dtype="bf16", phi="elu1",
                   normalize=True, gate=None, steps=1000, scale=1.0 / math.sqrt(128),
                   state_std=0.1),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def retention_gammas(H, step=0.25):
    """Multi-scale decays gamma_h = 1 - 2^(-5 - h*step), h = 0..H-1.
    step=1 is the learnllm m22 multi-scale rule; the retention workload uses
    step=1/4 so that 16 heads span the same range."""
    return torch.tensor([1.0 - 2.0 ** (-5.0 - h * step) for h in range(H)],
                        dtype=torch.float32)


def workload(name, **override):
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    return cfg


def chunk_inputs(cfg, seed=0):
    """q, k, v (and the gate) for a chunk-forward workload, on the CPU.

    Returns a dict with q, k [B,H,L,dk], v [B,H,L,dv] in the workload dtype,
    and ``gate``: None, gamma[H] float32, or g [B,H,L,dk] in the workload dtype.
    """
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    gen = torch.Generator("cpu").manual_seed(seed)
    s = cfg["scale"]
    q = (torch.randn(B, H, L, dk, generator=gen) * s).to(dt)
    k = (torch.randn(B, H, L, dk, generator=gen) * s).to(dt)
    v = (torch.randn(B, H, L, dv, generator=gen) * s).to(dt)
    gate = None
    if cfg["gate"] == "head":
        gate = retention_gammas(H, cfg.get("gamma_step", 0.25))
    elif cfg["gate"] == "channel":
        gate = torch.randn(B, H, L, dk, generator=gen).to(dt)
    return dict(q=q, k=k, v=v, gate=gate)


def decode_state(cfg, seed=0):
    """Initial decode state: S [B,H,dk,dv] ~ N(0, std^2) and, when normalised,
    z [B,H,dk] ~ U(0,1), both float32, packed per (b,h) as S then z.
    Returns the packed [B,H,blk] float32 tensor."""
    B, H, dk, dv = cfg["B"], cfg["H"], cfg["dk"], cfg["dv"]
    gen = torch.Generator("cpu").manual_seed(seed)
    S = torch.randn(B, H, dk * dv, generator=gen) * cfg["state_std"]
    if not cfg["normalize"]:
        return S.contiguous()
    z = torch.rand(B, H, dk, generator=gen)
    return torch.cat([S, z], dim=2).contiguous()


def decode_tokens(cfg, step, seed=0, batch=None):
    """One decode token per sequence for ``step``: q, k [B,H,dk], v [B,H,dv]
    (and g [B,H,dk] for the per-channel gate). Each (step, sequence) pair has
    its own generator, so any subset of sequences can be drawn on its own.
    ``batch`` selects the sequences (default: all B)."""
    H, dk, dv = cfg["H"], cfg["dk"], cfg["dv"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    s = cfg["scale"]
    seqs = range(cfg["B"]) if batch is None else batch
    qs, ks, vs, gs = [], [], [], []
    for b in seqs:
        gen = torch.Generator("cpu").manual_seed(
            (seed * 1_000_003 + step) * 1_048_576 + int(b) + 1)
        qs.append(torch.randn(H, dk, generator=gen) * s)
        ks.append(torch.randn(H, dk, generator=gen) * s)
        vs.append(torch.randn(H, dv, generator=gen) * s)
        if cfg["gate"] == "channel":
            gs.append(torch.randn(H, dk, generator=gen))
    out = dict(q=torch.stack(qs).to(dt), k=torch.stack(ks).to(dt), v=torch.stack(vs).to(dt),
               gate=None)
    if cfg["gate"] == "channel":
        out["gate"] = torch.stack(gs).to(dt)
    elif cfg["gate"] == "head":
        out["gate"] = retention_gammas(H, cfg.get("gamma_step", 0.25))
    return out


def delta_inputs(cfg, seed=0):
    """q, k, v and beta for the delta rule, on the CPU: q, k [B,H,L,dk] rows of
    unit length (the page normalises its keys), v [B,H,L,dv] N(0,1) scaled,
    beta [B,H,L] = sigmoid(N(0,1)); all in the workload dtype."""
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    dt = TORCH_DTYPES[cfg["dtype"]]
    gen = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, H, L, dk, generator=gen)
    k = torch.randn(B, H, L, dk, generator=gen)
    v = torch.randn(B, H, L, dv, generator=gen) * cfg["scale"]
    beta = torch.sigmoid(torch.randn(B, H, L, generator=gen))
    q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), beta=beta.to(dt))


def epilogue_inputs(cfg, seed=0):
    """The RetNet output epilogue's inputs, on the CPU, from a generator of
    their own (seed offset by 7919 from the chunk inputs' seed): the output
    gate og [B,H,L,dv] = N(0,1) in the workload dtype, then the GroupNorm
    weight [H,dv] ~ N(1, 0.1^2) and bias [H,dv] ~ N(0, 0.1^2), float32."""
    B, H, L, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dv"]
    gen = torch.Generator("cpu").manual_seed(seed + 7919)
    og = torch.randn(B, H, L, dv, generator=gen).to(TORCH_DTYPES[cfg["dtype"]])
    weight = 1.0 + 0.1 * torch.randn(H, dv, generator=gen)
    bias = 0.1 * torch.randn(H, dv, generator=gen)
    return dict(og=og, weight=weight, bias=bias)


def bwd_inputs(cfg, seed=0):
    """The output gradient for a backward workload, on the CPU, from a
    generator of its own (seed offset by 104729): dout [B,H,L,dv] = N(0,1) in
    the workload dtype."""
    B, H, L, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dv"]
    gen = torch.Generator("cpu").manual_seed(seed + 104729)
    return torch.randn(B, H, L, dv, generator=gen).to(TORCH_DTYPES[cfg["dtype"]])
