#!/usr/bin/env python3
"""Benchmark of the chunkwise linear-attention forward on one GB300.

A step is one la_chunk_fwd over the linear-attention training-shape workload
(B=8, H=16, L=4096, d_k=d_v=128, bf16, phi = elu+1, normalised, A = 1,
chunk 64): every row of the path (feature map, masked intra-chunk QK^T.V,
inter-chunk state, normaliser, fp32 final state) runs in that one call.
``value`` is tokens/s (tokens = B * L per step, all heads included) with the
inputs resident in HBM; the inputs (402 MB) are larger than L2, so no flush is
needed between steps. ``e2e`` is the same metric through the same call with
host buffers, the host<->device copies inside the timed region. The JSON line
also carries the decode step (HBM GB/s over 1000 consecutive steps) and the
retention and gated workloads.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from retention_gb300 import workloads as W  # noqa: E402

METRIC = "chunk-fwd tokens/s & % roofline (B=8,H=16,L=4096,d=128 bf16); decode HBM GB/s"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def chunk_work(cfg):
    """Algorithmic bytes and flops of one la_chunk_fwd (per-(token, head)
    flops 2*C*dk + 2*C*dv + 2*dk*dv + 2*dk*dv; bytes: q, k, v (+g) read once,
    out written once, final state written once; with the RetNet epilogue the
    output gate is read once too)."""
    B, H, L, dk, dv, C = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"], cfg["chunk"]
    esz = 2 if cfg["dtype"] == "bf16" else 4
    n = B * H * L
    flops = n * (2 * C * dk + 2 * C * dv + 4 * dk * dv)
    inb = n * (2 * dk + dv) * esz + (n * dk * esz if cfg["gate"] == "channel" else 0)
    if "gn_eps" in cfg:
        inb += n * dv * esz
    outb = n * dv * esz
    stb = B * H * (dk * dv + (dk if cfg["normalize"] else 0)) * 4
    return inb + outb + stb, flops


def decode_work(cfg):
    """Bytes of one decode step: the fp32 state (and z) read and written,
    q, k, v read, out written."""
    B, H, dk, dv = cfg["B"], cfg["H"], cfg["dk"], cfg["dv"]
    st = B * H * (dk * dv + (dk if cfg["normalize"] else 0)) * 4
    tok = B * H * (2 * dk + 2 * dv) * 2
    return 2 * st + tok


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, srcs):
    """dram bytes per launch recorded by an ncu capture (profiles/traffic.json),
    or None when the kernel source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
        if rec and rec.get("source_hash") == source_hash(srcs):
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        # LA_DIST_BACKEND=gloo keeps the ranks on the CPU even where a GPU is visible
        backend = os.environ.get("LA_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU leg

def _host(t):
    return None if t is None else t.float().numpy()


def _oracle_mode(oracle, cfg):
    m = oracle.PHI_ELU1 if cfg["phi"] == "elu1" else 0
    if cfg["normalize"]:
        m |= oracle.NORMALIZE
    if cfg["gate"] == "head":
        m |= oracle.GATE_HEAD
    elif cfg["gate"] == "channel":
        m |= oracle.GATE_CHANNEL
    return m


def _cpu_line(value, unit, threads, seqs, desc):
    """A cpu_baseline object: the oracle's threads work on one (b, h) sequence
    each, so the cores it used are at most the sample's sequences."""
    return {"value": value, "unit": unit, "cores": min(threads, seqs), "kind": "oracle", "sample": desc}


def oracle_sample(sample_B=2):
    """The oracle, as it stands, on a bounded sample of the linear-attention
    workload: sample_B batch rows x all 16 heads x L = 4096. Returns
    (tokens/s, threads used, description)."""
    import oracle
    cfg = W.workload("la", B=sample_B)
    inp = W.chunk_inputs(cfg, 0)
    t0 = time.perf_counter()
    oracle.forward(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]), None, _oracle_mode(oracle, cfg))
    dt = time.perf_counter() - t0
    desc = "oracle (fp64 recurrent C, OpenMP over sequences) on B=%d of 8 batch rows, all 16 heads, L=4096" % sample_B
    return sample_B * cfg["L"] / dt, min(oracle.max_threads(), sample_B * cfg["H"]), desc


def oracle_baselines():
    """The oracle, as it stands, timed on a bounded sample of each further
    workload the benchmark reports, in that line's own unit (tokens/s: B * L
    tokens per step, all heads; decode: the GPU line's algorithmic bytes per
    step / time). Samples keep the workload's shapes and cut the batch, or
    the sequence length of the single long-context batch row."""
    import oracle
    thr = oracle.max_threads()
    res = {}

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    # retention and RetNet (retention + GroupNorm/swish epilogue): B=2 of 8
    for name in ("retention", "retnet"):
        cfg = W.workload(name, B=2)
        inp = W.chunk_inputs(cfg, 0)
        mode = _oracle_mode(oracle, cfg)
        args = (_host(inp["q"]), _host(inp["k"]), _host(inp["v"]), _host(inp["gate"]), mode)
        if name == "retnet":
            ep = W.epilogue_inputs(cfg, 0)

            def run():
                o, _ = oracle.forward(*args)
                oracle.group_norm_swish(o, _host(ep["og"]), _host(ep["weight"]), _host(ep["bias"]), cfg["gn_eps"])
        else:
            def run():
                oracle.forward(*args)
        dt = timed(run)
        res[name] = _cpu_line(cfg["B"] * cfg["L"] / dt, UNIT, thr, cfg["B"] * cfg["H"],
                              "oracle (fp64 recurrent C%s) on B=2 of 8 batch rows, 16 heads, L=4096"
                              % (" + fp64 GroupNorm/swish" if name == "retnet" else ""))
    # gated long context: the first 32768 of 131072 tokens, all 8 heads
    cfg = W.workload("gla", L=32768)
    inp = W.chunk_inputs(cfg, 0)
    dt = timed(lambda: oracle.forward(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]), _host(inp["gate"]),
                                      _oracle_mode(oracle, cfg)))
    res["gla"] = _cpu_line(cfg["B"] * cfg["L"] / dt, UNIT, thr, cfg["H"],
                           "oracle (fp64 recurrent C) on the first 32768 of 131072 tokens, 8 heads")
    # delta rule: B=2 of 8
    cfg = W.workload("delta", B=2)
    d = W.delta_inputs(cfg, 0)
    dt = timed(lambda: oracle.delta_forward(_host(d["q"]), _host(d["k"]), _host(d["v"]), _host(d["beta"])))
    res["delta"] = _cpu_line(cfg["B"] * cfg["L"] / dt, UNIT, thr, cfg["B"] * cfg["H"],
                             "oracle delta rule (fp64 recurrent C) on B=2 of 8 batch rows, 16 heads, L=4096")
    # backward: B=1 of 8 (retention, linear attention); gated: first 8192 tokens
    for name, over in (("retention", dict(B=1)), ("la", dict(B=1)), ("gla", dict(L=8192))):
        cfg = W.workload(name, **over)
        inp = W.chunk_inputs(cfg, 0)
        dout = W.bwd_inputs(cfg, 0)
        dt = timed(lambda: oracle.backward(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]), _host(dout),
                                           _host(inp["gate"]), _oracle_mode(oracle, cfg)))
        what = "B=1 of 8 batch rows, 16 heads, L=4096" if name != "gla" else "the first 8192 of 131072 tokens, 8 heads"
        res[name + "_bwd"] = _cpu_line(cfg["B"] * cfg["L"] / dt, UNIT, thr, cfg["B"] * cfg["H"],
                                       "oracle backward (fp64 chain rule on the recurrence, C) on " + what)
    # decode: one step of the full batch (256 sequences x 32 heads), fp64 state
    cfg = W.workload("decode")
    st = W.decode_state(cfg, 0).double().numpy()
    tok = W.decode_tokens(cfg, 0, 0)
    dt = timed(lambda: oracle.decode_step(_host(tok["q"]), _host(tok["k"]), _host(tok["v"]), st, None,
                                          oracle.PHI_ELU1 | oracle.NORMALIZE))
    del st
    res["decode"] = _cpu_line(decode_work(cfg) / dt / 1e9, "GB/s", thr, cfg["B"] * cfg["H"],
                              "oracle decode step (fp64 C) on the full batch, one step; GB/s of the GPU "
                              "line's algorithmic bytes (fp32 state read and written, tokens) per step time")
    return res


# ----------------------------------------------------------------- GPU legs

def time_calls(fn, steps, warmup, world):
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1) / 1000.0


def device_inputs(cfg, seed=0):
    """Same recipe as workloads.chunk_inputs, drawn on the device (timing
    only; parity tests draw on the host so the oracle reads the same values)."""
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    dt = W.TORCH_DTYPES[cfg["dtype"]]
    g = torch.Generator(device="cuda").manual_seed(seed)
    s = cfg["scale"]
    q = (torch.randn(B, H, L, dk, generator=g, device="cuda") * s).to(dt)
    k = (torch.randn(B, H, L, dk, generator=g, device="cuda") * s).to(dt)
    v = (torch.randn(B, H, L, dv, generator=g, device="cuda") * s).to(dt)
    gate = None
    if cfg["gate"] == "head":
        gate = W.retention_gammas(H, cfg.get("gamma_step", 0.25)).cuda()
    elif cfg["gate"] == "channel":
        gate = torch.randn(B, H, L, dk, generator=g, device="cuda").to(dt)
    return q, k, v, gate


def bench_chunk(name, steps, warmup, world, pk):
    from retention_gb300 import la
    cfg = W.workload(name)
    q, k, v, gate = device_inputs(cfg)
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    out = torch.empty(B, H, L, dv, dtype=q.dtype, device="cuda")
    st = torch.empty(B, H, la.state_block(dk, dv, cfg["normalize"]), dtype=torch.float32,
                     device="cuda")

    if "gn_eps" in cfg:
        # RetNet: the output epilogue swish(og) * GroupNorm_h(o) in the same call
        g = torch.Generator(device="cuda").manual_seed(1)
        og = torch.randn(B, H, L, dv, generator=g, device="cuda").to(q.dtype)
        gw = 1.0 + 0.1 * torch.randn(H, dv, generator=g, device="cuda")
        gb = 0.1 * torch.randn(H, dv, generator=g, device="cuda")

        def step():
            la.chunk_fwd_gn_swish(q, k, v, og, gate, gn_weight=gw, gn_bias=gb, gn_eps=cfg["gn_eps"],
                                  phi=cfg["phi"], normalize=cfg["normalize"], gate_kind=cfg["gate"],
                                  chunk=cfg["chunk"], out=out, final_state=st)
    else:
        def step():
            la.chunk_fwd(q, k, v, gate, phi=cfg["phi"], normalize=cfg["normalize"],
                         gate_kind=cfg["gate"], chunk=cfg["chunk"], out=out, final_state=st)

    n0 = la.kernel_launches()
    step()
    torch.cuda.synchronize()
    per_step_launches = la.kernel_launches() - n0
    n1 = la.kernel_launches()
    secs = time_calls(step, steps, warmup, world)
    launches = la.kernel_launches() - n1 - warmup * per_step_launches
    secs = max_over_ranks(secs, world)
    bytes_, flops = chunk_work(cfg)
    t = secs / steps
    t_roof = max(bytes_ / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    return {
        "cfg": cfg, "secs": secs, "ms_per_step": t * 1e3, "tokens_per_s": world * B * L / t,
        "launches": launches, "launches_per_step": per_step_launches,
        "gbs": bytes_ / t / 1e9, "tflops": flops / t / 1e12, "bytes": bytes_, "flops": flops,
        "roofline_frac": t_roof / t, "inputs": (q, k, v, gate, out, st),
    }


def bench_delta(steps, warmup, world, pk):
    """The delta rule (la_delta_fwd) on its workload. The default path works
    in chunks of 64 on the tensor cores (one kernel: T of the next chunk made
    beside the state recurrence); its roofline is HBM (read q, k, v, beta,
    write out and the final state once) against the chunked form's products
    (about 10.5 MFLOP per 64-token chunk and head). The recurrent kernel
    (LA_KERNEL_SIMT) is timed beside it against the FP32 FMA pipe: 6 d_k d_v
    flops per token and head, SMs x 128 lanes x 2 flops x 2070 MHz."""
    from retention_gb300 import la
    cfg = W.workload("delta")
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    g = torch.Generator(device="cuda").manual_seed(0)
    q = torch.randn(B, H, L, dk, generator=g, device="cuda")
    k = torch.randn(B, H, L, dk, generator=g, device="cuda")
    v = (torch.randn(B, H, L, dv, generator=g, device="cuda") * cfg["scale"]).bfloat16()
    beta = torch.sigmoid(torch.randn(B, H, L, generator=g, device="cuda")).bfloat16()
    q = (q / q.norm(dim=-1, keepdim=True)).bfloat16()
    k = (k / k.norm(dim=-1, keepdim=True)).bfloat16()
    out = torch.empty_like(v)
    st = torch.empty(B, H, dv * dk, device="cuda")
    res = {}
    for simt in (False, True):
        secs = max_over_ranks(time_calls(lambda: la.delta_fwd(q, k, v, beta, out=out, final_state=st, simt=simt),
                                         steps, warmup, world), world)
        res[simt] = secs / steps
    t, tr = res[False], res[True]
    n = B * H * L
    bytes_ = n * (2 * dk + 2 * dv + 1) * 2 + B * H * dk * dv * 4
    C = 64
    # per chunk: K K^T, Q K^T; K S0^T, Q S0^T, K^T Ut; T Vt, P Ut
    flops = n / C * (2 * 2 * C * C * dk + 3 * 2 * C * dk * dv + 2 * 2 * C * C * dv)
    t_roof = max(bytes_ / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    fma_peak = torch.cuda.get_device_properties(0).multi_processor_count * 128 * 2 * 2.07e9 / 1e12
    rflops = 6.0 * n * dk * dv
    return {"tokens_per_s": world * B * L / t, "ms_per_step": t * 1e3, "launches_per_step": 1,
            "roofline": {"bound": "hbm", "frac": t_roof / t, "algorithmic_bytes": bytes_,
                         "tensor_tflops": flops / t / 1e12},
            "recurrent": {"ms_per_step": tr * 1e3, "tflops": rflops / tr / 1e12,
                          "frac_of_fp32_fma": rflops / tr / 1e12 / fma_peak},
            "workload": "delta rule: B=8, H=16, L=4096, d=128 bf16, unit q/k, beta=sigmoid(N(0,1))"}


def bench_bwd(name, steps, warmup, world, pk):
    """la_chunk_bwd on a workload's shapes (dout ~ N(0,1)). Roofline: the
    gradients' HBM floor, reading q, k, v, dout (and g) and writing dq, dk, dv
    (and dg) once each, against the flops of a chunkwise backward (twice the
    forward's dense products)."""
    from retention_gb300 import la
    cfg = W.workload(name)
    q, k, v, gate = device_inputs(cfg)
    g = torch.Generator(device="cuda").manual_seed(2)
    d = torch.randn(v.shape, generator=g, device="cuda").to(v.dtype)
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    dq, dkk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty_like(q) if cfg["gate"] == "channel" else None

    def step():
        la.chunk_bwd(q, k, v, d, gate, phi=cfg["phi"], normalize=cfg["normalize"], gate_kind=cfg["gate"],
                     dq=dq, dk=dkk, dv=dvv, dgate=dg)

    n0 = la.kernel_launches()
    step()
    torch.cuda.synchronize()
    per_step = la.kernel_launches() - n0
    secs = max_over_ranks(time_calls(step, steps, warmup, world), world)
    t = secs / steps
    n = B * H * L
    esz = 2 if cfg["dtype"] == "bf16" else 4
    gated = cfg["gate"] == "channel"
    bytes_ = n * (4 * dk + 3 * dv + (2 * dk if gated else 0)) * esz  # read q, k, v, dout (g); write dq, dk, dv (dg)
    flops = 2 * n * (2 * cfg["chunk"] * dk + 2 * cfg["chunk"] * dv + 4 * dk * dv)
    t_roof = max(bytes_ / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    route = "CUDA-core sweeps" if (cfg["gate"] == "channel" and cfg["normalize"]) else "tensor-core forwards"
    return {"tokens_per_s": world * B * L / t, "ms_per_step": t * 1e3, "launches_per_step": per_step,
            "roofline_frac": t_roof / t, "route": route, "algorithmic_bytes": bytes_}


def bench_e2e(cfg, steps, warmup, world):
    """The same call with the inputs in pinned host memory: every step copies
    q, k, v to the device, runs la_chunk_fwd, and copies the output and final
    state back, all inside the timed region. Steps are pipelined the way a
    serving loop would run them: two device buffer sets and three streams
    (upload, compute, read-back), so step i+1's upload overlaps step i's
    compute and read-back."""
    from retention_gb300 import la
    gen = torch.Generator("cpu").manual_seed(1)
    B, H, L, dk, dv = cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"]
    dt = W.TORCH_DTYPES[cfg["dtype"]]
    hq = torch.empty(B, H, L, dk, dtype=dt).pin_memory()
    hk = torch.empty_like(hq).pin_memory()
    hv = torch.empty(B, H, L, dv, dtype=dt).pin_memory()
    for t in (hq, hk, hv):
        t.copy_((torch.randn(t.shape, generator=gen) * cfg["scale"]).to(dt))
    ho = torch.empty(B, H, L, dv, dtype=dt).pin_memory()
    blk = la.state_block(dk, dv, cfg["normalize"])
    hs = torch.empty(B, H, blk, dtype=torch.float32).pin_memory()
    dev = [dict(q=torch.empty_like(hq, device="cuda"), k=torch.empty_like(hk, device="cuda"),
                v=torch.empty_like(hv, device="cuda"), o=torch.empty_like(ho, device="cuda"),
                s=torch.empty_like(hs, device="cuda")) for _ in range(2)]
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in range(2)]
    run_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        cur = torch.cuda.current_stream()
        for st in (s_up, s_run, s_down):
            st.wait_stream(cur)
        for i in range(n):
            b, d = i % 2, dev[i % 2]
            with torch.cuda.stream(s_up):
                s_up.wait_event(run_done[b])      # step i-2 is done with these inputs
                d["q"].copy_(hq, non_blocking=True)
                d["k"].copy_(hk, non_blocking=True)
                d["v"].copy_(hv, non_blocking=True)
                up_done[b].record(s_up)
            with torch.cuda.stream(s_run):
                s_run.wait_event(up_done[b])
                s_run.wait_event(down_done[b])    # step i-2's results have left
                la.chunk_fwd(d["q"], d["k"], d["v"], None, phi=cfg["phi"], normalize=cfg["normalize"],
                             gate_kind=cfg["gate"], chunk=cfg["chunk"], out=d["o"], final_state=d["s"],
                             stream=s_run)
                run_done[b].record(s_run)
            with torch.cuda.stream(s_down):
                s_down.wait_event(run_done[b])
                ho.copy_(d["o"], non_blocking=True)
                hs.copy_(d["s"], non_blocking=True)
                down_done[b].record(s_down)
        cur.wait_stream(s_down)

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    secs = max_over_ranks(e0.elapsed_time(e1) / 1000.0, world)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hs.numel() * hs.element_size()
    return {"value": world * B * L * steps / secs, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": secs / steps * 1e3,
            "pipelined": "2 buffer sets, upload / compute / read-back streams"}


def bench_decode(steps_total, world, pk):
    from retention_gb300 import la
    cfg = W.workload("decode")
    B, H, dk, dv = cfg["B"], cfg["H"], cfg["dk"], cfg["dv"]
    g = torch.Generator(device="cuda").manual_seed(0)
    st = torch.randn(B, H, dk * dv + dk, generator=g, device="cuda") * cfg["state_std"]
    st[:, :, dk * dv:] = torch.rand(B, H, dk, generator=g, device="cuda")
    s = cfg["scale"]
    toks = [(torch.randn(steps_total, B, H, dk, generator=g, device="cuda") * s).to(torch.bfloat16)
            for _ in range(3)]
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    warm = 3
    for i in range(warm):
        la.decode_step(toks[0][i], toks[1][i], toks[2][i], st, phi="elu1", normalize=True, out=out)
    torch.cuda.synchronize()
    barrier(world)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n1 = la.kernel_launches()
    e0.record(stream)
    for i in range(steps_total):
        la.decode_step(toks[0][i], toks[1][i], toks[2][i], st, phi="elu1", normalize=True, out=out)
    e1.record(stream)
    torch.cuda.synchronize()
    secs = max_over_ranks(e0.elapsed_time(e1) / 1000.0, world)
    bytes_ = decode_work(cfg)
    t = secs / steps_total
    gbs = bytes_ / t / 1e9
    return {"steps": steps_total, "us_per_step": t * 1e6, "gbs": gbs,
            "bytes_per_step": bytes_, "frac_of_hbm": gbs / pk["hbm_gbs"],
            "launches": la.kernel_launches() - n1,
            "seq_tokens_per_s": world * B * steps_total / secs}


# ----------------------------------------------------------------- main

def reference_arm(args, warmup, sample_B=1):
    """W untimed and K timed oracle runs, each on a bounded sample of the
    workload (sample_B batch rows x 16 heads x 4096 tokens)."""
    cfg = W.workload("la")
    for _ in range(warmup):
        oracle_sample(sample_B)
    secs, cores, desc = 0.0, None, None
    for _ in range(args.steps):
        v, cores, desc = oracle_sample(sample_B)
        secs += sample_B * cfg["L"] / v          # the oracle call alone, not the input draw
    val = args.steps * sample_B * cfg["L"] / secs
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "la: B=8,H=16,L=4096,d_k=d_v=128, elu+1, normalised, A=1, "
                                   "chunk 64 (each step: a B=%d sample)" % sample_B},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the retention/retnet/gated/delta/backward lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--only", default=None,
                    choices=["la", "retention", "retnet", "gla", "delta", "retention_bwd", "la_bwd", "gla_bwd"],
                    help="time one workload alone and print its line (for profiling)")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    if args.impl == "reference":
        # The reference arm is the oracle itself, timed as it stands on the
        # host cores; under torchrun only rank 0 runs it.
        if int(os.environ.get("RANK", "0")) != 0:
            return
        reference_arm(args, warmup)
        return
    world, rank, local = dist_init()

    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        sys.exit(1)
    pk = peaks()
    from retention_gb300 import la
    la.load()
    if args.only:
        name = args.only
        if name == "delta":
            r = bench_delta(args.steps, warmup, world, pk)
        elif name.endswith("_bwd"):
            r = bench_bwd(name[:-4], args.steps, warmup, world, pk)
        else:
            r = bench_chunk(name, args.steps, warmup, world, pk)
            r = {key: r[key] for key in ("tokens_per_s", "ms_per_step", "gbs", "roofline_frac", "launches_per_step")}
        if rank == 0:
            print(json.dumps({"only": name, **r}), flush=True)
        return

    with Clocks(local) as clk:
        la_res = bench_chunk("la", args.steps, warmup, world, pk)
    clocks = clk.summary()
    cfg = la_res["cfg"]
    e2e = bench_e2e(cfg, max(8, args.steps // 2), 2, world)
    del la_res["inputs"]
    dec = bench_decode(args.decode_steps, world, pk)
    extra = {}
    if not args.no_extra:
        for name in ("retention", "retnet", "gla"):
            r = bench_chunk(name, max(5, args.steps // 2), warmup, world, pk)
            del r["inputs"]
            extra[name] = {"tokens_per_s": r["tokens_per_s"], "ms_per_step": r["ms_per_step"],
                           "gbs": r["gbs"], "roofline_frac": r["roofline_frac"],
                           "launches_per_step": r["launches_per_step"]}
            torch.cuda.empty_cache()
        extra["delta"] = bench_delta(max(3, args.steps // 4), 3, world, pk)
        torch.cuda.empty_cache()
        for name, st in (("retention", max(5, args.steps // 4)), ("la", 3), ("gla", 2)):
            extra[name + "_bwd"] = bench_bwd(name, st, 1 if name == "gla" else 3, world, pk)
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, cores, desc = oracle_sample(2)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
        # the oracle beside every other line too
        for name, base in oracle_baselines().items():
            if name == "decode":
                dec["cpu_baseline"] = base
            elif name in extra:
                extra[name]["cpu_baseline"] = base

    tc = la.chunk_fwd_path(cfg["B"], cfg["H"], cfg["L"], cfg["dk"], cfg["dv"],
                           la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"]), cfg["chunk"]) == 1
    kernel = "la_chunk_tc_kernel" if tc else "chunk_simt_kernel"
    srcs = (["retention_gb300/csrc/la_tc.cu", "retention_gb300/csrc/sm100.cuh"] if tc
            else ["retention_gb300/csrc/la_simt.cu"]) + ["retention_gb300/csrc/la_common.cuh"]
    t_kernel = la_res["secs"] / args.steps / max(1, la_res["launches_per_step"])
    achieved = la_res["bytes"] / t_kernel / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": traffic_for(kernel, srcs),
            "kernel": kernel, "peak_source": pk["source"],
            "algorithmic_bytes_per_launch": la_res["bytes"],
            "tensor": {"achieved_tflops": la_res["flops"] / t_kernel / 1e12,
                       "peak_tflops": pk["bf16_tflops"],
                       "frac": la_res["flops"] / t_kernel / 1e12 / pk["bf16_tflops"]},
            "roofline_time_frac": la_res["roofline_frac"]}
    if rank == 0:
        line = {
            "metric": METRIC, "value": la_res["tokens_per_s"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": la_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "la: B=8,H=16,L=4096,d_k=d_v=128 bf16, elu+1, normalised, "
                                   "A=1, chunk 64, fp32 state", "global_batch": cfg["B"] * world,
                       "seq_len": cfg["L"], "heads": cfg["H"], "parallelism": "replicas x%d" % world,
                       "l2": "inputs (402 MB) larger than L2; no flush"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": la_res["launches"], "clocks": clocks,
            "decode": {"metric": "decode HBM GB/s", "value": dec["gbs"], "unit": "GB/s",
                       "us_per_step": dec["us_per_step"], "steps": dec["steps"],
                       "frac": dec["frac_of_hbm"], "peak": pk["hbm_gbs"],
                       "bytes_per_step": dec["bytes_per_step"], "launches": dec["launches"],
                       "workload": "256 seqs x 32 heads, d=128, fp32 state, elu+1, normalised",
                       "cpu_baseline": dec.get("cpu_baseline")},
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
