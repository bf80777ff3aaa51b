"""The library's scratch memory leaves the process's default memory pool
alone: the split chunk forward and the backward take their stream-ordered
scratch from a pool of the library's own (the chunked delta rule takes none). The default
pool's release threshold and reserved size are read through the CUDA driver
before and after those calls and must not change."""
import ctypes

import pytest
import torch

from retention_gb300 import la, workloads as W

pytestmark = pytest.mark.gpu

CU_MEMPOOL_ATTR_RELEASE_THRESHOLD = 4
CU_MEMPOOL_ATTR_RESERVED_MEM_CURRENT = 5


def _default_pool_attrs():
    cu = ctypes.CDLL("libcuda.so.1")
    dev = ctypes.c_int()
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    pool = ctypes.c_void_p()
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    out = []
    for attr in (CU_MEMPOOL_ATTR_RELEASE_THRESHOLD, CU_MEMPOOL_ATTR_RESERVED_MEM_CURRENT):
        val = ctypes.c_uint64()
        assert cu.cuMemPoolGetAttribute(pool, attr, ctypes.byref(val)) == 0
        out.append(val.value)
    return tuple(out)


def test_scratch_leaves_the_default_pool_unchanged():
    torch.cuda.synchronize()
    before = _default_pool_attrs()
    # split forward (8 sequences): segment states in scratch
    cfg = W.workload("gla", B=1, H=8, L=4096)
    x = {n: t.cuda() for n, t in W.chunk_inputs(cfg, 3).items() if t is not None}
    mode = la.mode_bits(cfg["phi"], cfg["normalize"], cfg["gate"])
    assert la.chunk_fwd_path(1, 8, 4096, 128, 128, mode, 64) == 1
    la.chunk_fwd(x["q"], x["k"], x["v"], x["gate"], phi="elu1", gate_kind="channel", chunk=64)
    # chunked delta rule: no scratch at all
    dcfg = W.workload("delta", B=1, H=4, L=512)
    d = {n: t.cuda() for n, t in W.delta_inputs(dcfg, 3).items()}
    la.delta_fwd(d["q"], d["k"], d["v"], d["beta"])
    # backward of a short batch: the split forwards' segment states in scratch
    rcfg = W.workload("retention", B=1, H=4, L=512)
    r = {n: t.cuda() for n, t in W.chunk_inputs(rcfg, 3).items() if t is not None}
    dout = torch.randn_like(r["v"])
    la.chunk_bwd(r["q"], r["k"], r["v"], dout, r["gate"], phi="identity", gate_kind="head")
    torch.cuda.synchronize()
    assert la.device_status() == 0
    assert _default_pool_attrs() == before


def test_split_forward_replays_from_a_cuda_graph():
    """The split forward takes its scratch from the library's pool with
    stream-ordered calls, so after one ordinary call (which creates the pool)
    it can be captured into a CUDA graph; the replay matches the oracle."""
    from parity import TOL, rel_err, run_oracle
    cfg = W.workload("gla", B=1, H=8, L=4096)
    inp = W.chunk_inputs(cfg, 3)
    x = {n: t.cuda() for n, t in inp.items() if t is not None}
    out = torch.empty(1, 8, 4096, 128, dtype=torch.bfloat16, device="cuda")
    st = torch.empty(1, 8, 128 * 128, device="cuda")

    def call():
        la.chunk_fwd(x["q"], x["k"], x["v"], x["gate"], phi="elu1", gate_kind="channel", chunk=64, out=out,
                     final_state=st)

    call()
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        call()
    out.fill_(float("nan"))
    st.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    ro, rs = run_oracle(inp, cfg)
    assert rel_err(out.float().cpu().numpy(), ro) <= TOL["bf16"]
    assert rel_err(st.cpu().numpy(), rs) <= TOL["bf16"]
    assert la.device_status() == 0
