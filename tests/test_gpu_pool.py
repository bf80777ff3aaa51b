"""The library's scratch memory leaves the process's default memory pool
alone: the split chunk forward, the chunked delta rule and the backward take
their stream-ordered scratch from a pool of the library's own. The default
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
    # chunked delta rule: W | U images in scratch
    dcfg = W.workload("delta", B=1, H=4, L=512)
    d = {n: t.cuda() for n, t in W.delta_inputs(dcfg, 3).items()}
    la.delta_fwd(d["q"], d["k"], d["v"], d["beta"])
    # backward: reversed copies and partial gradients in scratch
    rcfg = W.workload("retention", B=1, H=4, L=512)
    r = {n: t.cuda() for n, t in W.chunk_inputs(rcfg, 3).items() if t is not None}
    dout = torch.randn_like(r["v"])
    la.chunk_bwd(r["q"], r["k"], r["v"], dout, r["gate"], phi="identity", gate_kind="head")
    torch.cuda.synchronize()
    assert la.device_status() == 0
    assert _default_pool_attrs() == before
