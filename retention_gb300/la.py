"""Thin Python binding of ``include/la.h``: the same calls, argument
marshalling only (torch CUDA tensors in, data pointers and sizes out). Every
step of the computation runs in the CUDA library; if the library has not been
built, or there is no CUDA device, the calls raise instead of computing
anything another way.
"""
import contextlib
import ctypes
import os

import torch

from . import build as _build

# mode bits (include/la.h)
LA_PHI_IDENTITY = 0x0
LA_PHI_ELU1 = 0x1
LA_NORMALIZE = 0x2
LA_GATE_NONE = 0x0
LA_GATE_HEAD = 0x4
LA_GATE_CHANNEL = 0x8
LA_DTYPE_F32 = 0x10
LA_KERNEL_SIMT = 0x20
LA_REVERSE = 0x40

LA_OK = 0
STATUS = {0: "LA_OK", -1: "LA_ERR_INVALID_ARG", -2: "LA_ERR_UNSUPPORTED", -3: "LA_ERR_MISALIGNED",
          -4: "LA_ERR_CUDA", -5: "LA_ERR_TIMEOUT", -6: "LA_ERR_INTERNAL"}

# every function include/la.h declares, with its ctypes signature
_VP, _I = ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "la_chunk_fwd": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_decode_step": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP], _I),
    "la_chunk_fwd_noalloc": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_chunk_fwd_from_state": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_delta_fwd": ([_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_group_norm_swish": ([_VP, _VP, _VP, _VP, ctypes.c_float, _VP, _I, _I, _I, _I, _I, _VP], _I),
    "la_chunk_fwd_gn_swish": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_float, _VP, _VP,
                               _I, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_chunk_bwd": ([_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _VP], _I),
    "la_chunk_fwd_path": ([_I, _I, _I, _I, _I, _I, _I], _I),
    "la_status_string": ([_I], ctypes.c_char_p),
    "la_kernel_launches": ([], ctypes.c_ulonglong),
    "la_device_status": ([_VP], _I),
    "la_chunk_fwd_stall_test": ([_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, ctypes.c_longlong, _VP], _I),
}

_lib = None


class LAError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s returned %d (%s)" % (fn, status, STATUS.get(status, "?")))


def library_path():
    return _build.LIB


def _open(path):
    if not os.path.exists(path):
        raise RuntimeError("the CUDA library %s is not built; run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load():
    """Load the built library (building it is ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        _lib = _open(_build.LIB)
    return _lib


@contextlib.contextmanager
def library(path):
    """Route every call of this module to the library at ``path`` (e.g. the
    bounds-checking build ``build.LIB_DEBUG``) inside the ``with`` block."""
    global _lib
    saved = load()
    _lib = _open(path)
    try:
        yield _lib
    finally:
        _lib = saved


def mode_bits(phi="elu1", normalize=False, gate=None, dtype=torch.bfloat16, simt=False, reverse=False):
    m = LA_PHI_ELU1 if phi == "elu1" else LA_PHI_IDENTITY
    if normalize:
        m |= LA_NORMALIZE
    if gate == "head":
        m |= LA_GATE_HEAD
    elif gate == "channel":
        m |= LA_GATE_CHANNEL
    elif gate is not None:
        raise ValueError("gate must be None, 'head' or 'channel'")
    if dtype == torch.float32:
        m |= LA_DTYPE_F32
    elif dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bfloat16 or float32")
    if simt:
        m |= LA_KERNEL_SIMT
    if reverse:
        m |= LA_REVERSE
    return m


def _dev(t, name):
    if t is None:
        return None
    if not (isinstance(t, torch.Tensor) and t.is_cuda):
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def state_block(dk, dv, normalize):
    return dk * dv + (dk if normalize else 0)


def chunk_fwd(q, k, v, gate=None, *, phi="elu1", normalize=False, gate_kind=None, chunk=64,
              out=None, final_state=None, want_state=True, simt=False, stream=None, initial_state=None,
              reverse=False):
    """la_chunk_fwd over q, k [B,H,L,dk], v [B,H,L,dv]. Returns (out, final_state).
    With ``initial_state`` ([B,H,block] fp32) it is la_chunk_fwd_from_state: the
    sequences continue from that state instead of zero. ``reverse`` sets
    LA_REVERSE (the anti-causal form)."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty(B, H, state_block(dk, dv, normalize), dtype=torch.float32,
                                  device=q.device)
    mode = mode_bits(phi, normalize, gate_kind, q.dtype, simt, reverse)
    if initial_state is None:
        rc = load().la_chunk_fwd(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                                 _dev(out, "out"), _dev(final_state, "final_state"),
                                 B, H, L, dk, dv, mode, chunk, _stream(stream))
        if rc != LA_OK:
            raise LAError("la_chunk_fwd", rc)
    else:
        if initial_state.dtype != torch.float32:
            raise ValueError("initial_state must be float32")
        rc = load().la_chunk_fwd_from_state(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                                            _dev(initial_state, "initial_state"), _dev(out, "out"),
                                            _dev(final_state, "final_state"),
                                            B, H, L, dk, dv, mode, chunk, _stream(stream))
        if rc != LA_OK:
            raise LAError("la_chunk_fwd_from_state", rc)
    return out, final_state


def _gn_params(weight, bias, H, dv):
    for name, t in (("gn_weight", weight), ("gn_bias", bias)):
        if t is not None and (t.dtype != torch.float32 or t.numel() != H * dv):
            raise ValueError("%s must be float32 with H*dv elements" % name)
    return _dev(weight, "gn_weight"), _dev(bias, "gn_bias")


def chunk_fwd_gn_swish(q, k, v, ogate, gate=None, *, gn_weight=None, gn_bias=None, gn_eps=1e-5,
                       phi="elu1", normalize=False, gate_kind=None, chunk=64, out=None, final_state=None,
                       want_state=True, simt=False, stream=None, initial_state=None):
    """la_chunk_fwd_gn_swish: chunk_fwd whose output goes through the RetNet
    epilogue swish(ogate) * GroupNorm_h(o) (ogate [B,H,L,dv], q's dtype;
    gn_weight, gn_bias [H,dv] fp32 or None). Returns (out, final_state)."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty(B, H, state_block(dk, dv, normalize), dtype=torch.float32,
                                  device=q.device)
    if ogate.dtype != q.dtype or ogate.shape != out.shape:
        raise ValueError("ogate must have out's shape and q's dtype")
    if initial_state is not None and initial_state.dtype != torch.float32:
        raise ValueError("initial_state must be float32")
    w, b = _gn_params(gn_weight, gn_bias, H, dv)
    mode = mode_bits(phi, normalize, gate_kind, q.dtype, simt)
    rc = load().la_chunk_fwd_gn_swish(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                                      _dev(initial_state, "initial_state"), _dev(ogate, "ogate"), w, b,
                                      float(gn_eps), _dev(out, "out"), _dev(final_state, "final_state"),
                                      B, H, L, dk, dv, mode, chunk, _stream(stream))
    if rc != LA_OK:
        raise LAError("la_chunk_fwd_gn_swish", rc)
    return out, final_state


def group_norm_swish(x, ogate, *, gn_weight=None, gn_bias=None, gn_eps=1e-5, out=None, stream=None):
    """la_group_norm_swish over x [B,H,L,dv] (or [B,H,dv], a decode output):
    swish(ogate) * GroupNorm_h(x). ``out`` may be ``x``."""
    shape = x.shape
    if x.dim() == 3:
        B, H, dv = shape
        L = 1
    else:
        B, H, L, dv = shape
    if out is None:
        out = torch.empty_like(x)
    if ogate.dtype != x.dtype or ogate.shape != shape or out.shape != shape or out.dtype != x.dtype:
        raise ValueError("x, ogate and out must share shape and dtype")
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("x must be bfloat16 or float32")
    w, b = _gn_params(gn_weight, gn_bias, H, dv)
    mode = LA_DTYPE_F32 if x.dtype == torch.float32 else 0
    rc = load().la_group_norm_swish(_dev(x, "x"), _dev(ogate, "ogate"), w, b, float(gn_eps), _dev(out, "out"),
                                    B, H, L, dv, mode, _stream(stream))
    if rc != LA_OK:
        raise LAError("la_group_norm_swish", rc)
    return out


def chunk_bwd(q, k, v, dout, gate=None, *, phi="elu1", normalize=False, gate_kind=None,
              dq=None, dk=None, dv=None, dgate=None, want_dgate=True, simt=False, stream=None):
    """la_chunk_bwd: gradients of chunk_fwd (from a zero state) given dout.
    Returns (dq, dk, dv, dgate); dgate is None unless gate_kind == "channel".
    ``simt`` forces the CUDA-core sweeps."""
    B, H, L, d_k = q.shape
    d_v = v.shape[-1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if gate_kind == "channel" and want_dgate and dgate is None:
        dgate = torch.empty_like(q)
    if gate_kind != "channel":
        dgate = None
    mode = mode_bits(phi, normalize, gate_kind, q.dtype, simt)
    rc = load().la_chunk_bwd(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"), _dev(dout, "dout"), _dev(dq, "dq"), _dev(dk, "dk"), _dev(dv, "dv"),
                             _dev(dgate, "dgate"), B, H, L, d_k, d_v, mode, _stream(stream))
    if rc != LA_OK:
        raise LAError("la_chunk_bwd", rc)
    return dq, dk, dv, dgate


def chunk_fwd_noalloc(q, k, v, gate=None, *, phi="elu1", normalize=False, gate_kind=None, chunk=64,
                      out, final_state=None, simt=False, stream=None):
    """la_chunk_fwd_noalloc: like chunk_fwd, but the caller provides ``out`` (and
    ``final_state``) and the library allocates nothing; any scratch it needs is
    the library's fixed device array, shared by all calls on the device."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    mode = mode_bits(phi, normalize, gate_kind, q.dtype, simt)
    rc = load().la_chunk_fwd_noalloc(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                                     _dev(out, "out"), _dev(final_state, "final_state"),
                                     B, H, L, dk, dv, mode, chunk, _stream(stream))
    if rc != LA_OK:
        raise LAError("la_chunk_fwd_noalloc", rc)
    return out, final_state


def decode_step(q, k, v, state, gate=None, *, phi="elu1", normalize=False, gate_kind=None,
                out=None, stream=None):
    """la_decode_step: q, k [B,H,dk], v [B,H,dv]; ``state`` [B,H,block] fp32 updated in place."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    mode = mode_bits(phi, normalize, gate_kind, q.dtype)
    rc = load().la_decode_step(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                               _dev(state, "state"), _dev(out, "out"), B, H, dk, dv, mode,
                               _stream(stream))
    if rc != LA_OK:
        raise LAError("la_decode_step", rc)
    return out


def delta_fwd(q, k, v, beta, *, out=None, final_state=None, want_state=True, simt=False, stream=None):
    """la_delta_fwd: the delta rule over q, k [B,H,L,dk], v [B,H,L,dv], beta
    [B,H,L] (keys as given: normalise them first). Returns (out, final_state
    [B,H,dv*dk] fp32, rows = value dimensions)."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    if final_state is None and want_state:
        final_state = torch.empty(B, H, dv * dk, dtype=torch.float32, device=q.device)
    if beta.dtype != q.dtype or not beta.is_contiguous():
        raise ValueError("beta must be contiguous and of q's dtype")
    mode = (LA_DTYPE_F32 if q.dtype == torch.float32 else 0) | (LA_KERNEL_SIMT if simt else 0)
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("q, k, v must be bfloat16 or float32")
    rc = load().la_delta_fwd(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(beta, "beta"),
                             _dev(out, "out"), _dev(final_state, "final_state"),
                             B, H, L, dk, dv, mode, _stream(stream))
    if rc != LA_OK:
        raise LAError("la_delta_fwd", rc)
    return out, final_state


def chunk_fwd_path(B, H, L, dk, dv, mode, chunk):
    """1 = tensor-core kernel, 0 = general kernel, < 0 = rejected (la_status)."""
    return int(load().la_chunk_fwd_path(B, H, L, dk, dv, mode, chunk))


def kernel_launches():
    return int(load().la_kernel_launches())


def device_status(stream=None):
    """Wait for `stream` (default: torch's current stream) and return the
    la_status of the library's bounded device-side waits since the last call:
    0, or -5 (LA_ERR_TIMEOUT) if a kernel gave one up. Clears the flags."""
    return int(load().la_device_status(_stream(stream)))


def chunk_fwd_stall_test(q, k, v, gate=None, *, phi="elu1", normalize=False, gate_kind=None, stall_chunk=1,
                         wait_ns=20_000_000, out=None, stream=None):
    """la_chunk_fwd_stall_test: the tensor-core forward with its producer
    stopping before chunk ``stall_chunk`` and every bounded wait limited to
    ``wait_ns``; afterwards la_device_status reports LA_ERR_TIMEOUT. Returns
    ``out`` (not valid)."""
    B, H, L, dk = q.shape
    if out is None:
        out = torch.empty(B, H, L, v.shape[-1], dtype=q.dtype, device=q.device)
    mode = mode_bits(phi, normalize, gate_kind, q.dtype)
    rc = load().la_chunk_fwd_stall_test(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(gate, "gate"),
                                        _dev(out, "out"), B, H, L, mode, int(stall_chunk), int(wait_ns),
                                        _stream(stream))
    if rc != LA_OK:
        raise LAError("la_chunk_fwd_stall_test", rc)
    return out
