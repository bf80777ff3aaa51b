"""retention_gb300: causal linear attention, retention and gated linear
attention in chunkwise-parallel form, plus the recurrent decode step, as
hand-written CUDA for one GB300 (sm_103a) behind a C ABI (``include/la.h``).

``retention_gb300.la`` is the thin Python binding (argument marshalling over
torch CUDA tensors); ``retention_gb300.workloads`` draws the seeded synthetic
inputs. Importing the package loads nothing; the CUDA library is loaded on
first use of the binding and its absence is an error.
"""
__all__ = ["la", "workloads"]
