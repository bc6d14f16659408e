"""Shared-base, per-request LoRA projection on one GB300 (sm_103a).

    Y[t,:] = X[t,:] W^T + s_a (X[t,:] A_a^T) B_a^T   for rows of requests naming adapter a
    Y[t,:] = X[t,:] W^T                              for rows of requests naming none

The compute runs in the C-ABI library ``liblora_linear.so`` (hand-written sm_103a
kernels); this package is a thin ctypes binding around it. Importing the package does
not load the library; ``LoraLinear`` and ``plan`` do, and raise if it is missing.
"""
from .synth import WORKLOADS, Workload, make_inputs  # noqa: F401


def __getattr__(name):
    if name in ("LoraLinear", "plan", "LoraError", "validate", "w4_repack", "launch_shape", "host_chunks", "k_split"):
        from . import lora_linear as _ll
        return getattr(_ll, name)
    raise AttributeError(name)
