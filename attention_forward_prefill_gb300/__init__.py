"""GB300-native fused attention forward (prefill + split-K decode).

The compute path is the CUDA library ``libfa_gb300.so`` built from ``csrc/``
for sm_103a; ``binding`` is a thin ctypes layer over its C ABI.  Importing this
package does not load the library -- the first call does, and it raises if the
library is missing (there is no CPU fallback).
"""
__all__ = ["binding", "inputs"]
