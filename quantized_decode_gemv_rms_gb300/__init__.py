"""GB300-native (sm_103a) quantized decode GEMV with fused RMSNorm -> Q8_0.

The compute path is the CUDA library ``_lib/libqdg.so`` (sources in
``csrc/``, C ABI in ``include/qdg.h``); ``qdg`` is its Python binding.
"""
from . import workloads, synth  # noqa: F401  (no arithmetic; safe without a GPU)

__all__ = ["qdg", "workloads", "synth"]
