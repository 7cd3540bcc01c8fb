"""GB300-native NVFP4 training quantizer.

The compute path is the C-ABI library ``libnvfp4.so`` (hand-written sm_103a
CUDA kernels, declared in ``include/nvfp4.h``); ``tensor_quantization_gb300.nvfp4``
is its thin Python binding (argument marshalling only).  The library is loaded
on first use, and every call raises if it is missing: there is no fallback.
"""
__all__ = ["nvfp4", "workloads"]
