"""GB300-native (sm_103a) Kimi Delta Attention core: chunked prefill and decode.

The computation lives in hand-written CUDA kernels behind the C ABI of
``include/kda.h`` (``_build/libkda.so``); ``kda`` is the thin Python binding,
``workloads`` the seeded synthetic inputs and ``build`` the nvcc build step.
"""
__all__ = ["kda", "workloads", "build"]
