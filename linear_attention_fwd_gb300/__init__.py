"""Kimi Delta Attention (KDA) forward for one GB300 (sm_103a).

The compute lives in ``libkda.so`` (C ABI declared in ``include/kda.h``);
``linear_attention_fwd_gb300.kda`` is its thin ctypes binding.  The library is
loaded lazily on the first call, so that ``inputs`` (the seeded workload
generators) can be imported on machines without the built library.
"""
__all__ = ["kda", "inputs"]
