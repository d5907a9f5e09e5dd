"""GB300 (sm_103a) chunked-prefill causal attention.

The compute path is the C-ABI library ``libvpp.so`` (hand-written CUDA for
sm_103a, declared in ``include/vpp.h``); ``chunked_prefill_causal_gb300.vpp``
is its thin ctypes binding.  There is no CPU fallback: every binding call
raises if the library or a CUDA device is missing.
"""

__all__ = ["vpp", "workloads"]
