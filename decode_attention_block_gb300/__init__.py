"""spark2_5 single-token decode attention block on NVIDIA GB300 (sm_103a).

The block runs in ``libspark_attn.so`` (hand-written CUDA kernels behind the C
ABI of ``include/spark_attn.h``); ``binding`` is its ctypes binding,
``synth`` the seeded synthetic inputs, ``build_lib`` the in-tree nvcc build.
"""

from . import build_lib  # noqa: F401

__all__ = ["build_lib", "binding", "synth"]
