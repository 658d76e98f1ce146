"""GB300 (sm_103a) decode-step paged-KV attention.

Three hand-written CUDA stages behind the C ABI in include/pa.h, chained with
Programmatic Dependent Launch: the fused metadata update, the split-K paged-attention
producer and the log-sum-exp reducer.  ``binding`` is the ctypes binding (one Python
function per C entry point), ``runtime`` holds device buffers for a step, and
``synthetic`` draws seeded workloads.
"""

from . import synthetic  # noqa: F401

__all__ = ["binding", "runtime", "synthetic", "build"]
