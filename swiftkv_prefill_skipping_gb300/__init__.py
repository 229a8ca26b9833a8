"""SwiftKV prefill skipping on one NVIDIA GB300 (sm_103a).

``binding`` wraps the C ABI of ``libswiftkv.so`` (include/swiftkv.h);
``api`` (import it explicitly) is the torch-facing layer: device memory,
streams, paged caches. Importing the package does not touch the GPU or build
the library; the first call that needs it does.
"""
from . import binding, flops  # noqa: F401

__all__ = ["binding", "flops"]
