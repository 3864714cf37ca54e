"""Quantised KV-cache append and decode attention for one GB300 GPU.

The product is the C-ABI library ``libkvq.so`` (``include/kvq.h``) built from
``csrc/`` by ``build.build()``; ``binding`` is its thin ctypes binding
(``binding.KVCache``). ``workloads`` holds the seeded synthetic inputs.
Nothing is imported eagerly, so the input generator can be used without the
library.
"""

__all__ = ["binding", "build", "workloads"]
