"""Seeded synthetic inputs for ubatch attention over a cell-indexed KV cache.

This package is the one place the CUDA path's tests / benchmark and the CPU
oracle meet: it produces batches (positions, sequence sets) and fp16 Q/K/V
rows from fixed seeds.  It holds none of the method's arithmetic: no
splitting, no cell assignment, no mask, no attention.

* ``gen``      seeded fp16 rows, indexed by (config, layer, content, kind, pos)
* ``configs``  the five workloads: model shapes, cache parameters and the
               decode calls (setup calls that fill the cache, then the
               measured calls)
"""

from . import gen, configs  # noqa: F401
