"""CPU oracle for ubatch attention over a cell-indexed KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only the tests, the smoke check and the benchmark's
CPU-baseline / reference arm use it.  It shares no code with the CUDA path
(no kernels, headers, helpers or table generators); the two meet only in the
seeded input generators of the ``workloads`` package.

The oracle is plain, slow and meant to be read against the pages it follows:

* "llama.cpp and the ubatch" (joelfernandes.org, 2026-08-14) -- below UBATCH;
* "Batch、Ubatch 与解码主循环" (jonathanding.github.io, llama.cpp source
  reading #4) -- below BATCH-ZH;
* "What does llama.cpp's KV cache actually look like in memory?"
  (joelfernandes.org, 2026-10-05) -- below KV-MEM;
* "Iteration-Level Batching: Reforming the Batch at Every Token"
  (mercemay.com) -- below ITER.

Every function cites the section it restates.  Floating point is float64
(inputs are exact fp16 values widened to float64).

Modules
-------
params     context-parameter clamps (n_batch / n_ubatch)
batch      batch validation and auto-fill, split_simple / split_equal /
           split_seq, the init_batch strategy choice, caller-side chunking
cells      per-stream cell state, first-fit slot finder (prepare), n_kv,
           sequence removal and sharing (seq_rm / seq_cp)
mask       the KQ mask rule (causal order, optional sliding window)
attention  float64 masked-softmax GQA attention and the K/V scatter
layout     cache sizes, strides, byte offsets, the fixed-batch duty cycle
session    the whole path for one cache (split, prepare, store, attention)
sched      the iteration-level batching loop (retire, admit, assemble)

Parity status: every function is pinned by a ``-m "not gpu"`` test against a
value the pages print, a closed form, a library routine, brute force or an
invariant, except the exact tie-breaks of split_equal / split_seq and the
first-fit slot policy, which the pages do not fix (they are pinned only by the
written reading and by invariants; see each function's docstring).  The
sliding-window term and the scheduler's policy details are readings of
passages that name them without defining them; they are pinned by closed forms,
brute force, the page's duty cycles and a hand-worked trace.
"""

from . import params, batch, cells, mask, attention, layout, session, sched  # noqa: F401
