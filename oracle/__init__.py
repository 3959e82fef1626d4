"""CPU oracle for the CSA2 sparse-attention path over an FP4 global KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, calls or
links this code; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` use it.  It shares no code, table or constant
generator with the CUDA path (``fp4_kv_cache_rope_gb300/csrc``); the two meet
only in the seeded inputs of ``synth``.

It is written to be read against the pages it follows, in plain numpy:

* ``formats`` -- the E2M1 and E4M3 element formats, encoders written as
  "nearest representable value, ties to the even code, saturate at the largest
  finite value", decoders as the format formulas.
* ``csa2`` -- the five steps of the path: RoPE then FP4 quantisation of main-KV
  rows, lightning-indexer scores, top-k selection with the block pool,
  dequantisation, and one softmax over the selected rows and the SWA window.
* ``workload`` -- the reference results of one sequence of a seeded workload.
* ``cref`` -- the same definitions restated in plain C++ (``cref.cpp``, one
  thread per host core), pinned against ``csa2`` and ``formats``; the timed
  CPU baseline, and the oracle side of the exhaustive codec sweep.

Floating point is fp64 except where the method's fp32 arithmetic decides an
integer (the RoPE rotation, the FP4 scale and code choice): there the oracle
computes in fp32 with one rounding per operation, as the kernels do.

Parity status per function is listed in each docstring; every function is
pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py`` except where a
docstring says "parity unpinned".
"""
from . import formats, csa2  # noqa: F401
