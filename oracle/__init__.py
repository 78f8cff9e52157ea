"""CPU oracle for decode attention over a block-quantized, paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 restatement
of what the CUDA library computes.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library never calls
it and shares no code with it (the only common module is the seeded input
generator ``workloads``, which holds none of the method's arithmetic).

What it follows:

* The KV formats are the ones the memra-bench card names in its
  "drafts/kf4/ - archived experiment" section: K in q8_0 or fp8, V in q5_1,
  q4_0 or fp8, default q8_0/q5_1.  The per-block rules are the library's
  stated definitions of those formats (``quant.py``).
* Attention is the plain definition softmax(q K^T / sqrt(D)) V on the
  dequantized cache, with grouped query heads and the causal rule of
  speculative verify (the memra README, "Speculative decoding" item of the
  serving surface: MTP drafts are verified as K+1 query rows).
* The pool byte layout (``layout.py``) is this library's own ABI; the pages
  define none.

Pins (the checks that tie each function to something other than itself) are
listed in each module's docstring and live in ``tests/test_oracle_*.py``.
"""
from . import quant, layout, attention  # noqa: F401
