"""Plain fp64 CPU oracle for speculative-decoding batched verification.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run it.  It shares no code with the CUDA path
(``speculative_decoding_verification_07_gb300/csrc``); the two meet only in the
seeded input generators, which hold none of the method's arithmetic.

Modules
  philox    Philox4x32-10 counter RNG and the uniform / exponential maps.
  sampling  temperature / top-p / greedy-limit transforms, the accept test,
            the residual and bonus exponential races, the per-request walk.
  kvcache   reference paged-KV cache manager (block free list, lookahead
            reserve, commit/rollback, prefix fork, release) and the contiguous
            write-pointer rollback.

Every function names the passage of the source pages it follows.  Where the
pages are silent the docstring says which reading was taken.
"""

from . import philox, sampling, kvcache  # noqa: F401
