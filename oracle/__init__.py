"""fp64 CPU oracle for top-k sparse attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
may import this package.  The product library never calls it, and it shares
no code with the CUDA path.  See ``dsa_oracle.h`` for the definition and the
passages it follows.
"""

from .oracle import build, load, attn, pairs, rowhead, max_threads, topk, oproj, LIB_PATH  # noqa: F401
