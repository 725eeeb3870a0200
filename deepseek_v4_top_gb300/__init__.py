"""GB300-native top-k sparse attention (DeepSeek-V4.1 dsv41_sparse_attention).

The product is the C-ABI library ``libdsa.so`` (include/dsa.h) with its
sm_103a kernels; ``dsa`` is its Python binding and ``inputs`` the seeded
synthetic workload generator.
"""

from . import inputs  # noqa: F401
