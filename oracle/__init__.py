"""fp64 CPU oracle for causal grouped-query attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never does, and the product
path fails loudly instead of falling back to it.
"""
from .oracle import (attn_fwd, attn_bwd, attn_bwd_dq_rows, attn_bwd_dkdv_rows,  # noqa: F401
                     attn_decode, rowdot, rope, build, num_threads, lib_path)
