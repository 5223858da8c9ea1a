"""CPU oracle for the dual-flow decode step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, calls or links anything here, and nothing here
imports the product path.
"""

from .dualflow import (  # noqa: F401
    Oracle,
    bf16_rne,
    rmsnorm,
    silu,
    rope,
    attend,
    log_softmax,
    mixture,
    topk_desc,
)
