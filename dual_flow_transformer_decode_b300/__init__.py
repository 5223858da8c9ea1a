"""Dual-flow Transformer grouped decode step on one B300 (sm_103a).

The compute path is the C-ABI library ``libdf.so`` (hand-written CUDA); this
package holds its build script, the ctypes binding and a thin model wrapper
that allocates device memory with torch.
"""

__all__ = ["binding", "model", "build"]
