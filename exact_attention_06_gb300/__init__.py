"""libfattn: exact fused attention forward and split-KV decode for GB300 (sm_103a).

The compute runs in the CUDA library ``libfattn.so`` built from ``csrc/``;
``fattn`` is its thin ctypes binding.  Importing this package loads nothing:
the library is opened on first use, and an error is raised if it is missing.
"""

__all__ = ["fattn", "inputs"]
