"""Frame-aligned block-sparse attention forward for B300 (sm_103a).

    from block_sparse_video_row_b300 import bsattn     # ctypes binding of libbsattn.so
    from block_sparse_video_row_b300 import synth      # seeded synthetic workloads

The compute path is the CUDA library built from ``csrc/`` (see
``block_sparse_video_row_b300._build``); importing this package loads nothing.
"""

__all__ = ["bsattn", "synth"]
