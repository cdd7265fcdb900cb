"""GB300-native paged KV-cache decode attention.

The compute path is a C-ABI CUDA library (``include/pagedattn.h``) built for
sm_103a; this package holds its thin Python binding plus the host-side pieces
that feed it: the block manager, byte accounting and the seeded workloads.
"""
__all__ = ["block_manager", "workloads", "accounting"]
