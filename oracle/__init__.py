"""CPU oracle for the attention path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The CUDA path never does.
"""
from .attention import *  # noqa: F401,F403
from .attention import (BlockMask, attn_bwd, attn_decode, attn_fwd, attn_fwd_online,
                        attn_probs, build_block_mask, keep_matrix, visited_tiles)
