"""Exact softmax attention for one GB300 (sm_103a): a C-ABI CUDA library and its binding.

The package holds the CUDA sources (``csrc/``), the build script
(``build.py``), the ctypes binding (``_lib.py``), the seeded input generators
(``inputs.py``) and the named workloads (``workloads.py``).  Importing it does
not load the library; the first call does, and raises if it is not built.
"""

from ._lib import (ATTN_ERR_ALIGN, ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG, ATTN_ERR_SHAPE, ATTN_ERR_TIMEOUT,
                   ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_OK, LIB_PATH, MODS, OP_BWD, OP_DECODE,
                   OP_DECODE_CHUNK, OP_FWD,
                   SYMBOLS, AttnError, BlockMask, DenseMask, Shape, attn_bwd, attn_bwd_dkdv, attn_bwd_dq,
                   attn_bwd_preprocess, attn_decode, attn_decode_chunk, attn_fwd, create_block_mask, load, make_shape,
                   pack_dense_mask, poll_status, poll_status_all, status_string, workspace, workspace_size, UserScoreMod,
                   compile_score_mod, compile_mask_mod, flash_attention, causal_flash_attention)

__all__ = [
    "flash_attention", "causal_flash_attention", "attn_fwd", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_dkdv", "attn_bwd_dq", "attn_decode", "attn_decode_chunk",
    "create_block_mask", "BlockMask", "pack_dense_mask", "DenseMask", "compile_score_mod", "compile_mask_mod", "UserScoreMod",
    "workspace", "workspace_size",
    "poll_status", "poll_status_all", "status_string", "load", "AttnError", "Shape", "make_shape", "LIB_PATH", "SYMBOLS", "MODS",
    "OP_FWD", "OP_BWD", "OP_DECODE", "OP_DECODE_CHUNK", "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_SHAPE", "ATTN_ERR_ALIGN",
    "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT",
]
