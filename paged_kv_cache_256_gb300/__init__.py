"""Paged decode attention for one GB300 GPU (sm_103a).

The product is ``libpkv.so``, a C-ABI library of hand-written CUDA kernels
(declared in ``include/pkv.h``):

* ``pkv_kv_append``          -- write each step's new K/V into the paged cache;
* ``pkv_paged_decode_attn``  -- one decode step of attention over the paged
  cache, GQA/MQA groups sharing each KV tile, ragged contexts, long contexts
  split across CTAs and combined by a log-sum-exp merge.

This package holds the CUDA sources (``csrc/``), the in-tree build
(``build.py``), the ctypes binding under the C names (``_lib.py``) and the
seeded synthetic inputs (``workloads.py``).  PyTorch is used only for device
memory and streams.
"""
from ._lib import (  # noqa: F401
    PKV_ERR_BAD_BLOCK_TABLE, PKV_ERR_CUDA, PKV_ERR_INVALID_ARG, PKV_ERR_TIMEOUT,
    PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_FLAG_CHECKED, PKV_FLAG_GRID, PKV_FLAG_TEST_STALL, PKV_OK, PKV_OUT_BF16,
    PKV_ERR_OUT_OF_BLOCKS, PKV_OUT_F32, BlockPool, PkvError, alloc_workspace, load_library,
    PKV_FLAG_KV_FP8, PKV_FLAG_NO_EARLY_START, PKV_KV_BF16, PKV_KV_FP8_E4M3,
    PKV_FLAG_KV_BLOCK_SCALES, PKV_FLAG_TILE_2D, PKV_FLAG_ONE_TILE, PKV_KV_FP8_E4M3_BLOCK, pkv_kv_append_fp8_block,
    pkv_check_error, pkv_copy_blocks, pkv_kv_append, pkv_kv_append_fp8, pkv_pool_alloc, pkv_pool_append_slots,
    pkv_pool_create, pkv_pool_destroy, pkv_pool_num_free, pkv_pool_refcount, pkv_pool_release,
    pkv_pool_share,
    pkv_kv_bytes, pkv_paged_decode_attn, pkv_paged_decode_attn_ex, pkv_paged_decode_attn_noalloc,
    pkv_attn_params,
    pkv_paged_decode_attn_workspace_size,
    pkv_read_stream, pkv_status_string, pkv_version)
