"""ctypes binding of libpkv.so: the C ABI of include/pkv.h, under the same names.

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, passes raw pointers and sizes to the C entry point, and raises
:class:`PkvError` for a non-zero status.  No computation happens here and
there is no CPU fallback: if the shared library cannot be built or loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_WORKSPACE = 3
PKV_ERR_CUDA = 4
PKV_ERR_BAD_BLOCK_TABLE = 5
PKV_ERR_TIMEOUT = 6
PKV_ERR_OUT_OF_BLOCKS = 7

PKV_OUT_BF16 = 0
PKV_OUT_F32 = 1
PKV_FLAG_CHECKED = 0x1
PKV_FLAG_TEST_STALL = 0x2
PKV_FLAG_KV_FP8 = 0x4
PKV_FLAG_NO_EARLY_START = 0x8
PKV_FLAG_KV_BLOCK_SCALES = 0x10
PKV_FLAG_TILE_2D = 0x20
PKV_FLAG_ONE_TILE = 0x40
PKV_KV_BF16 = 0
PKV_KV_FP8_E4M3 = 1
PKV_KV_FP8_E4M3_BLOCK = 2
PKV_FLAG_GRID_SHIFT = 16


def PKV_FLAG_GRID(n: int) -> int:
    return (int(n) & 0xFFFF) << PKV_FLAG_GRID_SHIFT


class pkv_attn_params(ctypes.Structure):
    """The struct of include/pkv.h, field for field."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int), ("q_len", ctypes.c_int), ("n_q", ctypes.c_int),
        ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
        ("max_blocks_per_seq", ctypes.c_int), ("num_blocks", ctypes.c_int),
        ("scale", ctypes.c_float), ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("flags", ctypes.c_uint), ("window", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("kv_scales", ctypes.c_void_p),
    ]


# Every symbol include/pkv.h declares, with its ctypes signature.
_c_int, _c_float, _c_size = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_vp, _i32p = ctypes.c_void_p, ctypes.c_void_p
SIGNATURES = {
    "pkv_paged_decode_attn": ([_vp, _vp, _vp, _i32p, _i32p] + [_c_int] * 8 +
                              [_c_float, _vp, _c_int, _vp, _c_size, ctypes.c_uint, _vp], _c_int),
    "pkv_paged_decode_attn_ex": ([ctypes.POINTER(pkv_attn_params), _vp], _c_int),
    "pkv_paged_decode_attn_workspace_size": ([_c_int] * 7 + [ctypes.c_uint], _c_size),
    "pkv_paged_decode_attn_noalloc": ([_vp, _vp, _vp, _i32p, _i32p] + [_c_int] * 8 +
                                      [_c_float, _vp, _c_int, ctypes.c_uint, _vp], _c_int),
    "pkv_kv_append": ([_vp, _vp, _i32p] + [_c_int] * 5 + [_vp, _vp, ctypes.c_uint, _vp], _c_int),
    "pkv_kv_append_fp8": ([_vp, _vp, _i32p] + [_c_int] * 5 + [_vp] * 3 + [ctypes.c_uint, _vp],
                          _c_int),
    "pkv_kv_append_fp8_block": ([_vp, _vp, _i32p] + [_c_int] * 5 + [_vp] * 2 +
                                [ctypes.c_uint, _vp], _c_int),
    "pkv_check_error": ([_vp, _vp], _c_int),
    "pkv_copy_blocks": ([_vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, ctypes.c_uint,
                         _vp], _c_int),
    "pkv_pool_create": ([_c_int, _c_int], _vp),
    "pkv_pool_destroy": ([_vp], None),
    "pkv_pool_num_free": ([_vp], _c_int),
    "pkv_pool_refcount": ([_vp, _c_int], _c_int),
    "pkv_pool_alloc": ([_vp, _c_int, _vp], _c_int),
    "pkv_pool_share": ([_vp, _vp, _c_int], _c_int),
    "pkv_pool_release": ([_vp, _vp, _c_int], _c_int),
    "pkv_pool_append_slots": ([_vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp], _c_int),
    "pkv_kv_bytes": ([_c_int] * 4 + [ctypes.c_int64], ctypes.c_int64),
    "pkv_status_string": ([_c_int], ctypes.c_char_p),
    "pkv_version": ([], _c_int),
    "pkv_read_stream": ([_vp, _c_size, _vp, _c_int, _vp], _c_int),
}


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_name(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Load (building first if needed) the CUDA library; raises if that fails."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            lib_path = path or _build.build()
            lib = ctypes.CDLL(lib_path)
            for name, (argtypes, restype) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            if path is not None:
                return lib
            _lib = lib
        return _lib


def status_name(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != PKV_OK:
        raise PkvError(status, where)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _bf16_like(t, name):
    import torch
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must hold bf16 (torch.bfloat16 or a 16-bit view), got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _fp8_like(t, name):
    import torch
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must hold e4m3 codes (torch.uint8 or float8_e4m3fn), got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _scales_tensor(t, num_blocks, n_kv, name="kv_scales"):
    import torch
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or \
            tuple(t.shape) != (num_blocks, n_kv, 4):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape "
                         f"({num_blocks}, {n_kv}, 4)")


def _f32_vec(t, n, name):
    import torch
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or \
            tuple(t.shape) != (n,):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape ({n},)")


def _i32(t, name):
    import torch
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")


# ---------------------------------------------------------------------------
def pkv_kv_bytes(layers: int, n_kv: int, head_dim: int, elem_bytes: int, tokens: int) -> int:
    return int(load_library().pkv_kv_bytes(layers, n_kv, head_dim, elem_bytes, tokens))


def pkv_status_string(status: int) -> str:
    return status_name(status)


def pkv_version() -> int:
    return int(load_library().pkv_version())


def pkv_paged_decode_attn_workspace_size(num_seqs, q_len, n_q, n_kv, head_dim, block_size,
                                         max_context_len=0, flags=0) -> int:
    return int(load_library().pkv_paged_decode_attn_workspace_size(
        num_seqs, q_len, n_q, n_kv, head_dim, block_size, max_context_len, flags))


def alloc_workspace(num_seqs, q_len, n_q, n_kv, head_dim, block_size, flags=0, device=None):
    """A zero-filled uint8 CUDA tensor of the size the library asks for."""
    import torch
    n = pkv_paged_decode_attn_workspace_size(num_seqs, q_len, n_q, n_kv, head_dim, block_size,
                                             0, flags)
    if n == 0:
        raise PkvError(PKV_ERR_INVALID_ARG, "pkv_paged_decode_attn_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _attn_shapes(q, k_cache, v_cache, block_tables, context_lens, out, workspace, kv8=False):
    """Checks shared by the attention entry points; returns (dims, out_dtype).

    bf16: k_cache / v_cache [num_blocks, n_kv, bs, d]; 8-bit: k_cache is the
    interleaved cache [num_blocks, n_kv, 2, bs, d] and v_cache is None.
    """
    import torch
    _bf16_like(q, "q")
    _i32(block_tables, "block_tables")
    _i32(context_lens, "context_lens")
    if kv8:
        _fp8_like(k_cache, "kv_cache")
        if v_cache is not None or k_cache.dim() != 5 or k_cache.shape[2] != 2:
            raise ValueError("an 8-bit cache is one [num_blocks, n_kv, 2, bs, d] tensor")
        num_blocks, n_kv, _, bs, d2 = k_cache.shape
    else:
        _bf16_like(k_cache, "k_cache")
        _bf16_like(v_cache, "v_cache")
        if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
            raise ValueError("k_cache / v_cache must be 4-D of equal shape")
        num_blocks, n_kv, bs, d2 = k_cache.shape
    if q.dim() != 4:
        raise ValueError("q must be 4-D")
    num_seqs, q_len, n_q, d = q.shape
    if d2 != d or block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or \
            context_lens.shape != (num_seqs,) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("inconsistent shapes")
    if out.dtype == torch.float32:
        out_dtype = PKV_OUT_F32
    elif out.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        out_dtype = PKV_OUT_BF16
    else:
        raise TypeError("out must be bfloat16 or float32")
    if not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA tensor")
    if workspace is not None and not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    return (num_seqs, q_len, n_q, n_kv, d, bs, block_tables.shape[1], num_blocks), out_dtype


def pkv_paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                          flags=0, stream=None):
    """out <- paged decode attention (see include/pkv.h for the full contract).

    q [num_seqs, q_len, n_q, d] bf16; k_cache/v_cache [num_blocks, n_kv, bs, d]
    bf16; block_tables [num_seqs, max_blocks] int32; context_lens [num_seqs]
    int32; out like q, bf16 or float32; workspace a uint8 CUDA tensor.
    """
    (num_seqs, q_len, n_q, n_kv, d, bs, max_blocks, num_blocks), out_dtype = _attn_shapes(
        q, k_cache, v_cache, block_tables, context_lens, out, workspace)
    st = load_library().pkv_paged_decode_attn(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), num_seqs, q_len, n_q, n_kv, d, bs, max_blocks,
        num_blocks, float(scale), out.data_ptr(), out_dtype, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), int(flags), _stream_ptr(stream))
    _check(st, "pkv_paged_decode_attn")


def pkv_paged_decode_attn_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                             workspace, flags=0, stream=None, window=0, k_scale=None,
                             v_scale=None, kv_scales=None):
    """pkv_paged_decode_attn through the parameter struct.

    window > 0: sliding window of that many positions.  With k_scale / v_scale
    (float32 CUDA [n_kv]) the cache is 8-bit: k_cache is the interleaved
    e4m3 cache [num_blocks, n_kv, 2, bs, d] (uint8 or float8_e4m3fn) and
    v_cache is None.  With kv_scales (float32 CUDA [num_blocks, n_kv, 4]) the
    8-bit cache has one K and one V scale per (block, KV head) instead.
    """
    blk = kv_scales is not None
    kv8 = blk or k_scale is not None or v_scale is not None
    (num_seqs, q_len, n_q, n_kv, d, bs, max_blocks, num_blocks), out_dtype = _attn_shapes(
        q, k_cache, v_cache, block_tables, context_lens, out, workspace, kv8)
    if blk:
        if k_scale is not None or v_scale is not None:
            raise ValueError("pass either per-head scales or per-block scales, not both")
        _scales_tensor(kv_scales, num_blocks, n_kv)
    elif kv8:
        _f32_vec(k_scale, n_kv, "k_scale")
        _f32_vec(v_scale, n_kv, "v_scale")
    p = pkv_attn_params(
        q=q.data_ptr(), k_cache=k_cache.data_ptr(),
        v_cache=None if v_cache is None else v_cache.data_ptr(),
        block_tables=block_tables.data_ptr(), context_lens=context_lens.data_ptr(),
        num_seqs=num_seqs, q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs,
        max_blocks_per_seq=max_blocks, num_blocks=num_blocks, scale=float(scale),
        out=out.data_ptr(), out_dtype=out_dtype, workspace=workspace.data_ptr(),
        workspace_bytes=workspace.numel() * workspace.element_size(), flags=int(flags),
        window=int(window),
        kv_dtype=PKV_KV_FP8_E4M3_BLOCK if blk else PKV_KV_FP8_E4M3 if kv8 else PKV_KV_BF16,
        k_scale=k_scale.data_ptr() if kv8 and not blk else None,
        v_scale=v_scale.data_ptr() if kv8 and not blk else None,
        kv_scales=kv_scales.data_ptr() if blk else None)
    st = load_library().pkv_paged_decode_attn_ex(ctypes.byref(p), _stream_ptr(stream))
    _check(st, "pkv_paged_decode_attn_ex")


def pkv_paged_decode_attn_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                  flags=0, stream=None):
    """pkv_paged_decode_attn using the library's own fixed scratch (no workspace argument).

    For callers that cannot allocate device memory; see include/pkv.h for the
    24 MiB limit, the shared-scratch caveats and the first-call set-up.
    """
    (num_seqs, q_len, n_q, n_kv, d, bs, _, num_blocks), out_dtype = _attn_shapes(
        q, k_cache, v_cache, block_tables, context_lens, out, None)
    st = load_library().pkv_paged_decode_attn_noalloc(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), num_seqs, q_len, n_q, n_kv, d, bs, block_tables.shape[1],
        num_blocks, float(scale), out.data_ptr(), out_dtype, int(flags), _stream_ptr(stream))
    _check(st, "pkv_paged_decode_attn_noalloc")


def pkv_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, flags=0, stream=None):
    """Scatter k_new/v_new [T, n_kv, d] into their cache slots (bit copy)."""
    _bf16_like(k_new, "k_new")
    _bf16_like(v_new, "v_new")
    _bf16_like(k_cache, "k_cache")
    _bf16_like(v_cache, "v_cache")
    _i32(slot_mapping, "slot_mapping")
    T, n_kv, d = k_new.shape
    num_blocks, n_kv2, bs, d2 = k_cache.shape
    if v_new.shape != k_new.shape or n_kv2 != n_kv or d2 != d or slot_mapping.shape != (T,) \
            or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent shapes")
    st = load_library().pkv_kv_append(
        k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T, n_kv, d, bs, num_blocks,
        k_cache.data_ptr(), v_cache.data_ptr(), int(flags), _stream_ptr(stream))
    _check(st, "pkv_kv_append")


def pkv_kv_append_fp8(k_new, v_new, slot_mapping, kv_cache, k_scale, v_scale, flags=0,
                      stream=None):
    """Quantise k_new/v_new [T, n_kv, d] (bf16) via per-head scales into the interleaved
    e4m3 cache [num_blocks, n_kv, 2, bs, d]."""
    _bf16_like(k_new, "k_new")
    _bf16_like(v_new, "v_new")
    _fp8_like(kv_cache, "kv_cache")
    _i32(slot_mapping, "slot_mapping")
    T, n_kv, d = k_new.shape
    if kv_cache.dim() != 5 or kv_cache.shape[2] != 2:
        raise ValueError("kv_cache must be [num_blocks, n_kv, 2, bs, d]")
    num_blocks, n_kv2, _, bs, d2 = kv_cache.shape
    if v_new.shape != k_new.shape or n_kv2 != n_kv or d2 != d or slot_mapping.shape != (T,):
        raise ValueError("inconsistent shapes")
    _f32_vec(k_scale, n_kv, "k_scale")
    _f32_vec(v_scale, n_kv, "v_scale")
    st = load_library().pkv_kv_append_fp8(
        k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T, n_kv, d, bs, num_blocks,
        k_scale.data_ptr(), v_scale.data_ptr(), kv_cache.data_ptr(), int(flags),
        _stream_ptr(stream))
    _check(st, "pkv_kv_append_fp8")


def pkv_copy_blocks(k_cache, v_cache, pairs, flags=0, stream=None):
    """Copy whole blocks (all KV heads, K and V): block pairs[p,1] <- block pairs[p,0].

    bf16 caches, or the interleaved e4m3 cache [num_blocks, n_kv, 2, bs, d] as k_cache with
    v_cache None (PKV_FLAG_KV_FP8 is then set) or, for a cache with per-block scales, its
    float32 scale tensor [num_blocks, n_kv, 4] (copied with the blocks).
    """
    import torch
    kv8 = k_cache.dtype in (torch.uint8, torch.float8_e4m3fn)
    if kv8:
        _fp8_like(k_cache, "kv_cache")
        if k_cache.dim() != 5 or k_cache.shape[2] != 2:
            raise ValueError("an 8-bit cache is one [num_blocks, n_kv, 2, bs, d] tensor")
        flags = int(flags) | PKV_FLAG_KV_FP8
        if v_cache is not None:
            _scales_tensor(v_cache, k_cache.shape[0], k_cache.shape[1])
            flags |= PKV_FLAG_KV_BLOCK_SCALES
    else:
        _bf16_like(k_cache, "k_cache")
        _bf16_like(v_cache, "v_cache")
    if pairs.dtype != torch.int32 or not pairs.is_cuda or not pairs.is_contiguous() or \
            pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be a contiguous int32 CUDA tensor of shape [n, 2]")
    if kv8:
        num_blocks, n_kv, _, bs, d = k_cache.shape
    else:
        num_blocks, n_kv, bs, d = k_cache.shape
        if v_cache.shape != k_cache.shape:
            raise ValueError("inconsistent shapes")
    st = load_library().pkv_copy_blocks(k_cache.data_ptr(),
                                        None if v_cache is None else v_cache.data_ptr(),
                                        pairs.data_ptr(), pairs.shape[0], num_blocks, n_kv, d, bs,
                                        int(flags), _stream_ptr(stream))
    _check(st, "pkv_copy_blocks")


def pkv_kv_append_fp8_block(k_new, v_new, slot_mapping, kv_cache, kv_scales, flags=0,
                            stream=None):
    """Quantise k_new/v_new [T, n_kv, d] (bf16) into the interleaved e4m3 cache
    [num_blocks, n_kv, 2, bs, d], setting the per-(block, KV head) scales kv_scales
    (float32 [num_blocks, n_kv, 4]) from the data; see include/pkv.h for the rule."""
    _bf16_like(k_new, "k_new")
    _bf16_like(v_new, "v_new")
    _fp8_like(kv_cache, "kv_cache")
    _i32(slot_mapping, "slot_mapping")
    T, n_kv, d = k_new.shape
    if kv_cache.dim() != 5 or kv_cache.shape[2] != 2:
        raise ValueError("kv_cache must be [num_blocks, n_kv, 2, bs, d]")
    num_blocks, n_kv2, _, bs, d2 = kv_cache.shape
    if v_new.shape != k_new.shape or n_kv2 != n_kv or d2 != d or slot_mapping.shape != (T,):
        raise ValueError("inconsistent shapes")
    _scales_tensor(kv_scales, num_blocks, n_kv)
    st = load_library().pkv_kv_append_fp8_block(
        k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T, n_kv, d, bs, num_blocks,
        kv_cache.data_ptr(), kv_scales.data_ptr(), int(flags), _stream_ptr(stream))
    _check(st, "pkv_kv_append_fp8_block")


# ---- block pool (host memory only; numpy int32 arrays are passed by pointer)
def _i32_host(a):
    import numpy as np
    if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
        raise TypeError("expected a contiguous numpy int32 array")
    return a.ctypes.data


def pkv_pool_create(num_blocks: int, block_size: int):
    h = load_library().pkv_pool_create(num_blocks, block_size)
    if not h:
        raise PkvError(PKV_ERR_INVALID_ARG, "pkv_pool_create")
    return h


def pkv_pool_destroy(pool) -> None:
    load_library().pkv_pool_destroy(pool)


def pkv_pool_num_free(pool) -> int:
    return int(load_library().pkv_pool_num_free(pool))


def pkv_pool_refcount(pool, block: int) -> int:
    return int(load_library().pkv_pool_refcount(pool, block))


def pkv_pool_alloc(pool, n: int):
    import numpy as np
    out = np.zeros(max(n, 0), dtype=np.int32)
    _check(load_library().pkv_pool_alloc(pool, n, _i32_host(out)), "pkv_pool_alloc")
    return out


def pkv_pool_share(pool, blocks) -> None:
    _check(load_library().pkv_pool_share(pool, _i32_host(blocks), blocks.shape[0]),
           "pkv_pool_share")


def pkv_pool_release(pool, blocks) -> None:
    _check(load_library().pkv_pool_release(pool, _i32_host(blocks), blocks.shape[0]),
           "pkv_pool_release")


def pkv_pool_append_slots(pool, table, nblocks: int, ctx: int, n_new: int, block_size: int):
    """Reserve slots for n_new tokens (copy-on-write); returns (nblocks, slots, copy_pairs).

    table: numpy int32 row of max_blocks entries, updated in place.
    copy_pairs: numpy int32 [k, 2] of (shared source, fresh destination) blocks.
    """
    import numpy as np
    nb = ctypes.c_int(nblocks)
    npairs = ctypes.c_int(0)
    slots = np.zeros(max(n_new, 1), dtype=np.int32)
    pairs = np.zeros((n_new // block_size + 2) * 2, dtype=np.int32)
    st = load_library().pkv_pool_append_slots(
        pool, _i32_host(table), ctypes.addressof(nb), table.shape[0], ctx, n_new,
        _i32_host(slots), _i32_host(pairs), ctypes.addressof(npairs))
    _check(st, "pkv_pool_append_slots")
    return nb.value, slots[:n_new], pairs[: 2 * npairs.value].reshape(-1, 2)


class BlockPool:
    """Owning wrapper of a pkv_block_pool handle."""

    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.handle = pkv_pool_create(num_blocks, block_size)

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h:
            pkv_pool_destroy(h)

    def num_free(self):
        return pkv_pool_num_free(self.handle)

    def refcount(self, b):
        return pkv_pool_refcount(self.handle, b)

    def alloc(self, n):
        return pkv_pool_alloc(self.handle, n)

    def share(self, blocks):
        pkv_pool_share(self.handle, blocks)

    def release(self, blocks):
        pkv_pool_release(self.handle, blocks)

    def append_slots(self, table, nblocks, ctx, n_new):
        return pkv_pool_append_slots(self.handle, table, nblocks, ctx, n_new, self.block_size)


def pkv_read_stream(buf, sink, ctas_per_sm=2, stream=None) -> None:
    """Read all of `buf` (a contiguous CUDA tensor) once, XOR-folding it into `sink`
    (an int32 CUDA tensor of one element): a read-bandwidth probe and L2 evictor."""
    import torch
    if not buf.is_cuda or not buf.is_contiguous() or sink.dtype != torch.int32 or \
            not sink.is_cuda or sink.numel() < 1:
        raise ValueError("buf must be a contiguous CUDA tensor and sink an int32 CUDA tensor")
    nbytes = buf.numel() * buf.element_size()
    _check(load_library().pkv_read_stream(buf.data_ptr(), nbytes - nbytes % 16, sink.data_ptr(),
                                          int(ctas_per_sm), _stream_ptr(stream)),
           "pkv_read_stream")


def pkv_check_error(workspace, stream=None) -> int:
    """Synchronise and return (and clear) the workspace's device status as a pkv_status."""
    return int(load_library().pkv_check_error(workspace.data_ptr(), _stream_ptr(stream)))
