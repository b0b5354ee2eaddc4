"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` leg may import this package.  The CUDA
library never links, loads or calls it, and it imports nothing from the CUDA
package.  ``pkv_oracle.c`` holds the arithmetic (fp64 over the exact bf16
input values); this module compiles it with gcc and marshals numpy arrays.

Functions (each follows the passage cited in ``pkv_oracle.c``):

* :func:`paged_attn`   -- softmax(q K^T * scale + causal_mask) V per query row,
  K/V gathered through the block table, GQA group map h -> h // (n_q/n_kv).
* :func:`attn_partial` -- (o, m, l) of one key range: the online-softmax state.
* :func:`lse_merge`    -- exact combination of partials.
* :func:`paged_attn_fp8` -- the same attention over an e4m3 cache with per-KV-head scales.
* :func:`paged_attn_fp8_block` -- the same with one scale per (block, KV head).
* :func:`kv_append`    -- bit copy of new K/V rows into their slots.
* :func:`kv_append_fp8` -- quantising append into an e4m3 cache.
* :func:`kv_append_fp8_block` -- quantising append that sets per-(block, KV head) scales.
* :func:`e4m3_encode`, :func:`e4m3_decode` -- the 8-bit float codec.
* :func:`copy_blocks`  -- whole-block copies (copy-on-write).
* :func:`kv_bytes`     -- M_kv = 2 L n_kv d_h (s b) p.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pkv_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libpkv_oracle.so")

_lock = threading.Lock()
_default = None


def compile_oracle(src: str = SOURCE, out: str = LIB_PATH, openmp: bool = True) -> str:
    """Compile the C oracle into a shared library with gcc (IEEE fp64, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o", out, src, "-lm"]
    if openmp:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                           capture_output=True, text=True)
            return out
        except subprocess.CalledProcessError:
            pass  # no OpenMP runtime on this host: build the serial oracle
    subprocess.run(base, check=True, capture_output=True, text=True)
    return out


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.lib_path = lib_path
        lib = ctypes.CDLL(lib_path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        c_int = ctypes.c_int
        lib.oracle_paged_attn.argtypes = [u16p, u16p, u16p, i32p, i32p] + [c_int] * 8 + \
            [ctypes.c_double, c_int, f64p]
        lib.oracle_paged_attn.restype = c_int
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_paged_attn_fp8.argtypes = [u16p, u8p, f32p, f32p, i32p, i32p] + \
            [c_int] * 8 + [ctypes.c_double, c_int, f64p]
        lib.oracle_paged_attn_fp8.restype = c_int
        lib.oracle_kv_append_fp8.argtypes = [u16p, u16p, i32p] + [c_int] * 5 + \
            [f32p, f32p, u8p]
        lib.oracle_kv_append_fp8.restype = c_int
        lib.oracle_paged_attn_fp8_block.argtypes = [u16p, u8p, f32p, i32p, i32p] + \
            [c_int] * 8 + [ctypes.c_double, c_int, f64p]
        lib.oracle_paged_attn_fp8_block.restype = c_int
        lib.oracle_kv_append_fp8_block.argtypes = [u16p, u16p, i32p] + [c_int] * 5 + [u8p, f32p]
        lib.oracle_kv_append_fp8_block.restype = c_int
        lib.oracle_e4m3_encode.argtypes = [f32p, ctypes.c_long, u8p]
        lib.oracle_e4m3_encode.restype = None
        lib.oracle_e4m3_decode.argtypes = [u8p, ctypes.c_long, f64p]
        lib.oracle_e4m3_decode.restype = None
        lib.oracle_attn_partial.argtypes = [u16p, u16p, u16p, i32p, i32p] + [c_int] * 8 + \
            [ctypes.c_double, c_int, c_int, f64p, f64p, f64p]
        lib.oracle_attn_partial.restype = c_int
        lib.oracle_lse_merge.argtypes = [c_int, ctypes.c_long, c_int, f64p, f64p, f64p, f64p]
        lib.oracle_lse_merge.restype = None
        lib.oracle_kv_append.argtypes = [u16p, u16p, i32p] + [c_int] * 5 + [u16p, u16p]
        lib.oracle_kv_append.restype = c_int
        lib.oracle_kv_bytes.argtypes = [c_int, c_int, c_int, c_int, ctypes.c_int64]
        lib.oracle_kv_bytes.restype = ctypes.c_int64
        lib.oracle_copy_blocks.argtypes = [i32p, c_int, c_int, c_int, c_int, c_int, u16p, u16p]
        lib.oracle_copy_blocks.restype = c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = c_int
        self._lib = lib

    # -- attention ---------------------------------------------------------
    def paged_attn(self, q, k_cache, v_cache, block_tables, context_lens, *, n_q, n_kv,
                   head_dim, block_size, scale, num_blocks=None, q_len=None, window=0):
        """fp64 output [num_seqs, q_len, n_q, head_dim]; raises on invalid tables.

        window: 0 for full causal attention, W > 0 to see only the last W positions.
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
        v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        if q_len is None:
            q_len = q.shape[1]
        if num_blocks is None:
            num_blocks = k_cache.shape[0]
        max_blocks = bt.shape[1] if bt.ndim == 2 else 0
        out = np.zeros((num_seqs, q_len, n_q, head_dim), dtype=np.float64)
        st = self._lib.oracle_paged_attn(
            _ptr(q, ctypes.c_uint16), _ptr(k_cache, ctypes.c_uint16),
            _ptr(v_cache, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(cl, ctypes.c_int32),
            num_seqs, q_len, n_q, n_kv, head_dim, block_size, max_blocks, num_blocks,
            float(scale), int(window), _ptr(out, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_paged_attn rejected its inputs (status {st})")
        return out

    def paged_attn_fp8(self, q, kv_cache, k_scale, v_scale, block_tables, context_lens,
                       *, n_q, n_kv, head_dim, block_size, scale, num_blocks=None, q_len=None,
                       window=0):
        """paged_attn over an e4m3 cache [num_blocks, n_kv, 2, block_size, head_dim] (uint8
        codes; K rows then V rows) with fp32 per-KV-head scales [n_kv]."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kv_cache = np.ascontiguousarray(kv_cache, dtype=np.uint8)
        assert kv_cache.ndim == 5 and kv_cache.shape[2] == 2
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        assert ks.shape == (n_kv,) and vs.shape == (n_kv,)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        q_len = q.shape[1] if q_len is None else q_len
        if num_blocks is None:
            num_blocks = kv_cache.shape[0]
        out = np.zeros((num_seqs, q_len, n_q, head_dim), dtype=np.float64)
        st = self._lib.oracle_paged_attn_fp8(
            _ptr(q, ctypes.c_uint16), _ptr(kv_cache, ctypes.c_uint8),
            _ptr(ks, ctypes.c_float), _ptr(vs, ctypes.c_float), _ptr(bt, ctypes.c_int32),
            _ptr(cl, ctypes.c_int32), num_seqs, q_len, n_q, n_kv, head_dim, block_size,
            bt.shape[1], num_blocks, float(scale), int(window), _ptr(out, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_paged_attn_fp8 rejected its inputs (status {st})")
        return out

    def paged_attn_fp8_block(self, q, kv_cache, kv_scales, block_tables, context_lens, *, n_q,
                             n_kv, head_dim, block_size, scale, num_blocks=None, q_len=None,
                             window=0):
        """paged_attn over an e4m3 cache [num_blocks, n_kv, 2, block_size, head_dim] whose
        scales are per (block, KV head): kv_scales fp32 [num_blocks, n_kv, 4] = (K scale,
        V scale, reserved, reserved)."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        kv_cache = np.ascontiguousarray(kv_cache, dtype=np.uint8)
        assert kv_cache.ndim == 5 and kv_cache.shape[2] == 2
        sc = np.ascontiguousarray(kv_scales, dtype=np.float32)
        assert sc.shape == (kv_cache.shape[0], n_kv, 4)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs = cl.shape[0]
        q_len = q.shape[1] if q_len is None else q_len
        if num_blocks is None:
            num_blocks = kv_cache.shape[0]
        out = np.zeros((num_seqs, q_len, n_q, head_dim), dtype=np.float64)
        st = self._lib.oracle_paged_attn_fp8_block(
            _ptr(q, ctypes.c_uint16), _ptr(kv_cache, ctypes.c_uint8), _ptr(sc, ctypes.c_float),
            _ptr(bt, ctypes.c_int32), _ptr(cl, ctypes.c_int32), num_seqs, q_len, n_q, n_kv,
            head_dim, block_size, bt.shape[1], num_blocks, float(scale), int(window),
            _ptr(out, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_paged_attn_fp8_block rejected its inputs (status {st})")
        return out

    def e4m3_encode(self, x):
        """fp32 values -> e4m3 codes (nearest, ties to even, saturating at 448)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        codes = np.zeros(x.shape, dtype=np.uint8)
        self._lib.oracle_e4m3_encode(_ptr(x, ctypes.c_float), x.size, _ptr(codes, ctypes.c_uint8))
        return codes

    def e4m3_decode(self, codes):
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        x = np.zeros(codes.shape, dtype=np.float64)
        self._lib.oracle_e4m3_decode(_ptr(codes, ctypes.c_uint8), codes.size,
                                     _ptr(x, ctypes.c_double))
        return x

    def attn_partial(self, q, k_cache, v_cache, block_tables, context_lens, *, n_q, n_kv,
                     head_dim, block_size, scale, t_begin, t_end, num_blocks=None):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
        v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        num_seqs, q_len = cl.shape[0], q.shape[1]
        if num_blocks is None:
            num_blocks = k_cache.shape[0]
        o = np.zeros((num_seqs, q_len, n_q, head_dim), dtype=np.float64)
        m = np.zeros((num_seqs, q_len, n_q), dtype=np.float64)
        l = np.zeros((num_seqs, q_len, n_q), dtype=np.float64)
        st = self._lib.oracle_attn_partial(
            _ptr(q, ctypes.c_uint16), _ptr(k_cache, ctypes.c_uint16),
            _ptr(v_cache, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(cl, ctypes.c_int32),
            num_seqs, q_len, n_q, n_kv, head_dim, block_size, bt.shape[1], num_blocks,
            float(scale), int(t_begin), int(t_end), _ptr(o, ctypes.c_double),
            _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double))
        if st != 0:
            raise ValueError(f"oracle_attn_partial rejected its inputs (status {st})")
        return o, m, l

    def lse_merge(self, o, m, l):
        """o [nsplit, rows..., d], m/l [nsplit, rows...] -> out [rows..., d]."""
        o = np.ascontiguousarray(o, dtype=np.float64)
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        nsplit, d = o.shape[0], o.shape[-1]
        rows = int(np.prod(o.shape[1:-1]))
        out = np.zeros(o.shape[1:], dtype=np.float64)
        self._lib.oracle_lse_merge(nsplit, rows, d, _ptr(o, ctypes.c_double),
                                   _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double),
                                   _ptr(out, ctypes.c_double))
        return out

    # -- cache write ------------------------------------------------------
    def kv_append(self, k_new, v_new, slot_mapping, k_cache, v_cache, *, block_size):
        """In-place scatter into k_cache / v_cache (numpy uint16 arrays)."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
        num_blocks, n_kv, bs, d = k_cache.shape
        assert bs == block_size
        st = self._lib.oracle_kv_append(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16), _ptr(sm, ctypes.c_int32),
            sm.shape[0], n_kv, d, block_size, num_blocks,
            _ptr(k_cache, ctypes.c_uint16), _ptr(v_cache, ctypes.c_uint16))
        if st != 0:
            raise ValueError(f"oracle_kv_append rejected its inputs (status {st})")

    def kv_append_fp8(self, k_new, v_new, slot_mapping, kv_cache, k_scale, v_scale, *,
                      block_size):
        """In-place quantising scatter into an e4m3 cache [num_blocks, n_kv, 2, bs, d] (uint8)."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        ks = np.ascontiguousarray(k_scale, dtype=np.float32)
        vs = np.ascontiguousarray(v_scale, dtype=np.float32)
        assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
        num_blocks, n_kv, two, bs, d = kv_cache.shape
        assert two == 2 and bs == block_size and ks.shape == (n_kv,) and vs.shape == (n_kv,)
        st = self._lib.oracle_kv_append_fp8(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16), _ptr(sm, ctypes.c_int32),
            sm.shape[0], n_kv, d, block_size, num_blocks, _ptr(ks, ctypes.c_float),
            _ptr(vs, ctypes.c_float), _ptr(kv_cache, ctypes.c_uint8))
        if st != 0:
            raise ValueError(f"oracle_kv_append_fp8 rejected its inputs (status {st})")

    def kv_append_fp8_block(self, k_new, v_new, slot_mapping, kv_cache, kv_scales, *,
                            block_size):
        """In-place quantising scatter into an e4m3 cache [num_blocks, n_kv, 2, bs, d] (uint8)
        with per-(block, KV head) scales kv_scales [num_blocks, n_kv, 4] (float32, updated)."""
        k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
        v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
        sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        assert kv_cache.flags.c_contiguous and kv_cache.dtype == np.uint8
        assert kv_scales.flags.c_contiguous and kv_scales.dtype == np.float32
        num_blocks, n_kv, two, bs, d = kv_cache.shape
        assert two == 2 and bs == block_size and kv_scales.shape == (num_blocks, n_kv, 4)
        st = self._lib.oracle_kv_append_fp8_block(
            _ptr(k_new, ctypes.c_uint16), _ptr(v_new, ctypes.c_uint16), _ptr(sm, ctypes.c_int32),
            sm.shape[0], n_kv, d, block_size, num_blocks, _ptr(kv_cache, ctypes.c_uint8),
            _ptr(kv_scales, ctypes.c_float))
        if st != 0:
            raise ValueError(f"oracle_kv_append_fp8_block rejected its inputs (status {st})")

    def copy_blocks(self, pairs, k_cache, v_cache):
        """In-place whole-block copies: block pairs[p, 1] <- block pairs[p, 0]."""
        pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        num_blocks, n_kv, bs, d = k_cache.shape
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        st = self._lib.oracle_copy_blocks(_ptr(pairs, ctypes.c_int32), pairs.shape[0], num_blocks,
                                          n_kv, d, bs, _ptr(k_cache, ctypes.c_uint16),
                                          _ptr(v_cache, ctypes.c_uint16))
        if st != 0:
            raise ValueError(f"oracle_copy_blocks rejected its inputs (status {st})")

    # -- sizes --------------------------------------------------------------
    def kv_bytes(self, layers, n_kv, head_dim, elem_bytes, tokens):
        return int(self._lib.oracle_kv_bytes(layers, n_kv, head_dim, elem_bytes, tokens))

    def num_threads(self):
        return int(self._lib.oracle_num_threads())


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            if (not os.path.exists(LIB_PATH)
                    or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE)):
                compile_oracle()
            _default = Oracle(LIB_PATH)
        return _default
