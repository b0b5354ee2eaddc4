"""Sliding-window (local) attention on the GPU against the oracle.

A query at position pos sees positions pos - W + 1 .. pos (CS336 lecture-10
notes, Local attention & sparse variants).  Covered: every consumer mode
(rows <= 8, 8 < rows <= 64, rows > 64), windows that cut inside a block, on a
block edge, shorter than one block and longer than every context, split
units (forced CTA counts), fp32 and bf16 output, and that blocks before every
row's window are never read.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.workloads import make_custom

from .gpu_common import assert_close, bf16_to_host_bits, out_to_host, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # head_dim, block_size, n_q, n_kv, q_len, context_lens           (mode)
    (128, 16, 32, 8, 1, [1, 15, 16, 17, 200, 1000, 3]),             # narrow
    (64, 32, 8, 8, 2, [2, 3, 64, 65, 129, 700]),                    # narrow, q_len 2
    (128, 16, 16, 1, 3, [3, 100, 47, 1500]),                         # wide
    (128, 32, 64, 8, 2, [2, 70, 1030]),                              # wide
    (128, 16, 32, 1, 4, [4, 5, 31, 33, 500, 2000]),                  # tmem
    (64, 32, 128, 1, 1, [31, 1, 999]),                               # tmem
]
WINDOWS = [1, 2, 15, 16, 17, 100, 4096]


def _run_ex(dw, wl, kind, window, flags=0, block_tables=None):
    import torch
    dt = torch.bfloat16 if kind == "bf16" else torch.float32
    out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dt, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                             wl.block_size, flags=flags)
    bt = dw.block_tables if block_tables is None else block_tables
    pkv.pkv_paged_decode_attn_ex(dw.q, dw.k_cache, dw.v_cache, bt, dw.context_lens, wl.scale,
                                 out, ws, flags=flags, window=window)
    st = pkv.pkv_check_error(ws)
    assert st == pkv.PKV_OK, pkv.pkv_status_string(st)
    return out


def _setup(oracle, case, seed):
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=seed)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    oracle.kv_append(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=bs)
    return wl, dw, kc, vc


def _ref(oracle, wl, kc, vc, window):
    return oracle.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens, n_q=wl.n_q,
                             n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
                             scale=wl.scale, window=window)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
@pytest.mark.parametrize("grid", [0, 1, 7, 64])
def test_window_parity(oracle, case, grid):
    wl, dw, kc, vc = _setup(oracle, case, seed=301 + case[2] + case[4])
    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    for window in WINDOWS:
        ref = _ref(oracle, wl, kc, vc, window)
        for kind in ("bf16", "f32"):
            out = _run_ex(dw, wl, kind, window, flags)
            assert_close(out_to_host(out), ref, kind, f"{case} grid {grid} W {window} {kind}")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
def test_window_extremes_are_exact(oracle, case):
    """W = 0 and W >= every context equal the positional entry bit for bit; W = 1 is V.

    W = 1 leaves one key per row, whose weight is 1: exactly so on the mma.sync
    consumers (exponent (S - S_max) * scale), and to the rounding of S_max * scale
    on the tensor-memory consumer (>64 rows), which forms the exponent as one FMA
    S * scale - S_max * scale; its fp32 output is then V within 2^-20 relative
    (bf16 output: V exactly either way)."""
    import torch
    wl, dw, kc, vc = _setup(oracle, case, seed=311 + case[2])
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size)
    base = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                              wl.scale, base, ws)
    base = bf16_to_host_bits(base)
    wide = wl.block_tables.shape[1] * wl.block_size
    for window in (0, wide, wide + 1, 1 << 30):
        assert np.array_equal(bf16_to_host_bits(_run_ex(dw, wl, "bf16", window)), base), window
    G = wl.n_q // wl.n_kv
    for kind in ("bf16", "f32"):
        got = out_to_host(_run_ex(dw, wl, kind, 1))
        for b, ctx in enumerate(wl.context_lens):
            for i in range(wl.q_len):
                pos = ctx - wl.q_len + i
                if pos < 0:
                    assert not got[b, i].any()
                    continue
                blk = wl.block_tables[b, pos // wl.block_size]
                v = vc[blk, :, pos % wl.block_size]          # [n_kv, d] bf16 bits
                want = np.repeat(v[:, None], G, axis=1).reshape(wl.n_q, wl.head_dim)
                from paged_kv_cache_256_gb300.workloads import bf16_bits_to_f32
                vw = bf16_bits_to_f32(want).astype(np.float64)
                if kind == "f32" and G * wl.q_len > 64:
                    assert np.all(np.abs(got[b, i] - vw) <= 2.0 ** -20 * np.abs(vw)), (kind, b, i)
                else:
                    assert np.array_equal(got[b, i], vw), (kind, b, i)


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[4]], ids=["narrow", "wide", "tmem"])
def test_blocks_outside_every_window_are_not_read(oracle, case):
    """Table entries before the first block any row can see are made invalid;
    checked mode would report a read of one, and the output must not change."""
    import torch
    wl, dw, kc, vc = _setup(oracle, case, seed=321)
    for window in (1, 17, 100):
        ref = _ref(oracle, wl, kc, vc, window)
        bt = wl.block_tables.copy()
        skipped = 0
        for b, ctx in enumerate(wl.context_lens):
            lo = ctx - wl.q_len - window + 1
            first = lo // wl.block_size if lo > 0 else 0
            bt[b, :first] = wl.num_blocks + 7  # out of range: a read would be flagged
            skipped += first
        bad = torch.from_numpy(bt).cuda()
        for grid in (0, 5):
            flags = pkv.PKV_FLAG_CHECKED | (pkv.PKV_FLAG_GRID(grid) if grid else 0)
            out = _run_ex(dw, wl, "f32", window, flags, block_tables=bad)
            assert_close(out_to_host(out), ref, "f32", f"W {window} grid {grid}")
        assert window > 50 or skipped > 0
