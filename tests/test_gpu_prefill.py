"""Paged (chunked) prefill on the GPU against the oracle.

A call with many new tokens per sequence -- a whole prompt (q_len = ctx) or a
chunk of one appended to a cached prefix (q_len < ctx) -- has more than 128
query rows per KV head; they are processed in row tiles of 128, each tile
reading only the blocks its causal (and window) limits allow; over a bf16
cache with bf16 output two such tiles share each stage (256-row units),
unless PKV_FLAG_ONE_TILE or a smaller workspace keeps one.  Covered:
several tiles with a partial last one, every group size (MHA, GQA, MQA),
rows that see no key (ctx < q_len), windows, split units (forced CTA
counts), bf16 and fp32 output, bf16 and e4m3 caches, and the named
chunked-prefill workload at full size.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.device import fp8_to_device
from paged_kv_cache_256_gb300.workloads import fp8_cache_for, make_custom, make_workload

from .gpu_common import (assert_close, bf16_to_host_bits, oracle_after_append, out_to_host,
                         run_attn, to_device)

pytestmark = pytest.mark.gpu

CASES = [
    # head_dim, block_size, n_q, n_kv, q_len, context_lens          (tiles of 128 rows)
    (128, 16, 32, 8, 64, [64, 100, 1000, 79]),                      # GQA: 256 rows, 2 tiles
    (128, 16, 8, 8, 200, [200, 333, 1500]),                         # MHA: 200 rows, 128 + 72
    (64, 32, 32, 1, 9, [9, 40, 700]),                               # MQA: 288 rows, 3 tiles
    (128, 32, 64, 8, 50, [50, 77, 2000]),                           # G 8: 400 rows, 4 tiles
    (128, 16, 16, 2, 20, [20, 5, 300]),                             # ctx 5 < q_len: zero rows
    # groups that are not powers of two: tiles of whole tokens (126 rows), a
    # token's heads spread over tiles (256 = 2 x 128), one token per tile
    # (96), and tiles that split a token's heads (200: no single TMA box)
    (128, 16, 48, 8, 30, [30, 31, 400]),                            # G 6: 180 rows, 126 + 54
    (64, 16, 256, 1, 2, [2, 90, 600]),                              # G 256: 4 tiles of 128
    (128, 32, 96, 1, 3, [3, 64, 333]),                              # G 96: 3 tiles of one token
    (64, 32, 200, 1, 2, [2, 45, 500]),                              # G 200: 4 tiles, split tokens
]
FP8_CASES = CASES[:4] + CASES[5:]


def _setup(oracle, case, seed):
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=seed)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    kc, vc, _ = oracle_after_append(oracle, wl)
    assert np.array_equal(bf16_to_host_bits(dw.k_cache), kc)
    return wl, dw, kc, vc


def _run_ex(dw, wl, kind, flags=0, window=0, kv8=None):
    import torch
    dt = torch.bfloat16 if kind == "bf16" else torch.float32
    out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dt, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                             wl.block_size, flags=flags)
    kc, vc = (dw.k_cache, dw.v_cache) if kv8 is None else (kv8.kv_cache, None)
    pkv.pkv_paged_decode_attn_ex(dw.q, kc, vc, dw.block_tables, dw.context_lens, wl.scale, out,
                                 ws, flags=flags, window=window,
                                 k_scale=None if kv8 is None else kv8.k_scale,
                                 v_scale=None if kv8 is None else kv8.v_scale)
    st = pkv.pkv_check_error(ws)
    assert st == pkv.PKV_OK, pkv.pkv_status_string(st)
    return out


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
@pytest.mark.parametrize("grid", [0, 1, 7, 64])
def test_prefill_parity(oracle, case, grid):
    wl, dw, kc, vc = _setup(oracle, case, seed=501 + case[2] + case[4])
    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    for window in (0, 16, 100):
        ref = oracle.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens, n_q=wl.n_q,
                                n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
                                scale=wl.scale, window=window)
        # bf16 output over a bf16 cache takes two 128-row tiles per unit (the
        # paired form) where a KV head has more; PKV_FLAG_ONE_TILE keeps one.
        for kind, extra in (("bf16", 0), ("bf16", pkv.PKV_FLAG_ONE_TILE), ("f32", 0)):
            out = _run_ex(dw, wl, kind, flags | extra, window)
            assert_close(out_to_host(out), ref, kind,
                         f"{case} grid {grid} W {window} {kind} one_tile={bool(extra)}")


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
def test_prefill_fp8_parity(oracle, case):
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=601 + n_q)
    c8 = fp8_cache_for(wl)
    dw, d8 = to_device(wl), fp8_to_device(c8)
    pkv.pkv_kv_append_fp8(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache, d8.k_scale,
                          d8.v_scale)
    kv = c8.kv_cache.copy()
    oracle.kv_append_fp8(wl.k_new, wl.v_new, wl.slot_mapping, kv, c8.k_scale, c8.v_scale,
                         block_size=bs)
    assert np.array_equal(d8.kv_cache.cpu().numpy(), kv)
    for grid, window in ((0, 0), (7, 0), (0, 30)):
        ref = oracle.paged_attn_fp8(wl.q, kv, c8.k_scale, c8.v_scale, wl.block_tables,
                                    wl.context_lens, n_q=n_q, n_kv=n_kv, head_dim=d,
                                    block_size=bs, scale=wl.scale, window=window)
        flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
        for kind in ("bf16", "f32"):
            out = _run_ex(dw, wl, kind, flags, window, kv8=d8)
            assert_close(out_to_host(out), ref, kind, f"fp8 {case} grid {grid} W {window}")


def test_prefill_rows_match_decode_rows(oracle):
    """Row i of a prefill chunk equals a one-token decode call at its position."""
    import torch
    case = CASES[0]
    wl, dw, kc, vc = _setup(oracle, case, seed=777)
    full = out_to_host(_run_ex(dw, wl, "f32"))
    for i in (0, 31, 63):
        q1 = dw.q[:, i:i + 1].contiguous()
        ctx1 = (dw.context_lens - (wl.q_len - 1 - i)).contiguous()
        out1 = torch.empty(tuple(q1.shape), dtype=torch.float32, device="cuda")
        ws = pkv.alloc_workspace(wl.num_seqs, 1, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size)
        pkv.pkv_paged_decode_attn(q1, dw.k_cache, dw.v_cache, dw.block_tables, ctx1, wl.scale,
                                  out1, ws)
        assert pkv.pkv_check_error(ws) == pkv.PKV_OK
        np.testing.assert_allclose(out1.cpu().numpy()[:, 0], full[:, i], rtol=2e-4, atol=2e-4)


def test_named_chunked_prefill(oracle):
    import torch
    wl = make_workload("llama3_8b_chunked_prefill")
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    kc, vc, ref = oracle_after_append(oracle, wl)
    assert np.array_equal(bf16_to_host_bits(dw.k_cache), kc)
    for kind in ("bf16", "f32"):
        assert_close(out_to_host(run_attn(dw, wl, kind)), ref, kind, f"{wl.name}/{kind}")
    out = run_attn(dw, wl, "f32", flags=pkv.PKV_FLAG_GRID(300))
    assert_close(out_to_host(out), ref, "f32", f"{wl.name}/grid300")
    # bf16 output runs the paired form; its split units are combined by the
    # unit-list merge up to 256 CTAs and by the row-group merge beyond
    for grid in (256, 257, 2000):
        out = run_attn(dw, wl, "bf16", flags=pkv.PKV_FLAG_GRID(grid))
        assert_close(out_to_host(out), ref, "bf16", f"{wl.name}/bf16/grid{grid}")
    del dw
    torch.cuda.empty_cache()
