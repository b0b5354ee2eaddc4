"""Failure detection on the GPU without a fault: bounded waits that run out.

A test-only flag makes the attention kernel issue no loads, so every wait on
a shared-memory stage expires after about a second.  The kernel must wind
down on its own, the host must read PKV_ERR_TIMEOUT, and the next normal
call on the same context must be correct.
"""
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.workloads import make_custom
from tests.gpu_common import assert_close, oracle_after_append, out_to_host, run_attn, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (n_q, n_kv, q_len, head_dim, block_size, contexts): narrow, wide and TMEM
    # consumers, and the paired TMEM form (256-row units of a prefill chunk,
    # whose split units the unit-list merge combines)
    (8, 2, 1, 128, 16, [40, 300, 17]),
    (32, 2, 1, 128, 16, [64, 500]),
    (32, 1, 4, 128, 32, [90, 700, 33]),
    (32, 8, 64, 128, 16, [64, 100, 700]),
]


@pytest.mark.parametrize("case", CASES, ids=["narrow", "wide", "tmem", "paired"])
def test_expired_waits_are_reported_and_the_context_survives(oracle, case):
    import torch
    n_q, n_kv, q_len, d, bs, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=77)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    flags = pkv.PKV_FLAG_TEST_STALL | pkv.PKV_FLAG_GRID(4)
    ws = pkv.alloc_workspace(wl.num_seqs, q_len, n_q, n_kv, d, bs, flags=flags)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                              wl.scale, out, ws, flags=flags)
    assert pkv.pkv_check_error(ws) == pkv.PKV_ERR_TIMEOUT
    assert pkv.pkv_check_error(ws) == pkv.PKV_OK  # the report was cleared
    # the context is still usable and the next call is right
    _, _, ref = oracle_after_append(oracle, wl)
    assert_close(out_to_host(run_attn(dw, wl, "bf16")), ref, "bf16", "after a timed-out call")


def test_expired_waits_over_an_8bit_cache(oracle):
    """The same with an e4m3 cache and 128 rows per KV head (tensor-memory consumer
    with its f16-copy warps): every wait expires, the report arrives, the next call
    is right."""
    import torch
    from paged_kv_cache_256_gb300.device import fp8_to_device
    from paged_kv_cache_256_gb300.workloads import fp8_cache_for
    n_q, n_kv, q_len, d, bs, ctxs = 32, 1, 4, 128, 32, [90, 700, 33]
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=78)
    c8 = fp8_cache_for(wl)
    dw, d8 = to_device(wl), fp8_to_device(c8)
    pkv.pkv_kv_append_fp8(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache, d8.k_scale, d8.v_scale)
    kv = c8.kv_cache.copy()
    oracle.kv_append_fp8(wl.k_new, wl.v_new, wl.slot_mapping, kv, c8.k_scale, c8.v_scale,
                         block_size=bs)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.float32, device="cuda")

    def call(flags):
        ws = pkv.alloc_workspace(wl.num_seqs, q_len, n_q, n_kv, d, bs, flags=flags)
        pkv.pkv_paged_decode_attn_ex(dw.q, d8.kv_cache, None, dw.block_tables, dw.context_lens,
                                     wl.scale, out, ws, flags=flags, k_scale=d8.k_scale,
                                     v_scale=d8.v_scale)
        return pkv.pkv_check_error(ws)

    assert call(pkv.PKV_FLAG_TEST_STALL | pkv.PKV_FLAG_GRID(4)) == pkv.PKV_ERR_TIMEOUT
    assert call(0) == pkv.PKV_OK
    ref = oracle.paged_attn_fp8(wl.q, kv, c8.k_scale, c8.v_scale, wl.block_tables,
                                wl.context_lens, n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs,
                                scale=wl.scale)
    assert_close(out_to_host(out), ref, "f32", "8-bit cache after a timed-out call")

