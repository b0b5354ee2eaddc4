"""The no-allocation entry point agrees with the regular one and with the oracle.

pkv_paged_decode_attn_noalloc serves callers that cannot allocate device
memory (engine plugins whose step hook must not allocate, processes whose
device memory is pre-reserved by another pool, loops that must never reach
cudaMalloc/cudaFree); it keeps its split-K records in a fixed scratch array
owned by the library.  This file is collected last so that a run stopping at
the first failure has run everything else first.  It is self-contained: it
passes alone in a fresh process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300 import _lib
from paged_kv_cache_256_gb300.device import to_device
from paged_kv_cache_256_gb300.workloads import make_custom, make_workload

from .gpu_common import assert_close, oracle_after_append, out_to_host

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, wl, dw, out, flags=0):
    """One call through the C ABI, with no workspace argument."""
    out_dtype = pkv.PKV_OUT_F32 if out.dtype == torch.float32 else pkv.PKV_OUT_BF16
    return lib.pkv_paged_decode_attn_noalloc(
        dw.q.data_ptr(), dw.k_cache.data_ptr(), dw.v_cache.data_ptr(),
        dw.block_tables.data_ptr(), dw.context_lens.data_ptr(), wl.num_seqs, wl.q_len, wl.n_q,
        wl.n_kv, wl.head_dim, wl.block_size, wl.block_tables.shape[1], wl.num_blocks, wl.scale,
        out.data_ptr(), out_dtype, flags,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["llama3_8b_gqa", "mqa_spec_verify", "tiny"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_noalloc_matches_regular_entry_on_two_calls(name, dtype):
    """Same kernels on the same grid: the outputs are bit-identical, call after call."""
    lib = _lib.load_library()
    wl = make_workload(name)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)

    ref = torch.empty(tuple(dw.q.shape), dtype=dtype, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size)
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                              wl.scale, ref, ws)
    assert pkv.pkv_check_error(ws) == pkv.PKV_OK
    want = ref.view(torch.int32 if dtype == torch.float32 else torch.int16).cpu().numpy()

    for call in range(2):  # the second call reuses the scratch the first one left behind
        out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dtype, device="cuda")
        st = _call_noalloc(lib, wl, dw, out)
        assert st == pkv.PKV_OK, _lib.status_name(st)
        torch.cuda.synchronize()
        got = out.view(torch.int32 if dtype == torch.float32 else torch.int16).cpu().numpy()
        diff = int(np.count_nonzero(got != want))
        assert diff == 0, f"call {call}: {diff} elements differ from the regular entry point"


@pytest.mark.parametrize("n_q,n_kv,q_len", [(16, 2, 1), (32, 1, 4)], ids=["narrow", "tmem"])
def test_noalloc_many_ctas_then_few(oracle, n_q, n_kv, q_len):
    """A call split over many CTAs leaves records past the grid of the next, smaller call;
    both calls match the oracle."""
    lib = _lib.load_library()
    wl = make_custom(num_seqs=3, q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=128, block_size=16,
                     context_lens=[3000, 5003, 17], seed=77 + n_q)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    _, _, ref = oracle_after_append(oracle, wl)
    for grid in (150, 3):
        for dtype, kind in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
            out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dtype, device="cuda")
            st = _call_noalloc(lib, wl, dw, out, pkv.PKV_FLAG_GRID(grid))
            assert st == pkv.PKV_OK, _lib.status_name(st)
            torch.cuda.synchronize()
            assert_close(out_to_host(out), ref, kind, f"noalloc grid {grid} {kind}")


def test_noalloc_prefill_keeps_one_tile_when_the_paired_form_does_not_fit(oracle):
    """The named chunked prefill's paired form (two 128-row tiles per unit over a
    bf16 cache, bf16 output) needs ~40 MB of split records at one CTA per SM,
    more than the fixed scratch: the call keeps one tile per unit, bit-identical
    to the regular call with PKV_FLAG_ONE_TILE and within tolerance of the oracle."""
    lib = _lib.load_library()
    wl = make_workload("llama3_8b_chunked_prefill")
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    _, _, ref = oracle_after_append(oracle, wl)
    one = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")
    flags = pkv.PKV_FLAG_ONE_TILE
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size,
                             flags=flags)
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                              wl.scale, one, ws, flags=flags)
    assert pkv.pkv_check_error(ws) == pkv.PKV_OK
    got = torch.full(tuple(dw.q.shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = _call_noalloc(lib, wl, dw, got)
    assert st == pkv.PKV_OK, _lib.status_name(st)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), one.view(torch.int16))
    assert_close(out_to_host(got), ref, "bf16", "noalloc chunked prefill")


def test_noalloc_rejects_what_it_cannot_serve():
    lib = _lib.load_library()
    wl = make_workload("tiny")
    dw = to_device(wl)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [dw.q.data_ptr(), dw.k_cache.data_ptr(), dw.v_cache.data_ptr(),
            dw.block_tables.data_ptr(), dw.context_lens.data_ptr(), wl.num_seqs, wl.q_len,
            wl.n_q, wl.n_kv, wl.head_dim, wl.block_size, wl.block_tables.shape[1],
            wl.num_blocks, wl.scale, out.data_ptr(), 0]
    # Device-side reports (CHECKED mode, expired waits) would be unreadable here.
    assert lib.pkv_paged_decode_attn_noalloc(*args, pkv.PKV_FLAG_CHECKED, s) == \
        pkv.PKV_ERR_UNSUPPORTED
    assert lib.pkv_paged_decode_attn_noalloc(*args, pkv.PKV_FLAG_TEST_STALL, s) == \
        pkv.PKV_ERR_UNSUPPORTED
    # A forced CTA count whose split records exceed the fixed scratch.
    assert lib.pkv_paged_decode_attn_noalloc(*args, pkv.PKV_FLAG_GRID(60000), s) == \
        pkv.PKV_ERR_WORKSPACE
    # Bad shapes get the regular entry point's precise status.
    bad = list(args)
    bad[7], bad[8] = 6, 4  # n_q % n_kv != 0
    assert lib.pkv_paged_decode_attn_noalloc(*bad, 0, s) == pkv.PKV_ERR_INVALID_ARG
