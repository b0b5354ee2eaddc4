"""The no-allocation entry point agrees with the regular one.

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
from paged_kv_cache_256_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 1e-2, torch.float32: 1e-4}  # |a - b| <= tol + tol * |b|


def _call_noalloc(lib, wl, dw, out):
    """One call through the C ABI, with no workspace argument."""
    out_dtype = pkv.PKV_OUT_F32 if out.dtype == torch.float32 else pkv.PKV_OUT_BF16
    return lib.pkv_paged_decode_attn_noalloc(
        dw.q.data_ptr(), dw.k_cache.data_ptr(), dw.v_cache.data_ptr(),
        dw.block_tables.data_ptr(), dw.context_lens.data_ptr(), wl.num_seqs, wl.q_len, wl.n_q,
        wl.n_kv, wl.head_dim, wl.block_size, wl.block_tables.shape[1], wl.num_blocks, wl.scale,
        out.data_ptr(), out_dtype, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["llama3_8b_gqa", "mqa_spec_verify", "tiny"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_noalloc_matches_regular_entry_on_two_calls(name, dtype):
    lib = _lib.load_library()
    wl = make_workload(name)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)

    ref = torch.empty(tuple(dw.q.shape), dtype=dtype, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size)
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                              wl.scale, ref, ws)
    assert pkv.pkv_check_error(ws) == pkv.PKV_OK
    ref64 = ref.double().cpu().numpy()
    tol = TOL[dtype]

    for call in range(2):  # the second call reuses the scratch the first one left behind
        out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dtype, device="cuda")
        st = _call_noalloc(lib, wl, dw, out)
        assert st == pkv.PKV_OK, _lib.status_name(st)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        err = np.abs(got - ref64)
        assert np.all(err <= tol + tol * np.abs(ref64)), f"call {call}: max err {err.max():.3e}"


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
    # CHECKED mode's report would be unreadable here.
    assert lib.pkv_paged_decode_attn_noalloc(*args, pkv.PKV_FLAG_CHECKED, s) == \
        pkv.PKV_ERR_UNSUPPORTED
    # A forced CTA count whose split records exceed the fixed scratch.
    assert lib.pkv_paged_decode_attn_noalloc(*args, pkv.PKV_FLAG_GRID(60000), s) == \
        pkv.PKV_ERR_WORKSPACE
    # Bad shapes get the regular entry point's precise status.
    bad = list(args)
    bad[7], bad[8] = 6, 4  # n_q % n_kv != 0
    assert lib.pkv_paged_decode_attn_noalloc(*bad, 0, s) == pkv.PKV_ERR_INVALID_ARG
