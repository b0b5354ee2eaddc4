"""Shared pieces of the GPU parity tests: tolerances, runners, the oracle side."""
from __future__ import annotations

import numpy as np

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.device import bf16_to_host_bits, to_device
from paged_kv_cache_256_gb300.workloads import bf16_bits_to_f32

# Tolerances: element passes iff |gpu - ref| <= ATOL + RTOL * |ref|, with ref
# the fp64 oracle.  bf16 output: 1e-2 / 1e-2; fp32 output: 1e-4 / 1e-4.
TOL = {"bf16": (1e-2, 1e-2), "f32": (1e-4, 1e-4)}


def assert_close(got: np.ndarray, ref: np.ndarray, kind: str, what: str = ""):
    atol, rtol = TOL[kind]
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output ({np.sum(~np.isfinite(got))})"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.unravel_index(int(np.argmax(err - (atol + rtol * np.abs(ref)))), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance {kind}; "
            f"max abs err {err.max():.3e}; worst at {idx}: got {got[idx]!r} ref {ref[idx]!r}")
    return float(err.max())


def out_to_host(out) -> np.ndarray:
    import torch
    if out.dtype == torch.float32:
        return out.cpu().numpy().astype(np.float64)
    return bf16_bits_to_f32(bf16_to_host_bits(out)).astype(np.float64)


def run_attn(dw, wl, out_kind="bf16", flags=0, context_lens=None, ws=None):
    import torch
    dt = torch.bfloat16 if out_kind == "bf16" else torch.float32
    out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dt, device=dw.q.device)
    if ws is None:
        ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                                 wl.block_size, flags=flags)
    cl = dw.context_lens if context_lens is None else context_lens
    pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, cl, wl.scale,
                              out, ws, flags=flags)
    st = pkv.pkv_check_error(ws)
    assert st == pkv.PKV_OK, pkv.pkv_status_string(st)
    return out


def oracle_after_append(orc, wl):
    """Host copies of the caches with the new tokens appended, and the fp64 output."""
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    orc.kv_append(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=wl.block_size)
    ref = orc.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens, n_q=wl.n_q,
                         n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
                         scale=wl.scale)
    return kc, vc, ref


__all__ = ["TOL", "assert_close", "out_to_host", "run_attn", "oracle_after_append", "to_device",
           "bf16_to_host_bits"]
