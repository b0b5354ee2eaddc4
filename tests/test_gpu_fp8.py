"""8-bit (e4m3) KV cache on the GPU against the oracle.

The quantising append is compared bit for bit with the oracle's (fp32
division, nearest e4m3 with ties to even, saturation at 448), including exact
ties, saturating and non-finite inputs.  Attention over an e4m3 cache with
per-KV-head scales is compared element by element with the oracle's fp64
attention over the dequantised values, within the same tolerances as the
bf16 cache: every consumer mode, split units (forced CTA counts), windows,
and the named workloads at full size.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.device import fp8_to_device
from paged_kv_cache_256_gb300.workloads import (CONFIGS, f32_to_bf16_bits, fp8_cache_for,
                                                make_custom, make_workload)

from .gpu_common import assert_close, out_to_host, to_device

pytestmark = pytest.mark.gpu


def _append_both(oracle, wl, c8, dw, d8):
    """Quantising append of the workload's new tokens on the GPU and in the oracle."""
    pkv.pkv_kv_append_fp8(dw.k_new, dw.v_new, dw.slot_mapping, d8.kv_cache, d8.k_scale,
                          d8.v_scale)
    kv = c8.kv_cache.copy()
    oracle.kv_append_fp8(wl.k_new, wl.v_new, wl.slot_mapping, kv, c8.k_scale, c8.v_scale,
                         block_size=wl.block_size)
    return kv


def _run(dw, d8, wl, kind, flags=0, window=0):
    import torch
    dt = torch.bfloat16 if kind == "bf16" else torch.float32
    out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dt, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                             wl.block_size, flags=flags)
    pkv.pkv_paged_decode_attn_ex(dw.q, d8.kv_cache, None, dw.block_tables, dw.context_lens,
                                 wl.scale, out, ws, flags=flags, window=window,
                                 k_scale=d8.k_scale, v_scale=d8.v_scale)
    st = pkv.pkv_check_error(ws)
    assert st == pkv.PKV_OK, pkv.pkv_status_string(st)
    return out


def _ref(oracle, wl, c8, kv, window=0):
    return oracle.paged_attn_fp8(wl.q, kv, c8.k_scale, c8.v_scale, wl.block_tables,
                                 wl.context_lens, n_q=wl.n_q, n_kv=wl.n_kv,
                                 head_dim=wl.head_dim, block_size=wl.block_size,
                                 scale=wl.scale, window=window)


def test_append_special_values_bit_exact(oracle):
    """Ties, saturation, infinities, NaN, zeros and subnormal quotients."""
    import torch
    n_kv, d, bs, pool = 2, 64, 16, 4
    specials = np.asarray(
        [1.0625, 1.1875, -1.0625, 0.9375, 2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11, 240.0, 448.0,
         460.0, 464.0, 480.0, 1e5, -1e5, np.inf, -np.inf, np.nan, 0.0, -0.0, 2.0 ** -7,
         5 * 2.0 ** -10, 17.0, 0.013671875, 1e-30], dtype=np.float32)
    rng = np.random.default_rng(5)
    T = 6
    x = rng.standard_normal((T, n_kv, d)).astype(np.float32) * 4
    x.reshape(-1)[: specials.size] = specials
    kn = f32_to_bf16_bits(x)
    kn.reshape(-1)[16] = 0x7FC0  # a plain bf16 NaN (the helper maps NaN to its poison pattern)
    vn = f32_to_bf16_bits(-x[::-1].copy())
    slots = np.asarray([3, 17, 40, -1, 63, 5], dtype=np.int32)
    kv8 = rng.integers(0, 256, (pool, n_kv, 2, bs, d), dtype=np.uint8)
    for ks, vs in ([1.0, 1.0], [0.25, 3.0]), ([0.0078125, 1.5], [1.0, 0.1]):
        ks, vs = np.asarray(ks, np.float32), np.asarray(vs, np.float32)
        ref = kv8.copy()
        oracle.kv_append_fp8(kn, vn, slots, ref, ks, vs, block_size=bs)
        g = torch.from_numpy(kv8).cuda()
        to16 = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        pkv.pkv_kv_append_fp8(to16(kn), to16(vn), torch.from_numpy(slots).cuda(), g,
                              torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda())
        got = g.cpu().numpy()
        bad = np.nonzero(got != ref)
        assert bad[0].size == 0, (bad, got[bad][:8], ref[bad][:8])


CASES = [
    # head_dim, block_size, n_q, n_kv, q_len, context_lens           (consumer)
    (128, 16, 32, 8, 1, [1, 15, 16, 17, 200, 1000, 3]),             # narrow
    (64, 32, 8, 8, 2, [2, 3, 64, 65, 129, 700]),                    # narrow, d 64, q_len 2
    (64, 16, 4, 2, 1, [17, 40, 1, 0, 16, 33]),                      # narrow, d 64, empty seq
    (128, 16, 16, 1, 3, [3, 100, 47, 1500]),                         # wide
    (128, 32, 64, 8, 2, [2, 70, 1030]),                              # wide
    (128, 16, 32, 1, 4, [4, 5, 31, 33, 500, 2000]),                  # wide, 128 rows
    (64, 32, 128, 1, 1, [31, 1, 999]),                               # wide, 128 rows, d 64
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
@pytest.mark.parametrize("grid", [0, 1, 7, 64])
def test_fp8_parity(oracle, case, grid):
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=401 + n_q + q_len + d)
    c8 = fp8_cache_for(wl)
    dw, d8 = to_device(wl), fp8_to_device(c8)
    kv = _append_both(oracle, wl, c8, dw, d8)
    assert np.array_equal(d8.kv_cache.cpu().numpy(), kv)
    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    for window in (0, 17):
        ref = _ref(oracle, wl, c8, kv, window)
        for kind in ("bf16", "f32"):
            out = _run(dw, d8, wl, kind, flags, window)
            assert_close(out_to_host(out), ref, kind, f"{case} grid {grid} W {window} {kind}")


@pytest.fixture(scope="module", params=list(CONFIGS))
def named8(request, oracle):
    import torch
    wl = make_workload(request.param)
    c8 = fp8_cache_for(wl)
    dw, d8 = to_device(wl), fp8_to_device(c8)
    kv = _append_both(oracle, wl, c8, dw, d8)
    torch.cuda.synchronize()
    ref = _ref(oracle, wl, c8, kv)
    yield wl, dw, d8, kv, ref
    del dw, d8
    torch.cuda.empty_cache()


def test_named_fp8_append_bit_exact(named8):
    wl, dw, d8, kv, _ = named8
    assert np.array_equal(d8.kv_cache.cpu().numpy(), kv)


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_named_fp8_attention(named8, kind):
    wl, dw, d8, _, ref = named8
    assert_close(out_to_host(_run(dw, d8, wl, kind)), ref, kind, f"{wl.name}/fp8/{kind}")


def test_named_fp8_split_points(named8):
    wl, dw, d8, _, ref = named8
    for grid in (7, 300):
        out = _run(dw, d8, wl, "f32", flags=pkv.PKV_FLAG_GRID(grid))
        assert_close(out_to_host(out), ref, "f32", f"{wl.name}/fp8/grid{grid}")


def test_fp8_copy_blocks_bit_exact():
    import torch
    rng = np.random.default_rng(9)
    kv8 = rng.integers(0, 256, (10, 2, 2, 16, 64), dtype=np.uint8)
    pairs = np.asarray([[1, 4], [7, 2], [3, 3], [0, 11]], dtype=np.int32)
    g = torch.from_numpy(kv8).cuda()
    pkv.pkv_copy_blocks(g, None, torch.from_numpy(pairs).cuda())
    want = kv8.copy()
    want[4], want[2] = kv8[1], kv8[7]
    assert np.array_equal(g.cpu().numpy(), want)
