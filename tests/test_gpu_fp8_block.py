"""8-bit (e4m3) KV cache with one scale per (block, KV head), on the GPU against the oracle.

The quantising append that sets the block scales is compared bit for bit
(codes and scales) with the oracle's, call after call: fresh blocks, blocks
that grow (their resident rows re-quantised), blocks written again from
offset 0, all-zero and non-finite values, skipped slots inside a run, a
duplicated slot.  Attention over such caches is compared element by element
with the oracle's fp64 attention over the dequantised values, within the
tolerances of the bf16 cache: every consumer mode, split units (forced CTA
counts), windows, caches filled by the append and caches with arbitrary
(non power-of-two) block scales, and the named workloads at full size.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.workloads import (CONFIGS, E4M3_POISON, f32_to_bf16_bits,
                                                fp8_cache_for, make_custom, make_workload)

from .gpu_common import assert_close, out_to_host, to_device

pytestmark = pytest.mark.gpu


def _bf16_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _history(wl, split=0.5):
    """The resident tokens before the step's new ones (positions [0, ctx - q_len) of each
    sequence), as two append calls: the first `split` of every prefix, then the rest.  Each
    call is (k_rows, v_rows, slots), sequence by sequence, positions in order; the rows are
    the bf16 values the workload placed in those slots."""
    calls = [([], [], []), ([], [], [])]
    bs = wl.block_size
    for b in range(wl.num_seqs):
        n = max(0, int(wl.context_lens[b]) - wl.q_len)
        cut = int(n * split)
        for t in range(n):
            blk, off = int(wl.block_tables[b, t // bs]), t % bs
            c = calls[0 if t < cut else 1]
            c[0].append(wl.k_cache[blk, :, off, :])
            c[1].append(wl.v_cache[blk, :, off, :])
            c[2].append(blk * bs + off)
    out = []
    for k, v, s in calls:
        if s:
            out.append((np.stack(k), np.stack(v), np.asarray(s, dtype=np.int32)))
    return out


class BlockCache:
    """An 8-bit cache with per-block scales, on the GPU and in host memory side by side."""

    def __init__(self, wl, seed=0):
        import torch
        rng = np.random.default_rng(seed)
        shape = (wl.num_blocks, wl.n_kv, 2, wl.block_size, wl.head_dim)
        self.kv = np.full(shape, E4M3_POISON, dtype=np.uint8)
        # stale entries: a fresh block must not depend on them
        self.sc = rng.uniform(-3.0, 3.0, size=(wl.num_blocks, wl.n_kv, 4)).astype(np.float32)
        self.dkv = torch.from_numpy(self.kv.copy()).cuda()
        self.dsc = torch.from_numpy(self.sc.copy()).cuda()
        self.bs = wl.block_size

    def append(self, oracle, k, v, slots):
        import torch
        pkv.pkv_kv_append_fp8_block(_bf16_dev(k), _bf16_dev(v), torch.from_numpy(slots).cuda(),
                                    self.dkv, self.dsc)
        oracle.kv_append_fp8_block(k, v, slots, self.kv, self.sc, block_size=self.bs)

    def assert_same(self, what=""):
        got_kv, got_sc = self.dkv.cpu().numpy(), self.dsc.cpu().numpy()
        bad = np.nonzero(got_kv != self.kv)
        assert bad[0].size == 0, (what, [b[:5] for b in bad], got_kv[bad][:5], self.kv[bad][:5])
        badf = np.nonzero(got_sc.view(np.uint32) != self.sc.view(np.uint32))
        assert badf[0].size == 0, (what, [b[:5] for b in badf], got_sc[badf][:5],
                                   self.sc[badf][:5])


def _fill(oracle, wl, seed=0, check=True):
    """A block-scaled cache holding the workload's history and its step's new tokens."""
    import torch
    c = BlockCache(wl, seed)
    for i, (k, v, s) in enumerate(_history(wl)):
        c.append(oracle, k, v, s)
        if check:
            c.assert_same(f"history call {i}")
    c.append(oracle, wl.k_new, wl.v_new, wl.slot_mapping)
    torch.cuda.synchronize()
    if check:
        c.assert_same("step append")
    return c


def _run(dw, c, wl, kind, flags=0, window=0):
    import torch
    dt = torch.bfloat16 if kind == "bf16" else torch.float32
    out = torch.full(tuple(dw.q.shape), float("nan"), dtype=dt, device="cuda")
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim,
                             wl.block_size, flags=flags)
    pkv.pkv_paged_decode_attn_ex(dw.q, c.dkv, None, dw.block_tables, dw.context_lens, wl.scale,
                                 out, ws, flags=flags, window=window, kv_scales=c.dsc)
    st = pkv.pkv_check_error(ws)
    assert st == pkv.PKV_OK, pkv.pkv_status_string(st)
    return out


def _ref(oracle, wl, kv, sc, window=0):
    return oracle.paged_attn_fp8_block(wl.q, kv, sc, wl.block_tables, wl.context_lens,
                                       n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim,
                                       block_size=wl.block_size, scale=wl.scale, window=window)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_block_append_special_values_bit_exact(oracle, d):
    """Fresh blocks, growth, restart at offset 0, zeros, non-finite values, skipped slots
    and a duplicated slot inside a run, over three calls.  (head_dim 256: rows wider than
    a warp's 128 elements, which the append takes in several passes; the attention call
    supports 64 and 128 only.)"""
    import torch
    n_kv, bs, pool = 2, 16, 6
    rng = np.random.default_rng(60 + d)
    wl = make_custom(num_seqs=1, q_len=1, n_q=2, n_kv=n_kv, head_dim=d, block_size=bs,
                     context_lens=[1], seed=5, extra_poison=pool - 1)
    c = BlockCache(wl, seed=3)

    def rows(n, scale):
        return rng.standard_normal((n, n_kv, d)).astype(np.float32) * np.float32(scale)

    # call 1: block 1 offsets 0..4 with a skipped slot and a duplicate inside the run;
    # block 2 offset 0 all zeros; block 3 offsets 0, 1 with non-finite and tiny values;
    # block 0 full (offsets 0..15)
    s1 = [bs + 0, bs + 1, -1, bs + 2, bs + 2, bs + 3, bs + 4, 2 * bs, 3 * bs, 3 * bs + 1] + \
        list(range(0, bs))
    x = rows(len(s1), 3.0)
    x[7] = 0.0
    x[8, 0, :5] = [np.nan, np.inf, -np.inf, 1e-3, -0.0]
    x[9] = np.float32(2.0 ** -135) * np.sign(x[9])
    kx, vx = x, rows(len(s1), 0.01)
    vx[7] = -0.0
    c.append(oracle, f32_to_bf16_bits(kx), f32_to_bf16_bits(vx), np.asarray(s1, np.int32))
    torch.cuda.synchronize()
    c.assert_same("call 1")
    # call 2: block 1 grows (offset 5, values x100: the resident rows are re-quantised);
    # block 2 leaves scale 0 (offset 1); block 3 offset 2 smaller values (no growth);
    # block 0 restarts at offset 0 with small values
    s2 = [bs + 5, 2 * bs + 1, 3 * bs + 2, 0, 1]
    kx, vx = rows(len(s2), 1.0), rows(len(s2), 1.0)
    kx[0] *= 300.0
    vx[0] *= 1e4
    kx[2] *= 1e-3
    kx[3:] *= 1e-2
    c.append(oracle, f32_to_bf16_bits(kx), f32_to_bf16_bits(vx), np.asarray(s2, np.int32))
    torch.cuda.synchronize()
    c.assert_same("call 2")
    # call 3: growth by a factor of 2^20 (many resident values fall below the normal range)
    s3 = [bs + 6]
    kx, vx = rows(1, 3e6), rows(1, 1e4)
    c.append(oracle, f32_to_bf16_bits(kx), f32_to_bf16_bits(vx), np.asarray(s3, np.int32))
    torch.cuda.synchronize()
    c.assert_same("call 3")


CASES = [
    # head_dim, block_size, n_q, n_kv, q_len, context_lens           (consumer)
    (128, 16, 32, 8, 1, [1, 15, 16, 17, 200, 1000, 3]),             # narrow
    (64, 32, 8, 8, 2, [2, 3, 64, 65, 129, 700]),                    # narrow, d 64, q_len 2
    (64, 16, 4, 2, 1, [17, 40, 1, 0, 16, 33]),                      # narrow, d 64, empty seq
    (128, 16, 16, 1, 3, [3, 100, 47, 1500]),                         # wide
    (128, 32, 64, 8, 2, [2, 70, 1030]),                              # wide
    (128, 16, 32, 1, 4, [4, 5, 31, 33, 500, 2000]),                  # tensor memory, 128 rows
    (64, 32, 128, 1, 1, [31, 1, 999]),                               # tensor memory, d 64
    (128, 16, 32, 8, 40, [40, 300, 900]),                            # prefill tiles
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
def test_block_append_history_bit_exact_and_parity(oracle, case):
    """A cache filled by the block append (history in two calls, then the step) matches the
    oracle bit for bit, and attention over it matches the oracle at forced CTA counts,
    with and without a window."""
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=501 + n_q + q_len + d)
    c = _fill(oracle, wl, seed=7)
    dw = to_device(wl)
    for grid in (0, 1, 7, 64):
        flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
        for window in (0, 17):
            ref = _ref(oracle, wl, c.kv, c.sc, window)
            for kind in ("bf16", "f32"):
                out = _run(dw, c, wl, kind, flags, window)
                assert_close(out_to_host(out), ref, kind, f"{case} grid {grid} W {window} {kind}")


@pytest.mark.parametrize("case", CASES, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
@pytest.mark.parametrize("grid", [0, 7])
def test_block_parity_arbitrary_scales(oracle, case, grid):
    """Random codes with arbitrary positive block scales spanning nine binades (the
    running V-scale reference then grows by ratios that are not powers of two).  The
    scales keep values within 56, as attention inputs are: with codes up to 448 times
    scales near 4, log2-domain scores reach the thousands, where fp32's resolution
    alone moves each weight by ~1e-4 relative, and outputs that are small sums of
    large terms lose those digits to cancellation."""
    import torch
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=601 + n_q + q_len + d)
    c8 = fp8_cache_for(wl)
    rng = np.random.default_rng(602 + d)
    # the step's new tokens are resident too: give their (still poisoned) slots finite codes
    finite = np.asarray([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for sl in wl.slot_mapping:
        if sl >= 0:
            c8.kv_cache[sl // bs, :, :, sl % bs, :] = rng.choice(
                finite, size=c8.kv_cache[sl // bs, :, :, sl % bs, :].shape)
    sc = np.zeros((wl.num_blocks, n_kv, 4), dtype=np.float32)
    sc[:, :, 0:2] = (2.0 ** rng.uniform(-12.0, -3.0, size=(wl.num_blocks, n_kv, 2))).astype(np.float32)
    dw = to_device(wl)

    class C:
        dkv = torch.from_numpy(c8.kv_cache).cuda()
        dsc = torch.from_numpy(sc).cuda()

    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    ref = _ref(oracle, wl, c8.kv_cache, sc)
    for kind in ("bf16", "f32"):
        out = _run(dw, C, wl, kind, flags)
        assert_close(out_to_host(out), ref, kind, f"{case} grid {grid} {kind}")


@pytest.fixture(scope="module", params=list(CONFIGS))
def named_blk(request, oracle):
    import torch
    wl = make_workload(request.param)
    c = _fill(oracle, wl, seed=11, check=False)
    dw = to_device(wl)
    dw.k_cache = dw.v_cache = None
    torch.cuda.synchronize()
    ref = _ref(oracle, wl, c.kv, c.sc)
    yield wl, dw, c, ref
    del dw, c
    torch.cuda.empty_cache()


def test_named_block_append_bit_exact(named_blk):
    _, _, c, _ = named_blk
    c.assert_same("named")


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_named_block_attention(named_blk, kind):
    wl, dw, c, ref = named_blk
    assert_close(out_to_host(_run(dw, c, wl, kind)), ref, kind, f"{wl.name}/fp8-block/{kind}")


def test_named_block_split_points(named_blk):
    wl, dw, c, ref = named_blk
    for grid in (7, 300):
        out = _run(dw, c, wl, "f32", flags=pkv.PKV_FLAG_GRID(grid))
        assert_close(out_to_host(out), ref, "f32", f"{wl.name}/fp8-block/grid{grid}")


def test_block_copy_copies_scales():
    import torch
    rng = np.random.default_rng(9)
    kv8 = rng.integers(0, 256, (10, 2, 2, 16, 64), dtype=np.uint8)
    sc = rng.standard_normal((10, 2, 4)).astype(np.float32)
    pairs = np.asarray([[1, 4], [7, 2], [3, 3], [0, 11]], dtype=np.int32)
    g, gs = torch.from_numpy(kv8).cuda(), torch.from_numpy(sc).cuda()
    pkv.pkv_copy_blocks(g, gs, torch.from_numpy(pairs).cuda())
    want, want_sc = kv8.copy(), sc.copy()
    want[4], want[2] = kv8[1], kv8[7]
    want_sc[4], want_sc[2] = sc[1], sc[7]
    assert np.array_equal(g.cpu().numpy(), want)
    assert np.array_equal(gs.cpu().numpy(), want_sc)
