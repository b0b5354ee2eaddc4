"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

kv_append and all block-table indexing are compared bit for bit; attention
outputs element by element within |gpu - ref| <= 1e-2 + 1e-2|ref| (bf16
output) or 1e-4 + 1e-4|ref| (fp32 output).  The named workloads run at
their full sizes in the launch configuration the benchmark times (one CTA
per SM), and again with the split points moved by forcing other CTA counts.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.workloads import CONFIGS, make_custom, make_workload
from tests.gpu_common import (assert_close, bf16_to_host_bits, oracle_after_append, out_to_host,
                              run_attn, to_device)

pytestmark = pytest.mark.gpu

CONFIG_NAMES = list(CONFIGS)


@pytest.fixture(scope="module", params=CONFIG_NAMES)
def named(request, oracle):
    """(workload, device copy with the append done on the GPU, oracle caches, oracle output)."""
    import torch
    wl = make_workload(request.param)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    torch.cuda.synchronize()
    kc, vc, ref = oracle_after_append(oracle, wl)
    yield wl, dw, kc, vc, ref
    del dw
    torch.cuda.empty_cache()


def test_kv_append_bit_exact(named):
    wl, dw, kc, vc, _ = named
    assert np.array_equal(bf16_to_host_bits(dw.k_cache), kc)
    assert np.array_equal(bf16_to_host_bits(dw.v_cache), vc)


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_attention_matches_oracle(named, kind):
    wl, dw, _, _, ref = named
    out = run_attn(dw, wl, kind)
    assert_close(out_to_host(out), ref, kind, f"{wl.name}/{kind}")


@pytest.mark.parametrize("grid", [1, 7, 300, 2000])
def test_split_points_do_not_change_the_result(named, grid):
    wl, dw, _, _, ref = named
    if wl.name in ("llama2_7b_mha",) and grid == 1:
        pytest.skip("one CTA over 1 GB is slow and adds nothing over the other grids")
    out = run_attn(dw, wl, "f32", flags=pkv.PKV_FLAG_GRID(grid))
    assert_close(out_to_host(out), ref, "f32", f"{wl.name}/grid{grid}")


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_one_and_two_copy_tiles_agree_bit_for_bit(named, kind):
    """With more than 64 rows per KV head a bf16 head_dim-128 K or V tile arrives
    by one copy through a grouped 4-D view, or by two 64-column copies under
    PKV_FLAG_TILE_2D; the products read the same values, so the outputs match
    bit for bit."""
    wl, dw, _, _, _ = named
    a = run_attn(dw, wl, kind)
    b = run_attn(dw, wl, kind, flags=pkv.PKV_FLAG_TILE_2D)
    assert np.array_equal(a.cpu().view(torch_int_of(kind)).numpy(),
                          b.cpu().view(torch_int_of(kind)).numpy())


def torch_int_of(kind):
    import torch
    return torch.int16 if kind == "bf16" else torch.int32


def test_repeatable_bit_for_bit(named):
    wl, dw, _, _, _ = named
    a = bf16_to_host_bits(run_attn(dw, wl, "bf16"))
    b = bf16_to_host_bits(run_attn(dw, wl, "bf16"))
    assert np.array_equal(a, b)


def test_tiny_append_is_visible(oracle):
    """Tiny workload: attend at {17, 40}, append one token each, attend at {18, 41}."""
    import torch
    wl = make_workload("tiny")
    dw = to_device(wl)
    kw = dict(n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
              scale=wl.scale)
    before_ctx = wl.context_lens - 1
    ref0 = oracle.paged_attn(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, before_ctx, **kw)
    for kind in ("bf16", "f32"):
        out0 = run_attn(dw, wl, kind, context_lens=torch.from_numpy(before_ctx).cuda())
        assert_close(out_to_host(out0), ref0, kind, "tiny before append")
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    kc, vc, ref1 = oracle_after_append(oracle, wl)
    assert np.array_equal(bf16_to_host_bits(dw.k_cache), kc)
    assert np.array_equal(bf16_to_host_bits(dw.v_cache), vc)
    for kind in ("bf16", "f32"):
        out1 = run_attn(dw, wl, kind)
        assert_close(out_to_host(out1), ref1, kind, "tiny after append")
    assert not np.allclose(ref0, ref1)


SWEEP = [
    # head_dim, block_size, n_q, n_kv, q_len, context_lens
    (64, 16, 4, 2, 1, [17, 40, 1, 0, 16, 33]),
    (128, 16, 32, 8, 1, [1, 15, 16, 17, 200, 1000, 3]),
    (128, 32, 32, 1, 4, [4, 5, 31, 32, 33, 500, 2000]),
    (64, 32, 6, 3, 2, [2, 3, 64, 65, 129]),
    (128, 16, 16, 1, 3, [3, 100, 47]),
    (128, 16, 40, 40, 1, [10, 300]),
    (64, 16, 8, 8, 8, [8, 9, 100]),
    (128, 32, 64, 8, 2, [2, 70, 1030]),
    (128, 16, 7, 1, 1, [5, 77, 160]),
    (64, 32, 128, 1, 1, [31, 1, 999]),
    (128, 16, 8, 2, 4, [2, 0, 5, 1]),  # contexts shorter than q_len: rows with no key -> 0
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: "d{}_bs{}_q{}_kv{}_ql{}".format(*c[:5]))
@pytest.mark.parametrize("grid", [0, 1, 3, 64])
def test_shape_sweep(oracle, case, grid):
    d, bs, n_q, n_kv, q_len, ctxs = case
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=d,
                     block_size=bs, context_lens=ctxs, seed=7 + len(ctxs) * 31 + d)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    _, _, ref = oracle_after_append(oracle, wl)
    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    for kind in ("bf16", "f32"):
        out = run_attn(dw, wl, kind, flags=flags)
        assert_close(out_to_host(out), ref, kind, f"sweep {case} grid {grid} {kind}")


@pytest.mark.parametrize("num_seqs", [288, 289, 700, 3000])
@pytest.mark.parametrize("grid", [0, 7, 300])
def test_large_batches(oracle, num_seqs, grid):
    """Batches of many short sequences, some empty: the work partition scans
    the context lengths one sequence per thread (288 per round), so these
    sizes cover an exact round and several rounds."""
    rng = np.random.default_rng(num_seqs)
    ctxs = rng.integers(1, 80, num_seqs)
    ctxs[rng.random(num_seqs) < 0.1] = 0
    wl = make_custom(num_seqs=num_seqs, q_len=1, n_q=8, n_kv=2, head_dim=64, block_size=16,
                     context_lens=[int(c) for c in ctxs], seed=11 + num_seqs)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    _, _, ref = oracle_after_append(oracle, wl)
    flags = pkv.PKV_FLAG_GRID(grid) if grid else 0
    for kind in ("bf16", "f32"):
        out = run_attn(dw, wl, kind, flags=flags)
        assert_close(out_to_host(out), ref, kind, f"{num_seqs} seqs grid {grid} {kind}")


@pytest.mark.parametrize("flags", [0, pkv.PKV_FLAG_NO_EARLY_START], ids=["early", "no_early"])
@pytest.mark.parametrize("n_q,q_len", [(8, 1), (32, 4)], ids=["narrow", "tmem"])
def test_inputs_written_just_before_the_call_are_seen(oracle, n_q, q_len, flags):
    """Stream order with programmatic launches: q and the context lengths are
    rewritten by ordinary kernels, the append runs, and the attention call
    follows at once, with no synchronisation between them: the output must be
    that of the rewritten inputs (the attention's work partition may overlap
    the append, never the kernels before it; with PKV_FLAG_NO_EARLY_START it
    overlaps nothing)."""
    import torch
    ctxs = [33, 700, 5, 260]
    wl = make_custom(num_seqs=len(ctxs), q_len=q_len, n_q=n_q, n_kv=1 if n_q == 32 else 2,
                     head_dim=128, block_size=16, context_lens=ctxs, seed=91 + n_q)
    dw = to_device(wl)
    q_right, cl_right = dw.q.clone(), dw.context_lens.clone()
    _, _, ref = oracle_after_append(oracle, wl)
    ws = pkv.alloc_workspace(wl.num_seqs, wl.q_len, wl.n_q, wl.n_kv, wl.head_dim, wl.block_size)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        dw.q.zero_()
        dw.context_lens.fill_(1)
        dw.q.copy_(q_right)
        dw.context_lens.copy_(cl_right)
        pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
        pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                  dw.context_lens, wl.scale, out, ws, flags=flags)
        assert pkv.pkv_check_error(ws) == pkv.PKV_OK
        assert_close(out_to_host(out), ref, "f32", "inputs rewritten before the call")


def test_block_relabelling_is_bit_identical():
    """Moving physical blocks (and rewriting the table) leaves the output bit-identical."""
    import torch
    ctxs = [3, 100, 1000, 17, 2500, 64]
    wl = make_custom(num_seqs=6, q_len=1, n_q=32, n_kv=8, head_dim=128, block_size=16,
                     context_lens=ctxs, seed=5)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    base = {k: bf16_to_host_bits(run_attn(dw, wl, "bf16", flags=pkv.PKV_FLAG_GRID(g)))
            for k, g in (("a", 0), ("b", 5))}
    relabel = np.random.default_rng(3).permutation(wl.num_blocks)
    perm_t = torch.from_numpy(np.argsort(relabel)).cuda()  # new index -> old index
    dw.k_cache = dw.k_cache[perm_t].contiguous()
    dw.v_cache = dw.v_cache[perm_t].contiguous()
    dw.block_tables = torch.from_numpy(relabel[wl.block_tables].astype(np.int32)).cuda()
    for k, g in (("a", 0), ("b", 5)):
        got = bf16_to_host_bits(run_attn(dw, wl, "bf16", flags=pkv.PKV_FLAG_GRID(g)))
        assert np.array_equal(got, base[k])


def test_single_resident_token_returns_its_value():
    import torch
    wl = make_custom(num_seqs=5, q_len=1, n_q=16, n_kv=4, head_dim=128, block_size=16,
                     context_lens=[1] * 5, seed=8)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    G = wl.n_q // wl.n_kv
    want = np.repeat(wl.v_new.reshape(5, 1, wl.n_kv, 128), G, axis=2)  # [seq, 1, n_q, d]
    out = run_attn(dw, wl, "bf16")
    assert np.array_equal(bf16_to_host_bits(out), want)
    out32 = run_attn(dw, wl, "f32").cpu().numpy()
    assert np.array_equal(out32, (want.astype(np.uint32) << 16).view(np.float32))


def test_equal_scores_give_the_mean_of_values(oracle):
    import torch
    wl = make_custom(num_seqs=3, q_len=1, n_q=8, n_kv=2, head_dim=64, block_size=16,
                     context_lens=[5, 300, 48], seed=9)
    wl.q[...] = 0
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    _, vc, ref = oracle_after_append(oracle, wl)
    out = run_attn(dw, wl, "f32")
    assert_close(out_to_host(out), ref, "f32", "equal scores")


def test_checked_mode_reports_bad_tables():
    import torch
    wl = make_custom(num_seqs=3, q_len=1, n_q=8, n_kv=2, head_dim=128, block_size=16,
                     context_lens=[40, 70, 5], seed=10)
    dw = to_device(wl)
    flags = pkv.PKV_FLAG_CHECKED
    ws = pkv.alloc_workspace(3, 1, 8, 2, 128, 16, flags=flags)
    out = torch.empty(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")

    def call(bt, cl):
        pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, bt, cl, wl.scale, out, ws,
                                  flags=flags)
        return pkv.pkv_check_error(ws)

    assert call(dw.block_tables, dw.context_lens) == pkv.PKV_OK
    for bad in (wl.num_blocks, wl.num_blocks + 1000, -3):
        bt = wl.block_tables.copy()
        bt[1, 2] = bad  # a block the sequence uses
        assert call(torch.from_numpy(bt).cuda(), dw.context_lens) == pkv.PKV_ERR_BAD_BLOCK_TABLE
    cl = wl.context_lens.copy()
    cl[0] = wl.max_blocks_per_seq * 16 + 1  # longer than the table
    assert call(dw.block_tables, torch.from_numpy(cl).cuda()) == pkv.PKV_ERR_BAD_BLOCK_TABLE
    cl = wl.context_lens.copy()
    cl[2] = -4
    assert call(dw.block_tables, torch.from_numpy(cl).cuda()) == pkv.PKV_ERR_BAD_BLOCK_TABLE
    # and the workspace is clean again afterwards
    assert call(dw.block_tables, dw.context_lens) == pkv.PKV_OK


@pytest.mark.parametrize("n_q,n_kv,q_len,head_dim", [(4, 2, 1, 64), (8, 2, 1, 128),
                                                      (32, 1, 4, 128)],
                         ids=["narrow_d64", "narrow_d128", "tmem_d128"])
def test_unchecked_bad_block_id_reads_zeros_without_fault(n_q, n_kv, q_len, head_dim):
    """Without CHECKED, an out-of-range id is read as a zero tile (no access outside the cache)."""
    import torch
    wl = make_custom(num_seqs=2, q_len=q_len, n_q=n_q, n_kv=n_kv, head_dim=head_dim,
                     block_size=16, context_lens=[40, 20], seed=11)
    dw = to_device(wl)
    pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
    bt = wl.block_tables.copy()
    bt[0, 1] = 1 << 30
    dw.block_tables = torch.from_numpy(bt).cuda()
    out = run_attn(dw, wl, "f32")
    assert torch.isfinite(out).all()
    # the zero tile is the same whichever way the tiles are fetched
    out2 = run_attn(dw, wl, "f32", flags=pkv.PKV_FLAG_TILE_2D)
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))


def test_kv_append_skips_padding_and_out_of_range_slots():
    import torch
    rng = np.random.default_rng(12)
    pool, n_kv, bs, d = 6, 2, 16, 128
    kc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
    slots = np.asarray([5, -1, pool * bs, 17, pool * bs - 1, 0, -7], dtype=np.int32)
    kn = rng.integers(0, 1 << 16, size=(7, n_kv, d), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(7, n_kv, d), dtype=np.uint16)
    k_ref, v_ref = kc.copy(), vc.copy()
    for i, s in enumerate(slots):
        if 0 <= s < pool * bs:
            k_ref[s // bs, :, s % bs] = kn[i]
            v_ref[s // bs, :, s % bs] = vn[i]

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)

    kcd, vcd = dev(kc), dev(vc)
    pkv.pkv_kv_append(dev(kn), dev(vn), torch.from_numpy(slots).cuda(), kcd, vcd)
    assert np.array_equal(bf16_to_host_bits(kcd), k_ref)
    assert np.array_equal(bf16_to_host_bits(vcd), v_ref)


def test_cuda_graph_replay_matches_eager(oracle):
    """The append + attention + merge launches capture into one CUDA graph."""
    import torch
    wl = make_custom(num_seqs=8, q_len=1, n_q=32, n_kv=8, head_dim=128, block_size=16,
                     context_lens=[100, 2000, 37, 4096, 1, 640, 3000, 17], seed=13)
    dw = to_device(wl)
    ws = pkv.alloc_workspace(8, 1, 32, 8, 128, 16)
    out = torch.zeros(tuple(dw.q.shape), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkv.pkv_kv_append(dw.k_new, dw.v_new, dw.slot_mapping, dw.k_cache, dw.v_cache)
        pkv.pkv_paged_decode_attn(dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.context_lens,
                                  wl.scale, out, ws)
    g.replay()
    torch.cuda.synchronize()
    assert pkv.pkv_check_error(ws) == pkv.PKV_OK
    _, _, ref = oracle_after_append(oracle, wl)
    assert_close(out_to_host(out), ref, "bf16", "graph replay")
    eager = run_attn(dw, wl, "bf16")
    assert np.array_equal(bf16_to_host_bits(eager), bf16_to_host_bits(out))
