"""Prefix sharing with copy-on-write on the GPU, checked against a host replay with the oracle.

A 40-token prompt is written once and shared by three sequences (fork); each
then decodes its own tokens.  The host block pool hands out slots and asks for
copies of shared blocks before they are written; the device copies them
(pkv_copy_blocks), appends (pkv_kv_append) and attends (pkv_paged_decode_attn).
The same operations replayed on host arrays with the oracle must give
bit-identical caches and attention within tolerance, and the shared prompt
blocks must never change.
"""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv
from paged_kv_cache_256_gb300.device import bf16_to_host_bits
from paged_kv_cache_256_gb300.workloads import BF16_POISON, f32_to_bf16_bits
from tests.gpu_common import assert_close, out_to_host

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def test_copy_blocks_bit_exact(oracle):
    import torch
    rng = np.random.default_rng(31)
    shape = (40, 4, 16, 128)
    kc = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    pairs = np.asarray([[3, 17], [5, 5], [39, 0], [-2, 8], [12, 40], [21, 22], [7, 30]],
                       dtype=np.int32)
    kd, vd = _dev(kc), _dev(vc)
    pkv.pkv_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
    oracle.copy_blocks(pairs, kc, vc)
    assert np.array_equal(bf16_to_host_bits(kd), kc)
    assert np.array_equal(bf16_to_host_bits(vd), vc)


def test_forked_sequences_decode_with_copy_on_write(oracle):
    import torch
    rng = np.random.default_rng(32)
    n_q, n_kv, d, bs, num_blocks, max_blocks = 8, 2, 128, 16, 32, 8
    scale = float(np.float32(1 / np.sqrt(d)))
    kc = np.full((num_blocks, n_kv, bs, d), BF16_POISON, dtype=np.uint16)
    vc = kc.copy()
    pool = pkv.BlockPool(num_blocks, bs)

    def rows(n):
        return f32_to_bf16_bits(rng.standard_normal((n, n_kv, d)).astype(np.float32))

    # the shared 40-token prompt
    prompt = np.full(max_blocks, 0, dtype=np.int32)
    nb, slots, pairs = pool.append_slots(prompt, 0, 0, 40)
    assert pairs.shape == (0, 2)
    oracle.kv_append(rows(40), rows(40), slots, kc, vc, block_size=bs)
    prompt_blocks = prompt[:nb].copy()
    prompt_k = kc[prompt_blocks[:2]].copy()  # the two full blocks stay shared throughout
    kd, vd = _dev(kc), _dev(vc)

    seqs = []
    for _ in range(3):
        t = prompt.copy()
        pool.share(t[:nb])
        seqs.append([t, nb, 40])
    pool.release(prompt[:nb])  # the prompt's own reference goes away

    ws = pkv.alloc_workspace(3, 1, n_q, n_kv, d, bs)
    for step in range(3):
        all_slots, all_pairs = [], []
        for s in seqs:
            s[1], sl, pr = pool.append_slots(s[0], s[1], s[2], 1)
            s[2] += 1
            all_slots.append(sl)
            all_pairs.append(pr)
        pairs = np.concatenate(all_pairs).astype(np.int32)
        slots = np.concatenate(all_slots).astype(np.int32)
        k_new, v_new = rows(3), rows(3)
        q = f32_to_bf16_bits(rng.standard_normal((3, 1, n_q, d)).astype(np.float32))
        tables = np.stack([s[0] for s in seqs]).astype(np.int32)
        ctx = np.asarray([s[2] for s in seqs], dtype=np.int32)
        # device
        if pairs.shape[0]:
            pkv.pkv_copy_blocks(kd, vd, torch.from_numpy(pairs).cuda())
        pkv.pkv_kv_append(_dev(k_new), _dev(v_new), torch.from_numpy(slots).cuda(), kd, vd)
        out = torch.empty((3, 1, n_q, d), dtype=torch.bfloat16, device="cuda")
        pkv.pkv_paged_decode_attn(_dev(q), kd, vd, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(ctx).cuda(), scale, out, ws)
        assert pkv.pkv_check_error(ws) == pkv.PKV_OK
        # host replay
        if pairs.shape[0]:
            oracle.copy_blocks(pairs, kc, vc)
        oracle.kv_append(k_new, v_new, slots, kc, vc, block_size=bs)
        ref = oracle.paged_attn(q, kc, vc, tables, ctx, n_q=n_q, n_kv=n_kv, head_dim=d,
                                block_size=bs, scale=scale)
        assert np.array_equal(bf16_to_host_bits(kd), kc), step
        assert np.array_equal(bf16_to_host_bits(vd), vc), step
        assert_close(out_to_host(out), ref, "bf16", f"forked decode step {step}")
        if step == 0:
            assert pairs.shape[0] == 2  # two of the three forks copy the shared partial block
        assert np.array_equal(kc[prompt_blocks[:2]], prompt_k)
        assert all(pool.refcount(int(b)) == 3 for b in prompt_blocks[:2])
