"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an oracle handle (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with what the pages or the
mathematics fix.  ``test_oracle_pins.py`` runs them against the real oracle;
``test_oracle_mutants.py`` runs them against copies of the oracle with one
planted mistake each and requires every mutant to fail at least one pin.

What pins what:

* ``pin_library_sdpa``      -- torch's own scaled-dot-product attention (fp64,
  CPU) on the logical, contiguous K/V the paged cache was built from: the
  textbook definition softmax(QK^T/sqrt(d) + causal_mask)V ("Transformer
  inference mechanics", What Q, K, and V do in causal attention), with GQA
  expressed by the library's own head repeat.
* ``pin_equal_scores_mean`` -- q = 0 makes all scores equal, so the output is
  the plain mean of the visible V rows.
* ``pin_single_token``      -- one resident token: the output is that token's V.
* ``pin_hardmax``           -- a huge scale turns softmax into argmax: the output
  is V at the largest score.
* ``pin_block_permutation`` -- paging changes only where K/V live ("Transformer
  inference mechanics", FlashAttention versus PagedAttention): any relabelling
  of physical blocks gives the identical output.
* ``pin_gqa_equals_repeated_mha`` -- GQA over n_kv heads equals MHA over
  K/V heads repeated group-wise ("Transformer inference mechanics", MHA versus
  MQA versus GQA).
* ``pin_causal_rows``       -- draft token i of gamma equals a one-token query
  over the prefix ending at its own position.
* ``pin_prefill_sdpa``      -- a block of new tokens (pure or chunked prefill)
  against torch SDPA, including its own ``is_causal`` flag.
* ``pin_merge_exact``       -- partials of any split of the key range merge to
  the unsplit result ("Efficient inference", FlashAttention: partial results
  are rescaled and combined exactly).
* ``pin_kv_append``         -- slots written, everything else byte-identical.
* ``pin_kv_bytes_golden`` / ``pin_gqa_ratio`` -- the sizes printed on the pages.
* ``pin_e4m3_decode_library`` / ``pin_e4m3_encode_library`` -- the 8-bit float
  codec against torch's own ``float8_e4m3fn`` conversions (every code; exact
  ties, near-ties, subnormals, random values at every magnitude).
* ``pin_e4m3_saturation``   -- the saturating reading beyond 448, NaN, and
  decode-then-encode returning every finite code.
* ``pin_fp8_attention_sdpa`` -- attention over an e4m3 cache equals torch SDPA
  on the K/V that torch dequantises (code value times the head's scale).
* ``pin_kv_append_fp8``     -- the quantising append against numpy's fp32
  division and torch's encoder.
* ``pin_fp8_block_attention_sdpa`` -- attention over an e4m3 cache with one
  scale per (block, KV head) equals torch SDPA on K/V the test dequantises
  itself, logical block by logical block; unused blocks carry NaN scales.
* ``pin_fp8_block_equals_per_head`` -- block scales that are the same for every
  block of a head give the per-head result bit for bit.
* ``pin_fp8_block_append_fresh`` -- a block written from offset 0: its scale is
  the smallest power of two that keeps every finite value within 448 (checked
  as an inequality, not recomputed), the codes are torch's encoding of the fp32
  quotients, non-finite values are stored as they encode, all-zero blocks
  keep scale 0.
* ``pin_fp8_block_append_growth`` -- a later token with larger values raises
  the scale by a power of two: resident rows keep their exact value where it
  stays in the normal e4m3 range and move by at most half a subnormal step
  below it; rows past the new tokens are not touched; smaller values leave the
  scale and the resident rows alone.
* ``pin_fp8_block_append_then_attend`` -- bf16 rows appended through the block
  scales and attended over stay within the e4m3 rounding of the bf16 result.
"""
from __future__ import annotations

import math
import os

import numpy as np

from paged_kv_cache_256_gb300.workloads import (
    BF16_POISON, bf16_bits_to_f32, f32_to_bf16_bits, make_custom)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kv_bytes.txt")


# ---------------------------------------------------------------------------
# helpers (test-side only)
# ---------------------------------------------------------------------------
def _rand_bf16(rng, shape, scale=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def _paged_from_logical(rng, K, V, block_size, extra_blocks=3, poison=BF16_POISON):
    """Scatter logical K/V [num_seqs][n_kv][ctx_b][d] (lists) into a shuffled paged cache.

    Built by the test itself, independently of the oracle's gather.
    Returns (k_cache, v_cache, block_tables) with poison in every unused slot
    (the caches take the dtype of K).
    """
    num_seqs = len(K)
    n_kv, d = K[0].shape[0], K[0].shape[2]
    nblk = [max(0, math.ceil(k.shape[1] / block_size)) for k in K]
    used = sum(nblk)
    pool = used + extra_blocks
    perm = rng.permutation(pool)
    max_blocks = max(1, max(nblk))
    bt = np.full((num_seqs, max_blocks), perm[-1], dtype=np.int32)
    kc = np.full((pool, n_kv, block_size, d), poison, dtype=K[0].dtype)
    vc = np.full_like(kc, poison)
    o = 0
    for b in range(num_seqs):
        for j in range(nblk[b]):
            phys = perm[o]
            o += 1
            bt[b, j] = phys
            lo, hi = j * block_size, min((j + 1) * block_size, K[b].shape[1])
            kc[phys, :, : hi - lo, :] = K[b][:, lo:hi, :]
            vc[phys, :, : hi - lo, :] = V[b][:, lo:hi, :]
    return kc, vc, bt


def _case(rng, ctxs, n_q, n_kv, d, bs, q_len, kscale=1.0):
    K = [_rand_bf16(rng, (n_kv, c, d), kscale) for c in ctxs]
    V = [_rand_bf16(rng, (n_kv, c, d)) for c in ctxs]
    kc, vc, bt = _paged_from_logical(rng, K, V, bs)
    q = _rand_bf16(rng, (len(ctxs), q_len, n_q, d))
    return dict(q=q, K=K, V=V, k_cache=kc, v_cache=vc, block_tables=bt,
                context_lens=np.asarray(ctxs, dtype=np.int32), n_q=n_q, n_kv=n_kv,
                head_dim=d, block_size=bs, q_len=q_len)


def _run(orc, c, scale, window=0, **over):
    args = dict(c)
    args.update(over)
    return orc.paged_attn(args["q"], args["k_cache"], args["v_cache"], args["block_tables"],
                          args["context_lens"], n_q=args["n_q"], n_kv=args["n_kv"],
                          head_dim=args["head_dim"], block_size=args["block_size"],
                          scale=scale, window=window)


SHAPES = [
    # ctxs, n_q, n_kv, d, bs, q_len
    ([5, 17, 33], 4, 4, 16, 4, 1),       # MHA, ragged, partial last blocks
    ([1, 9, 40], 8, 2, 8, 4, 1),         # GQA G=4
    ([7, 23], 6, 1, 16, 8, 1),           # MQA
    ([6, 19, 12], 4, 2, 8, 4, 3),        # GQA + causal draft tokens
    ([4, 30], 8, 1, 16, 16, 4),          # MQA verify, gamma = 4
]


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------
def pin_library_sdpa(orc):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(11)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        scale = float(np.float32(1.0 / math.sqrt(d)))
        got = _run(orc, c, scale)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            q = torch.from_numpy(bf16_bits_to_f32(c["q"][b]).astype(np.float64))  # [q_len, n_q, d]
            k = torch.from_numpy(bf16_bits_to_f32(c["K"][b]).astype(np.float64))  # [n_kv, ctx, d]
            v = torch.from_numpy(bf16_bits_to_f32(c["V"][b]).astype(np.float64))
            k = k.repeat_interleave(G, dim=0)
            v = v.repeat_interleave(G, dim=0)
            qh = q.permute(1, 0, 2)  # [n_q, q_len, d]
            pos = ctx - q_len + torch.arange(q_len)
            mask = torch.arange(ctx)[None, :] <= pos[:, None]
            ref = F.scaled_dot_product_attention(qh[None], k[None], v[None],
                                                 attn_mask=mask[None, None], scale=scale)[0]
            ref = ref.permute(1, 0, 2).numpy()
            np.testing.assert_allclose(got[b], ref, rtol=1e-12, atol=1e-12)


def pin_numpy_dense(orc):
    """Dense matrix form: S = Q K^T * scale with -inf above the causal diagonal."""
    rng = np.random.default_rng(12)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        scale = 0.37
        got = _run(orc, c, scale)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            for h in range(n_q):
                Q = bf16_bits_to_f32(c["q"][b, :, h, :]).astype(np.float64)
                K = bf16_bits_to_f32(c["K"][b][h // G]).astype(np.float64)
                V = bf16_bits_to_f32(c["V"][b][h // G]).astype(np.float64)
                S = Q @ K.T * scale
                rows = (ctx - q_len + np.arange(q_len))[:, None]
                S = np.where(np.arange(ctx)[None, :] <= rows, S, -np.inf)
                P = np.exp(S - S.max(axis=1, keepdims=True))
                ref = (P / P.sum(axis=1, keepdims=True)) @ V
                np.testing.assert_allclose(got[b, :, h, :], ref, rtol=1e-12, atol=1e-12)


def pin_equal_scores_mean(orc):
    rng = np.random.default_rng(13)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        c["q"] = np.zeros_like(c["q"])
        got = _run(orc, c, 0.125)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            for i in range(q_len):
                nvis = ctx - q_len + i + 1
                for h in range(n_q):
                    V = bf16_bits_to_f32(c["V"][b][h // G][:nvis]).astype(np.float64)
                    np.testing.assert_allclose(got[b, i, h], V.mean(axis=0), rtol=1e-13,
                                               atol=1e-15)


def pin_single_token(orc):
    rng = np.random.default_rng(14)
    c = _case(rng, [1, 1, 1], 6, 3, 16, 4, 1)
    got = _run(orc, c, 0.25)
    for b in range(3):
        for h in range(6):
            ref = bf16_bits_to_f32(c["V"][b][h // 2][0]).astype(np.float64)
            assert np.array_equal(got[b, 0, h], ref), (b, h)


def pin_hardmax(orc):
    rng = np.random.default_rng(15)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        got = _run(orc, c, 1.0e6)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            for i in range(q_len):
                nvis = ctx - q_len + i + 1
                for h in range(n_q):
                    q = bf16_bits_to_f32(c["q"][b, i, h]).astype(np.float64)
                    K = bf16_bits_to_f32(c["K"][b][h // G][:nvis]).astype(np.float64)
                    V = bf16_bits_to_f32(c["V"][b][h // G][:nvis]).astype(np.float64)
                    s = K @ q
                    top = np.sort(s)[::-1]
                    if len(top) > 1 and (top[0] - top[1]) * 1.0e6 < 800:
                        continue  # a near tie: not a clean argmax case
                    assert np.array_equal(got[b, i, h], V[int(np.argmax(s))]), (b, i, h)


def pin_block_permutation(orc):
    rng = np.random.default_rng(16)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        base = _run(orc, c, 0.3)
        pool = c["k_cache"].shape[0]
        relabel = rng.permutation(pool)  # old physical index -> new physical index
        kc = np.empty_like(c["k_cache"])
        vc = np.empty_like(c["v_cache"])
        kc[relabel] = c["k_cache"]
        vc[relabel] = c["v_cache"]
        bt = relabel[c["block_tables"]].astype(np.int32)
        got = _run(orc, c, 0.3, k_cache=kc, v_cache=vc, block_tables=bt)
        assert np.array_equal(base, got)


def pin_gqa_equals_repeated_mha(orc):
    rng = np.random.default_rng(17)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        if n_q == n_kv:
            continue
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        G = n_q // n_kv
        gqa = _run(orc, c, 0.2)
        kc = np.repeat(c["k_cache"], G, axis=1)  # KV head g -> query heads g*G .. g*G+G-1
        vc = np.repeat(c["v_cache"], G, axis=1)
        mha = _run(orc, c, 0.2, k_cache=kc, v_cache=vc, n_kv=n_q)
        assert np.array_equal(gqa, mha)


def pin_causal_rows(orc):
    rng = np.random.default_rng(18)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        if q_len == 1:
            continue
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        full = _run(orc, c, 0.25)
        for i in range(q_len):
            ctx_i = np.asarray(ctxs, dtype=np.int32) - q_len + i + 1
            one = _run(orc, c, 0.25, q=np.ascontiguousarray(c["q"][:, i:i + 1]),
                       context_lens=ctx_i, q_len=1)
            assert np.array_equal(full[:, i:i + 1], one), i


WINDOWS = [1, 3, 4, 5, 17]


def pin_window_sdpa(orc):
    """Sliding window: torch SDPA with a banded causal mask (CS336 notes, Local attention)."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(23)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        G = n_q // n_kv
        for W in WINDOWS:
            got = _run(orc, c, 0.3, window=W)
            for b, ctx in enumerate(ctxs):
                q = torch.from_numpy(bf16_bits_to_f32(c["q"][b]).astype(np.float64))
                k = torch.from_numpy(bf16_bits_to_f32(c["K"][b]).astype(np.float64))
                v = torch.from_numpy(bf16_bits_to_f32(c["V"][b]).astype(np.float64))
                k, v = k.repeat_interleave(G, dim=0), v.repeat_interleave(G, dim=0)
                pos = ctx - q_len + torch.arange(q_len)
                t = torch.arange(ctx)[None, :]
                mask = (t <= pos[:, None]) & (t > pos[:, None] - W)
                ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k[None], v[None],
                                                     attn_mask=mask[None, None], scale=0.3)[0]
                np.testing.assert_allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=1e-12,
                                           atol=1e-12)


def pin_window_extremes(orc):
    """A window at least as long as the context is no window; a window of 1 is the own V."""
    rng = np.random.default_rng(24)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        assert np.array_equal(_run(orc, c, 0.3), _run(orc, c, 0.3, window=max(ctxs) + 5))
        one = _run(orc, c, 0.3, window=1)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            for i in range(q_len):
                pos = ctx - q_len + i
                for h in range(n_q):
                    want = bf16_bits_to_f32(c["V"][b][h // G][pos]).astype(np.float64)
                    assert np.array_equal(one[b, i, h], want), (b, i, h)


def pin_prefill_sdpa(orc):
    """Many new tokens at once (a prefill chunk): torch SDPA with the causal mask of the
    chunk's positions, pure prefill (q_len = ctx) and chunked (q_len < ctx), with and
    without a window."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(29)
    for ctxs, n_q, n_kv, d, bs, q_len in [([40, 40], 8, 2, 16, 4, 40),
                                          ([33, 70, 21], 4, 4, 8, 8, 21),
                                          ([50, 25], 6, 1, 16, 16, 25)]:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        G = n_q // n_kv
        for W in (0, 7):
            got = _run(orc, c, 0.25, window=W)
            for b, ctx in enumerate(ctxs):
                q = torch.from_numpy(bf16_bits_to_f32(c["q"][b]).astype(np.float64))
                k = torch.from_numpy(bf16_bits_to_f32(c["K"][b]).astype(np.float64))
                v = torch.from_numpy(bf16_bits_to_f32(c["V"][b]).astype(np.float64))
                k, v = k.repeat_interleave(G, dim=0), v.repeat_interleave(G, dim=0)
                pos = ctx - q_len + torch.arange(q_len)
                t = torch.arange(ctx)[None, :]
                mask = t <= pos[:, None]
                if W:
                    mask &= t > pos[:, None] - W
                if q_len == ctx and not W:  # pure prefill: the library's own causal flag
                    ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k[None],
                                                         v[None], is_causal=True, scale=0.25)[0]
                else:
                    ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k[None],
                                                         v[None], attn_mask=mask[None, None],
                                                         scale=0.25)[0]
                np.testing.assert_allclose(got[b], ref.permute(1, 0, 2).numpy(), rtol=1e-12,
                                           atol=1e-12)


def pin_empty_context(orc):
    rng = np.random.default_rng(19)
    c = _case(rng, [0, 5, 0], 4, 2, 8, 4, 1)
    got = _run(orc, c, 0.5)
    assert np.all(got[0] == 0.0) and np.all(got[2] == 0.0)
    assert np.all(np.isfinite(got[1])) and np.any(got[1] != 0.0)


def pin_merge_exact(orc):
    rng = np.random.default_rng(20)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _case(rng, ctxs, n_q, n_kv, d, bs, q_len, kscale=3.0)
        full = _run(orc, c, 0.4)
        hi = max(ctxs)
        for nsplit in (1, 2, 3, 5):
            cuts = np.sort(rng.integers(0, hi + 1, size=nsplit - 1))
            edges = [0] + [int(x) for x in cuts] + [hi]
            parts = [orc.attn_partial(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                      c["context_lens"], n_q=n_q, n_kv=n_kv, head_dim=d,
                                      block_size=bs, scale=0.4, t_begin=a, t_end=b)
                     for a, b in zip(edges[:-1], edges[1:])]
            o = np.stack([p[0] for p in parts])
            m = np.stack([p[1] for p in parts])
            l = np.stack([p[2] for p in parts])
            merged = orc.lse_merge(o, m, l)
            np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)
        # the whole range as one part: o / l is the output, m the largest score
        o, m, l = orc.attn_partial(c["q"], c["k_cache"], c["v_cache"], c["block_tables"],
                                   c["context_lens"], n_q=n_q, n_kv=n_kv, head_dim=d,
                                   block_size=bs, scale=0.4, t_begin=0, t_end=hi)
        np.testing.assert_allclose(o / l[..., None], full, rtol=1e-12, atol=1e-13)
        G = n_q // n_kv
        for b, ctx in enumerate(ctxs):
            for i in range(q_len):
                nvis = ctx - q_len + i + 1
                for h in range(n_q):
                    q = bf16_bits_to_f32(c["q"][b, i, h]).astype(np.float64)
                    K = bf16_bits_to_f32(c["K"][b][h // G][:nvis]).astype(np.float64)
                    assert math.isclose(m[b, i, h], 0.4 * float((K @ q).max()),
                                        rel_tol=1e-12, abs_tol=1e-12)


def pin_kv_append(orc):
    rng = np.random.default_rng(21)
    for n_kv, d, bs, pool in [(2, 8, 4, 6), (1, 16, 16, 3), (4, 64, 16, 5)]:
        kc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
        vc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
        nslots = pool * bs
        slots = rng.permutation(nslots)[:7].astype(np.int32)
        slots = np.concatenate([slots, np.asarray([-1, nslots, nslots + 5, -100], np.int32)])
        rng.shuffle(slots)
        T = slots.shape[0]
        kn = rng.integers(0, 1 << 16, size=(T, n_kv, d), dtype=np.uint16)
        vn = rng.integers(0, 1 << 16, size=(T, n_kv, d), dtype=np.uint16)
        k_ref, v_ref = kc.copy(), vc.copy()
        for i, s in enumerate(slots):
            if 0 <= s < nslots:
                k_ref[s // bs, :, s % bs, :] = kn[i]
                v_ref[s // bs, :, s % bs, :] = vn[i]
        k_got, v_got = kc.copy(), vc.copy()
        orc.kv_append(kn, vn, slots, k_got, v_got, block_size=bs)
        assert np.array_equal(k_got, k_ref) and np.array_equal(v_got, v_ref)


def pin_copy_blocks(orc):
    rng = np.random.default_rng(22)
    pool, n_kv, bs, d = 9, 3, 4, 8
    kc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(pool, n_kv, bs, d), dtype=np.uint16)
    pairs = np.asarray([[1, 5], [2, 2], [0, 7], [3, 9], [-1, 4], [8, 6]], dtype=np.int32)
    k_ref, v_ref = kc.copy(), vc.copy()
    for src, dst in pairs:
        if 0 <= src < pool and 0 <= dst < pool and src != dst:
            k_ref[dst] = kc[src]
            v_ref[dst] = vc[src]
    k_got, v_got = kc.copy(), vc.copy()
    orc.copy_blocks(pairs, k_got, v_got)
    assert np.array_equal(k_got, k_ref) and np.array_equal(v_got, v_ref)


def pin_append_then_attend(orc):
    """The tiny workload: attend at ctx - 1, append one token, attend at ctx."""
    wl = make_custom(num_seqs=2, q_len=1, n_q=4, n_kv=2, head_dim=64, block_size=16,
                     context_lens=[18, 41], seed=99)
    kc, vc = wl.k_cache.copy(), wl.v_cache.copy()
    kw = dict(n_q=4, n_kv=2, head_dim=64, block_size=16, scale=wl.scale)
    before = orc.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens - 1, **kw)
    assert np.all(np.isfinite(before))  # the not-yet-written slot is never read
    orc.kv_append(wl.k_new, wl.v_new, wl.slot_mapping, kc, vc, block_size=16)
    after = orc.paged_attn(wl.q, kc, vc, wl.block_tables, wl.context_lens, **kw)
    assert np.all(np.isfinite(after))
    # With a huge scale the appended token wins whenever its score is the top one.
    for b in range(2):
        pos = int(wl.context_lens[b]) - 1
        blk = wl.block_tables[b, pos // 16]
        assert np.array_equal(kc[blk, :, pos % 16], wl.k_new[b])


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            p = line.split()
            rows.append((p[0], *[int(x) for x in p[1:7]]))
    return rows


def pin_kv_bytes_golden(orc):
    rows = _golden_rows()
    assert len(rows) >= 6
    for name, L, n_kv, d, p, tokens, expected in rows:
        assert orc.kv_bytes(L, n_kv, d, p, tokens) == expected, name


def pin_gqa_ratio(orc):
    # ("Inference Engines", The Mathematics: M_MHA / M_GQA = n_h / n_kv; MQA is n_kv = 1)
    for n_h, n_kv in [(32, 8), (64, 8), (32, 1), (40, 8)]:
        mha = orc.kv_bytes(32, n_h, 128, 2, 4096)
        gqa = orc.kv_bytes(32, n_kv, 128, 2, 4096)
        assert mha * n_kv == gqa * n_h


# ---------------------------------------------------------------------------
# 8-bit (e4m3) KV cache
# ---------------------------------------------------------------------------
E4M3_NAN = 0x7F


def _torch_e4m3(x):
    """torch's fp32 -> float8_e4m3fn codes (round to nearest even)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_value(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_e4m3_decode_library(orc):
    codes = np.arange(256, dtype=np.uint8)
    got, ref = orc.e4m3_decode(codes), _torch_e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got[E4M3_NAN]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def pin_e4m3_encode_library(orc):
    rng = np.random.default_rng(41)
    vals = _torch_e4m3_value(np.arange(256, dtype=np.uint8))
    pos = np.unique(vals[(vals >= 0) & np.isfinite(vals)])      # 0 .. 448, increasing
    mids = (pos[:-1] + pos[1:]) / 2                               # exact ties (fp32-exact)
    tests = [pos, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
             np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
             np.asarray([2.0 ** -10, 2.0 ** -10 * 1.0000001, 2.0 ** -11, 1e-30, 0.0, 464.0])]
    for e in range(-12, 9):
        tests.append(np.abs(rng.standard_normal(2000)) * 2.0 ** e)
    x = np.concatenate([t.astype(np.float32).ravel() for t in tests])
    x = x[x <= 464.0]
    x = np.concatenate([x, -x])
    got = orc.e4m3_encode(x)
    ref = _torch_e4m3(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), int(got[i]), int(ref[i])) for i in bad[:5]]


def pin_e4m3_saturation(orc):
    big = np.asarray([448.0, 455.0, 464.0, 464.01, 479.9, 480.0, 1e6, 3.0e38, np.inf],
                     dtype=np.float32)
    assert np.all(orc.e4m3_encode(big) == 0x7E)
    assert np.all(orc.e4m3_encode(-big) == 0xFE)
    assert orc.e4m3_encode(np.asarray([np.nan], np.float32))[0] == E4M3_NAN
    codes = np.asarray([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(orc.e4m3_encode(orc.e4m3_decode(codes).astype(np.float32)), codes)


def _fp8_case(rng, ctxs, n_q, n_kv, d, bs, q_len):
    finite = np.asarray([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    K = [rng.choice(finite, size=(n_kv, c, d)).astype(np.uint8) for c in ctxs]
    V = [rng.choice(finite, size=(n_kv, c, d)).astype(np.uint8) for c in ctxs]
    kc, vc, bt = _paged_from_logical(rng, K, V, bs, poison=E4M3_NAN)
    # the 8-bit cache keeps each (block, head)'s K rows, then its V rows
    kv = np.ascontiguousarray(np.stack([kc, vc], axis=2))
    q = _rand_bf16(rng, (len(ctxs), q_len, n_q, d))
    ks = rng.uniform(0.002, 0.05, n_kv).astype(np.float32)
    vs = rng.uniform(0.002, 0.05, n_kv).astype(np.float32)
    return dict(q=q, K=K, V=V, kv_cache=kv, block_tables=bt, ks=ks, vs=vs,
                context_lens=np.asarray(ctxs, dtype=np.int32))


def pin_fp8_attention_sdpa(orc):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(43)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _fp8_case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        G = n_q // n_kv
        for window in (0, 5):
            got = orc.paged_attn_fp8(c["q"], c["kv_cache"], c["ks"], c["vs"],
                                     c["block_tables"], c["context_lens"], n_q=n_q, n_kv=n_kv,
                                     head_dim=d, block_size=bs, scale=0.2, window=window)
            for b, ctx in enumerate(ctxs):
                q = torch.from_numpy(bf16_bits_to_f32(c["q"][b]).astype(np.float64))
                k = torch.from_numpy(_torch_e4m3_value(c["K"][b]) *
                                     c["ks"].astype(np.float64)[:, None, None])
                v = torch.from_numpy(_torch_e4m3_value(c["V"][b]) *
                                     c["vs"].astype(np.float64)[:, None, None])
                k, v = k.repeat_interleave(G, dim=0), v.repeat_interleave(G, dim=0)
                pos = ctx - q_len + torch.arange(q_len)
                t = torch.arange(ctx)[None, :]
                mask = t <= pos[:, None]
                if window:
                    mask &= t > pos[:, None] - window
                ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k[None], v[None],
                                                     attn_mask=mask[None, None], scale=0.2)[0]
                ref = ref.permute(1, 0, 2).numpy()
                rows_seen = mask.any(dim=1).numpy()
                np.testing.assert_allclose(got[b][rows_seen], ref[rows_seen], rtol=1e-12,
                                           atol=1e-12)


def pin_kv_append_fp8(orc):
    rng = np.random.default_rng(44)
    for n_kv, d, bs, pool in [(2, 8, 4, 6), (4, 64, 16, 5)]:
        kv = rng.integers(0, 256, size=(pool, n_kv, 2, bs, d), dtype=np.uint8)
        nslots = pool * bs
        slots = np.concatenate([rng.permutation(nslots)[:7].astype(np.int32),
                                np.asarray([-1, nslots], np.int32)])
        T = slots.shape[0]
        kn = _rand_bf16(rng, (T, n_kv, d), 3.0)
        vn = _rand_bf16(rng, (T, n_kv, d), 3.0)
        kn[0, 0, :4] = f32_to_bf16_bits(np.asarray([1e4, -1e4, 0.0, -0.0], np.float32))
        ks = rng.uniform(0.005, 0.05, n_kv).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, n_kv).astype(np.float32)

        def expect(x_bits, scale):
            xq = bf16_bits_to_f32(x_bits).astype(np.float32) / scale[:, None]  # fp32 division
            codes = _torch_e4m3(np.clip(xq, np.float32(-464.0), np.float32(464.0)))
            codes = np.where(np.abs(xq) > 464.0, np.where(xq < 0, 0xFE, 0x7E), codes)
            return codes.astype(np.uint8)

        ref = kv.copy()
        for i, sl in enumerate(slots):
            if 0 <= sl < nslots:
                ref[sl // bs, :, 0, sl % bs, :] = expect(kn[i], ks)
                ref[sl // bs, :, 1, sl % bs, :] = expect(vn[i], vs)
        got = kv.copy()
        orc.kv_append_fp8(kn, vn, slots, got, ks, vs, block_size=bs)
        assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# 8-bit cache with one scale per (block, KV head)
# ---------------------------------------------------------------------------
def _fp8_block_case(rng, ctxs, n_q, n_kv, d, bs, q_len):
    """Codes as in _fp8_case, plus a K and a V scale per logical block of every sequence,
    placed into the physical scale tensor by the test; unused blocks get NaN scales."""
    c = _fp8_case(rng, ctxs, n_q, n_kv, d, bs, q_len)
    pool = c["kv_cache"].shape[0]
    scales = np.full((pool, n_kv, 4), np.nan, dtype=np.float32)
    logical = []  # per sequence: [n_kv][nblocks][2] scales
    for b, ctx in enumerate(ctxs):
        nb = math.ceil(ctx / bs)
        ls = rng.uniform(0.001, 0.08, size=(n_kv, nb, 2)).astype(np.float32)
        logical.append(ls)
        for j in range(nb):
            scales[c["block_tables"][b, j], :, 0:2] = ls[:, j, :]
            scales[c["block_tables"][b, j], :, 2:4] = 0.0
    c["scales"], c["logical_scales"] = scales, logical
    return c


def pin_fp8_block_attention_sdpa(orc):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(47)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES:
        c = _fp8_block_case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        G = n_q // n_kv
        for window in (0, 5):
            got = orc.paged_attn_fp8_block(c["q"], c["kv_cache"], c["scales"],
                                           c["block_tables"], c["context_lens"], n_q=n_q,
                                           n_kv=n_kv, head_dim=d, block_size=bs, scale=0.2,
                                           window=window)
            for b, ctx in enumerate(ctxs):
                ls = c["logical_scales"][b].astype(np.float64)      # [n_kv][nb][2]
                tok = np.arange(ctx) // bs                           # logical block of token t
                q = torch.from_numpy(bf16_bits_to_f32(c["q"][b]).astype(np.float64))
                k = torch.from_numpy(_torch_e4m3_value(c["K"][b]) * ls[:, tok, 0][:, :, None])
                v = torch.from_numpy(_torch_e4m3_value(c["V"][b]) * ls[:, tok, 1][:, :, None])
                k, v = k.repeat_interleave(G, dim=0), v.repeat_interleave(G, dim=0)
                pos = ctx - q_len + torch.arange(q_len)
                t = torch.arange(ctx)[None, :]
                mask = t <= pos[:, None]
                if window:
                    mask &= t > pos[:, None] - window
                ref = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k[None], v[None],
                                                     attn_mask=mask[None, None], scale=0.2)[0]
                ref = ref.permute(1, 0, 2).numpy()
                rows_seen = mask.any(dim=1).numpy()
                np.testing.assert_allclose(got[b][rows_seen], ref[rows_seen], rtol=1e-12,
                                           atol=1e-12)


def pin_fp8_block_equals_per_head(orc):
    rng = np.random.default_rng(48)
    for ctxs, n_q, n_kv, d, bs, q_len in SHAPES[:4]:
        c = _fp8_case(rng, ctxs, n_q, n_kv, d, bs, q_len)
        pool = c["kv_cache"].shape[0]
        scales = np.zeros((pool, n_kv, 4), dtype=np.float32)
        scales[:, :, 0], scales[:, :, 1] = c["ks"][None, :], c["vs"][None, :]
        kw = dict(n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs, scale=0.3)
        a = orc.paged_attn_fp8_block(c["q"], c["kv_cache"], scales, c["block_tables"],
                                     c["context_lens"], **kw)
        b = orc.paged_attn_fp8(c["q"], c["kv_cache"], c["ks"], c["vs"], c["block_tables"],
                               c["context_lens"], **kw)
        assert np.array_equal(a, b)


def _pow2_exponent(x):
    """e with x == 2^e exactly, or None."""
    m, e = math.frexp(float(x))
    return e - 1 if m == 0.5 else None


def _check_block_scale(s, rows_f32):
    """The stored scale of a block whose new values are rows_f32 (no resident rows)."""
    fin = rows_f32[np.isfinite(rows_f32)]
    a = float(np.abs(fin).max()) if fin.size else 0.0
    if a == 0.0:
        assert s == 0.0, s
        return
    e = _pow2_exponent(s)
    assert e is not None and e >= -126, s
    assert a <= 448.0 * s, (a, s)                        # nothing saturates ...
    assert e == -126 or a > 224.0 * s, (a, s)            # ... and half the scale would


def pin_fp8_block_append_fresh(orc):
    rng = np.random.default_rng(49)
    n_kv, d, bs, pool = 2, 16, 4, 6
    kv = rng.integers(0, 256, size=(pool, n_kv, 2, bs, d), dtype=np.uint8)
    scales = rng.uniform(1.0, 5.0, size=(pool, n_kv, 4)).astype(np.float32)  # stale entries
    # block 1 gets offsets 0..2 (a run), block 4 offset 0 with all-zero rows, block 3
    # offset 0 with non-finite values and tiny ones; -1 and out-of-range slots skipped
    slots = np.asarray([4, 5, 6, -1, 16, 12, pool * bs], dtype=np.int32)
    T = slots.shape[0]
    kx = rng.standard_normal((T, n_kv, d)).astype(np.float32) * np.float32(3.0)
    vx = rng.standard_normal((T, n_kv, d)).astype(np.float32) * np.float32(0.01)
    kx[4], vx[4] = 0.0, -0.0
    kx[5, 0, :4] = [np.nan, np.inf, -np.inf, 1e-3]
    kx[5, 1] = np.float32(2.0 ** -135)
    kn, vn = f32_to_bf16_bits(kx), f32_to_bf16_bits(vx)
    kn[5, 0, 0] = 0x7FC0
    got_kv, got_sc = kv.copy(), scales.copy()
    orc.kv_append_fp8_block(kn, vn, slots, got_kv, got_sc, block_size=bs)
    touched = {1: [0, 1, 2], 4: [4], 3: [5]}
    for blk, toks in touched.items():
        for g in range(n_kv):
            for which, bits in ((0, kn), (1, vn)):
                x = bf16_bits_to_f32(bits[toks, g, :])
                s = float(got_sc[blk, g, which])
                _check_block_scale(s, x)
                q = x / np.float32(s) if s > 0 else x               # fp32 division
                want = _torch_e4m3(np.clip(q, np.float32(-464.0), np.float32(464.0)))
                want = np.where(np.isinf(q), np.where(q < 0, 0xFE, 0x7E), want)
                want = np.where(np.isnan(q), 0x7F, want)
                offs = [int(slots[t]) % bs for t in toks]
                assert np.array_equal(got_kv[blk, g, which, offs], want.astype(np.uint8)), \
                    (blk, g, which)
            assert got_sc[blk, g, 2] == 0.0 and got_sc[blk, g, 3] == 0.0
    assert got_sc[4, 0, 0] == 0.0 and got_sc[4, 1, 1] == 0.0   # all zeros: scale 0
    # untouched blocks and the untouched rows of touched blocks keep their bytes
    for blk in range(pool):
        if blk not in touched:
            assert np.array_equal(got_kv[blk], kv[blk]) and np.array_equal(got_sc[blk], scales[blk])
    assert np.array_equal(got_kv[1, :, :, 3], kv[1, :, :, 3])
    assert np.array_equal(got_kv[4, :, :, 1:], kv[4, :, :, 1:])


def pin_fp8_block_append_growth(orc):
    rng = np.random.default_rng(50)
    n_kv, d, bs, pool = 2, 32, 8, 3
    finite = np.asarray([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for k in (1, 3, 9):
        kv = rng.choice(finite, size=(pool, n_kv, 2, bs, d)).astype(np.uint8)
        s_old = np.float32(2.0 ** -6)
        scales = np.zeros((pool, n_kv, 4), dtype=np.float32)
        scales[:, :, 0:2] = s_old
        # block 2 holds 3 resident rows; the new token at offset 3 needs 2^k times the range
        x = rng.standard_normal((1, n_kv, d)).astype(np.float32)
        x *= np.float32(448.0 * float(s_old) * 2.0 ** k * 0.9) / np.abs(x).max(axis=2, keepdims=True)
        slots = np.asarray([2 * bs + 3], dtype=np.int32)
        kn = vn = f32_to_bf16_bits(x)
        got_kv, got_sc = kv.copy(), scales.copy()
        orc.kv_append_fp8_block(kn, vn, slots, got_kv, got_sc, block_size=bs)
        for g in range(n_kv):
            for which in (0, 1):
                s_new = float(got_sc[2, g, which])
                assert s_new == float(s_old) * 2.0 ** k, (k, s_new)
                old_v = _torch_e4m3_value(kv[2, g, which, :3]) * float(s_old)
                new_v = _torch_e4m3_value(got_kv[2, g, which, :3]) * s_new
                normal = np.abs(old_v) >= 2.0 ** -6 * s_new
                assert np.array_equal(new_v[normal], old_v[normal]), (k, g, which)
                assert np.all(np.abs(new_v - old_v) <= 2.0 ** -10 * s_new), (k, g, which)
                # rows past the new token are not resident: untouched
                assert np.array_equal(got_kv[2, g, which, 4:], kv[2, g, which, 4:])
        assert np.array_equal(got_kv[:2], kv[:2]) and np.array_equal(got_sc[:2], scales[:2])
    # smaller values: the scale and the resident rows stay
    kv = rng.choice(finite, size=(pool, n_kv, 2, bs, d)).astype(np.uint8)
    scales = np.full((pool, n_kv, 4), 2.0 ** -3, dtype=np.float32)
    small = f32_to_bf16_bits(rng.standard_normal((1, n_kv, d)).astype(np.float32) * 1e-3)
    got_kv, got_sc = kv.copy(), scales.copy()
    orc.kv_append_fp8_block(small, small, np.asarray([bs + 5], np.int32), got_kv, got_sc,
                            block_size=bs)
    assert np.all(got_sc[1, :, 0:2] == np.float32(2.0 ** -3))
    assert np.array_equal(got_kv[1, :, :, :5], kv[1, :, :, :5])
    assert np.array_equal(got_kv[1, :, :, 6:], kv[1, :, :, 6:])


def pin_fp8_block_append_then_attend(orc):
    """Rows appended one decode step at a time through the block scales, then attended over:
    within the e4m3 rounding (relative 2^-4 per value) of attention over the bf16 rows."""
    rng = np.random.default_rng(51)
    n_q, n_kv, d, bs = 4, 2, 16, 4
    ctxs = [3, 9, 14]
    pool = 12
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.zeros((len(ctxs), 4), dtype=np.int32)
    o = 0
    for b, c in enumerate(ctxs):
        nb = math.ceil(c / bs)
        bt[b, :nb] = perm[o:o + nb]
        bt[b, nb:] = perm[-1]
        o += nb
    kv = np.full((pool, n_kv, 2, bs, d), E4M3_NAN, dtype=np.uint8)
    sc = np.full((pool, n_kv, 4), np.nan, dtype=np.float32)
    k16 = np.full((pool, n_kv, bs, d), BF16_POISON, dtype=np.uint16)
    v16 = np.full_like(k16, BF16_POISON)
    for t in range(max(ctxs)):                     # one token per live sequence per step
        live = [b for b, c in enumerate(ctxs) if t < c]
        slots = np.asarray([bt[b, t // bs] * bs + t % bs for b in live], dtype=np.int32)
        growth = np.float32(2.0 ** (t % 5))        # values that grow and shrink over time
        kn = _rand_bf16(rng, (len(live), n_kv, d), growth)
        vn = _rand_bf16(rng, (len(live), n_kv, d), 4.0 / growth)
        orc.kv_append_fp8_block(kn, vn, slots, kv, sc, block_size=bs)
        orc.kv_append(kn, vn, slots, k16, v16, block_size=bs)
    q = _rand_bf16(rng, (len(ctxs), 1, n_q, d), 0.3)
    kw = dict(n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs, scale=0.25)
    got = orc.paged_attn_fp8_block(q, kv, sc, bt, np.asarray(ctxs, np.int32), **kw)
    ref = orc.paged_attn(q, k16, v16, bt, np.asarray(ctxs, np.int32), **kw)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= 0.25 * np.abs(ref) + 0.25), float(err.max())
    assert np.mean(err) < 0.1, float(np.mean(err))


ALL_PINS = [
    pin_library_sdpa, pin_numpy_dense, pin_equal_scores_mean, pin_single_token, pin_hardmax,
    pin_block_permutation, pin_gqa_equals_repeated_mha, pin_causal_rows, pin_window_sdpa,
    pin_window_extremes, pin_prefill_sdpa, pin_empty_context,
    pin_merge_exact, pin_kv_append, pin_copy_blocks, pin_append_then_attend, pin_kv_bytes_golden,
    pin_gqa_ratio, pin_e4m3_decode_library, pin_e4m3_encode_library, pin_e4m3_saturation,
    pin_fp8_attention_sdpa, pin_kv_append_fp8, pin_fp8_block_attention_sdpa,
    pin_fp8_block_equals_per_head, pin_fp8_block_append_fresh, pin_fp8_block_append_growth,
    pin_fp8_block_append_then_attend,
]
