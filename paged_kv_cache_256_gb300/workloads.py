"""Seeded synthetic inputs for paged decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through its tests and the bench) and
the CPU oracle consume what it returns, so it imports nothing else from this
package and nothing from the oracle.

Every tensor is built on the host as numpy:

* ``q``            ``[num_seqs, q_len, n_q, head_dim]``          bf16 bits (uint16)
* ``k_cache``      ``[num_blocks, n_kv, block_size, head_dim]``  bf16 bits (uint16)
* ``v_cache``      same layout as ``k_cache``
* ``block_tables`` ``[num_seqs, max_blocks_per_seq]``             int32
* ``context_lens`` ``[num_seqs]``                                  int32
* ``k_new``/``v_new`` ``[num_seqs * q_len, n_kv, head_dim]``       bf16 bits
* ``slot_mapping`` ``[num_seqs * q_len]``                          int32

Conventions (the plain readings of the pages, "Inference Engines", The
Breakthrough, and "Transformer inference mechanics", What the KV cache stores
per layer):

* ``context_lens`` counts every resident token including the ``q_len`` new
  ones; the new tokens sit at logical positions ``ctx - q_len .. ctx - 1`` and
  ``slot_mapping`` points at exactly those cache slots.  Before ``kv_append``
  runs, those slots hold poison.
* Unused physical blocks, slots past ``ctx`` inside a sequence's last block,
  and the not-yet-appended slots are filled with a bf16 NaN, so any read that
  is used shows up as NaN in the output.
* Block-table entries past a sequence's last block point at a poison block
  (always a valid index, never out of range).
* Values: fp32 samples of N(0, 1) rounded to bf16 with round-to-nearest-even.

An 8-bit variant of any workload (:func:`fp8_cache_for`) draws e4m3 codes
directly -- random sign, exponent field 7 + round(N(0, 1.5)) clipped to
[1, 14], uniform mantissa -- into the same resident slots, with the e4m3 NaN
(0x7F) wherever the bf16 cache holds poison, and per-KV-head fp32 scales
drawn from U(0.05, 0.5).  No quantiser is involved: the codes are the data.
The 8-bit cache is one array ``[num_blocks, n_kv, 2, block_size, head_dim]``
holding each (block, KV head)'s K rows, then its V rows.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "BF16_POISON",
    "E4M3_POISON",
    "Fp8Cache",
    "fp8_cache_for",
    "fp8_block_scales_for",
    "CONFIGS",
    "Workload",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "make_workload",
    "make_custom",
]

# A quiet NaN with a payload, so poison is recognisable in a dump.
BF16_POISON = np.uint16(0x7FC1)
# The e4m3 NaN (S.1111.111).
E4M3_POISON = np.uint8(0x7F)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the bits.

    For every non-NaN input the 32-bit sum below cannot wrap (the largest
    finite pattern plus 0x8000 stays under 2**32); NaNs become BF16_POISON.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16))
    r = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = BF16_POISON
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    num_seqs: int
    q_len: int
    n_q: int
    n_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    scale: float  # an fp32 value, passed as-is to both sides
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    slot_mapping: np.ndarray
    description: str = ""

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv

    @property
    def num_tokens(self) -> int:
        return self.num_seqs * self.q_len

    def resident_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())


# The five workloads: name -> recipe.  ``ctx`` is either a list of lengths
# or a (kind, params) draw.  ``pool`` is the physical-block count, or None for
# "exactly the blocks in use" plus ``extra_poison`` poison blocks.
CONFIGS = {
    "tiny": dict(
        index=0, num_seqs=2, q_len=1, n_q=4, n_kv=2, head_dim=64, block_size=16,
        ctx=("fixed", [18, 41]), pool=8, extra_poison=0, k_head_scale=None,
        description="tiny paged decode: batch 2, ctx {17,40} then {18,41} after "
                    "appending one token per sequence, n_q 4, n_kv 2, d 64, bs 16, "
                    "8 physical blocks in a seeded permutation"),
    "llama2_7b_mha": dict(
        index=1, num_seqs=16, q_len=1, n_q=32, n_kv=32, head_dim=128, block_size=16,
        ctx=("fixed", [4096] * 16), pool=5000, extra_poison=0, k_head_scale=None,
        description="Llama-2-7B-shaped MHA decode layer: batch 16, ctx 4096, 32/32 heads, "
                    "d 128, bs 16, blocks shuffled from a 5000-block pool"),
    "llama3_8b_gqa": dict(
        index=2, num_seqs=64, q_len=1, n_q=32, n_kv=8, head_dim=128, block_size=16,
        ctx=("uniform", (128, 8192)), pool=None, extra_poison=64, k_head_scale=None,
        description="Llama-3-8B-shaped GQA continuous batch: batch 64, ctx uniform int "
                    "in [128, 8192], 32/8 heads, d 128, bs 16, blocks interleaved "
                    "across sequences in one shared pool"),
    "mqa_spec_verify": dict(
        index=3, num_seqs=128, q_len=4, n_q=32, n_kv=1, head_dim=128, block_size=32,
        ctx=("lognormal", (1024.0, 1.0, 16, 16384)), pool=None, extra_poison=64,
        k_head_scale=None,
        description="MQA speculative-verify step: batch 128, ctx lognormal (median 1024, "
                    "sigma 1, clipped to [16, 16384]), 32/1 heads, d 128, gamma=4 causal "
                    "draft tokens per sequence, bs 32"),
    "long_splitk": dict(
        index=4, num_seqs=4, q_len=1, n_q=64, n_kv=8, head_dim=128, block_size=16,
        ctx=("fixed", [131072] * 4), pool=None, extra_poison=16,
        k_head_scale=(0.5, 4.0),
        description="long-context split-K: batch 4, ctx 131072, 64/8 heads, d 128, bs 16, "
                    "shuffled blocks, K scaled per KV head by U(0.5, 4)"),
    "llama3_8b_chunked_prefill": dict(
        index=5, num_seqs=4, q_len=256, n_q=32, n_kv=8, head_dim=128, block_size=16,
        ctx=("uniform", (1024, 4096)), pool=None, extra_poison=16, k_head_scale=None,
        description="Llama-3-8B-shaped chunked prefill: batch 4, a 256-token chunk of each "
                    "prompt appended to a cached prefix (ctx uniform int in [1024, 4096] "
                    "including the chunk), 32/8 heads, d 128, bs 16: 1024 query rows per KV "
                    "head in 8 row tiles"),
}


def _normal_bf16(seed_seq: np.random.SeedSequence, shape, scale_per=None, chunk=1 << 23):
    """N(0,1) fp32 samples rounded to bf16 bits.

    The array is cut into fixed chunks; chunk c draws from the c-th child of
    ``seed_seq``, so the values depend only on the seed and the shape (not on
    the thread count).  ``scale_per(lo, hi)`` optionally multiplies the fp32
    samples of flat elements [lo, hi) before rounding.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + chunk - 1) // chunk
    kids = seed_seq.spawn(nchunks)

    def work(c):
        lo, hi = c * chunk, min(n, (c + 1) * chunk)
        x = np.random.Generator(np.random.PCG64(kids[c])).standard_normal(hi - lo, dtype=np.float32)
        if scale_per is not None:
            x *= scale_per(lo, hi)
        out[lo:hi] = f32_to_bf16_bits(x)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def _e4m3_codes(seed_seq: np.random.SeedSequence, n: int, chunk=1 << 23) -> np.ndarray:
    """n seeded e4m3 codes: sign, exponent field 7 + rint(N(0, 1.5)) in [1, 14], mantissa."""
    out = np.empty(n, dtype=np.uint8)
    nchunks = (n + chunk - 1) // chunk
    kids = seed_seq.spawn(max(nchunks, 1))

    def work(c):
        lo, hi = c * chunk, min(n, (c + 1) * chunk)
        g = np.random.Generator(np.random.PCG64(kids[c]))
        e = np.clip(np.rint(7.0 + 1.5 * g.standard_normal(hi - lo, dtype=np.float32)), 1, 14)
        bits = g.integers(0, 16, size=hi - lo, dtype=np.uint8)  # sign (bit 3) and mantissa
        out[lo:hi] = ((bits & 8) << 4) | (e.astype(np.uint8) << 3) | (bits & 7)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


@dataclasses.dataclass
class Fp8Cache:
    kv_cache: np.ndarray  # [num_blocks, n_kv, 2, block_size, head_dim] e4m3 codes (uint8)
    k_scale: np.ndarray   # [n_kv] float32: value of code c in head g = c * k_scale[g]
    v_scale: np.ndarray


def fp8_cache_for(wl: Workload, seed: int | None = None) -> Fp8Cache:
    """Seeded e4m3 caches laid out like ``wl``'s (same resident and poison slots)."""
    if seed is None:
        seed = 5000 + sum(wl.name.encode())
    s_k, s_v, s_s = np.random.SeedSequence([seed, 11]).spawn(3)
    n = wl.k_cache.size
    k8 = _e4m3_codes(s_k, n).reshape(wl.k_cache.shape)
    v8 = _e4m3_codes(s_v, n).reshape(wl.v_cache.shape)
    k8[wl.k_cache == BF16_POISON] = E4M3_POISON
    v8[wl.v_cache == BF16_POISON] = E4M3_POISON
    r = np.random.Generator(np.random.PCG64(s_s))
    ks = r.uniform(0.05, 0.5, size=wl.n_kv).astype(np.float32)
    vs = r.uniform(0.05, 0.5, size=wl.n_kv).astype(np.float32)
    kv = np.ascontiguousarray(np.stack([k8, v8], axis=2))
    return Fp8Cache(kv_cache=kv, k_scale=ks, v_scale=vs)


def fp8_block_scales_for(wl: Workload, seed: int | None = None) -> np.ndarray:
    """Seeded per-(block, KV head) scales [num_blocks, n_kv, 4] float32 for an 8-bit cache:
    a K and a V scale per block, powers of two 2^k with k uniform in [-8, -3], then two
    zero words."""
    if seed is None:
        seed = 7000 + sum(wl.name.encode())
    r = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 13])))
    sc = np.zeros((wl.num_blocks, wl.n_kv, 4), dtype=np.float32)
    sc[:, :, 0:2] = np.ldexp(np.float32(1.0), r.integers(-8, -2, size=(wl.num_blocks, wl.n_kv, 2)))
    return sc


def _draw_context_lens(rng, spec, num_seqs):
    kind, p = spec
    if kind == "fixed":
        return np.asarray(p, dtype=np.int32)
    if kind == "uniform":
        lo, hi = p
        return rng.integers(lo, hi + 1, size=num_seqs, dtype=np.int64).astype(np.int32)
    if kind == "lognormal":
        median, sigma, lo, hi = p
        x = rng.lognormal(mean=math.log(median), sigma=sigma, size=num_seqs)
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    raise ValueError(kind)


def _build(name, *, num_seqs, q_len, n_q, n_kv, head_dim, block_size, context_lens,
           pool, extra_poison, k_head_scale, seed, description="", max_blocks_per_seq=None):
    ss = np.random.SeedSequence(seed)
    s_perm, s_q, s_k, s_v, s_kn, s_vn, s_hs = ss.spawn(7)
    r_perm = np.random.Generator(np.random.PCG64(s_perm))
    r_hs = np.random.Generator(np.random.PCG64(s_hs))
    context_lens = np.asarray(context_lens, dtype=np.int32)
    assert context_lens.shape == (num_seqs,)
    nblk = (context_lens.astype(np.int64) + block_size - 1) // block_size
    used = int(nblk.sum())
    if pool is None:
        pool = used + extra_poison
    # At least one poison block is needed as the target of block-table padding.
    pool = max(pool, used + 1)
    if max_blocks_per_seq is None:
        max_blocks_per_seq = int(max(1, nblk.max(initial=1)))
    perm = r_perm.permutation(pool).astype(np.int32)
    poison_block = int(perm[used]) if used < pool else int(perm[-1])

    block_tables = np.full((num_seqs, max_blocks_per_seq), poison_block, dtype=np.int32)
    off = 0
    for b in range(num_seqs):
        block_tables[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += nblk[b]

    kv_shape = (pool, n_kv, block_size, head_dim)
    k_scale_fn = None
    if k_head_scale is not None:
        s = r_hs.uniform(k_head_scale[0], k_head_scale[1], size=n_kv).astype(np.float32)
        per_head = block_size * head_dim
        # element index e -> head (e // per_head) % n_kv
        def k_scale_fn(lo, hi, s=s):
            idx = np.arange(lo, hi, dtype=np.int64)
            return s[(idx // per_head) % n_kv]
    k_cache = _normal_bf16(s_k, kv_shape, k_scale_fn)
    v_cache = _normal_bf16(s_v, kv_shape)

    # Poison: every block not in use; slots at or past ctx in the last block;
    # the q_len slots the append will fill.
    in_use = np.zeros(pool, dtype=bool)
    in_use[perm[:used]] = True
    k_cache[~in_use] = BF16_POISON
    v_cache[~in_use] = BF16_POISON
    slot_mapping = np.empty(num_seqs * q_len, dtype=np.int32)
    for b in range(num_seqs):
        ctx = int(context_lens[b])
        if nblk[b] > 0:
            last = block_tables[b, nblk[b] - 1]
            tail = ctx - (nblk[b] - 1) * block_size
            k_cache[last, :, tail:, :] = BF16_POISON
            v_cache[last, :, tail:, :] = BF16_POISON
        for i in range(q_len):
            pos = ctx - q_len + i
            if pos < 0:
                slot_mapping[b * q_len + i] = -1
                continue
            blk = block_tables[b, pos // block_size]
            slot_mapping[b * q_len + i] = blk * block_size + pos % block_size
            k_cache[blk, :, pos % block_size, :] = BF16_POISON
            v_cache[blk, :, pos % block_size, :] = BF16_POISON

    q = _normal_bf16(s_q, (num_seqs, q_len, n_q, head_dim))
    kn_scale_fn = None
    if k_head_scale is not None:
        def kn_scale_fn(lo, hi, s=s):
            idx = np.arange(lo, hi, dtype=np.int64)
            return s[(idx // head_dim) % n_kv]
    k_new = _normal_bf16(s_kn, (num_seqs * q_len, n_kv, head_dim), kn_scale_fn)
    v_new = _normal_bf16(s_vn, (num_seqs * q_len, n_kv, head_dim))
    scale = float(np.float32(1.0 / math.sqrt(head_dim)))
    return Workload(name=name, num_seqs=num_seqs, q_len=q_len, n_q=n_q, n_kv=n_kv,
                    head_dim=head_dim, block_size=block_size, num_blocks=pool,
                    max_blocks_per_seq=max_blocks_per_seq, scale=scale, q=q,
                    k_cache=k_cache, v_cache=v_cache, block_tables=block_tables,
                    context_lens=context_lens, k_new=k_new, v_new=v_new,
                    slot_mapping=slot_mapping, description=description)


def make_workload(name: str, seed: int | None = None) -> Workload:
    """Build one of the five named workloads; seed defaults to 1000 + its index."""
    c = CONFIGS[name]
    if seed is None:
        seed = 1000 + c["index"]
    ss = np.random.SeedSequence([seed, 7])
    r_ctx = np.random.Generator(np.random.PCG64(ss))
    ctx = _draw_context_lens(r_ctx, c["ctx"], c["num_seqs"])
    max_blocks = None
    if c["ctx"][0] == "uniform":
        max_blocks = (c["ctx"][1][1] + c["block_size"] - 1) // c["block_size"]
    elif c["ctx"][0] == "lognormal":
        max_blocks = (c["ctx"][1][3] + c["block_size"] - 1) // c["block_size"]
    return _build(name, num_seqs=c["num_seqs"], q_len=c["q_len"], n_q=c["n_q"],
                  n_kv=c["n_kv"], head_dim=c["head_dim"], block_size=c["block_size"],
                  context_lens=ctx, pool=c["pool"], extra_poison=c["extra_poison"],
                  k_head_scale=c["k_head_scale"], seed=seed,
                  description=c["description"], max_blocks_per_seq=max_blocks)


def make_custom(*, num_seqs, q_len, n_q, n_kv, head_dim, block_size, context_lens,
                seed, extra_poison=3, max_blocks_per_seq=None, k_head_scale=None,
                name="custom") -> Workload:
    """A workload of any shape, for edge cases and small parity sizes."""
    return _build(name, num_seqs=num_seqs, q_len=q_len, n_q=n_q, n_kv=n_kv,
                  head_dim=head_dim, block_size=block_size, context_lens=context_lens,
                  pool=None, extra_poison=extra_poison, k_head_scale=k_head_scale,
                  seed=seed, max_blocks_per_seq=max_blocks_per_seq)
