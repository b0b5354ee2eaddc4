"""Host-side block pool: allocation, sharing, release and copy-on-write (CPU only)."""
import numpy as np
import pytest

import paged_kv_cache_256_gb300 as pkv


def test_alloc_release_counts():
    p = pkv.BlockPool(10, 16)
    assert p.num_free() == 10
    a = p.alloc(4)
    assert len(set(a.tolist())) == 4 and p.num_free() == 6
    assert all(p.refcount(int(b)) == 1 for b in a)
    p.release(a[:2])
    assert p.num_free() == 8 and p.refcount(int(a[0])) == 0
    with pytest.raises(pkv.PkvError) as e:
        p.alloc(9)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS and p.num_free() == 8


def test_share_and_release_are_all_or_nothing():
    p = pkv.BlockPool(6, 16)
    a = p.alloc(3)
    p.share(a)
    assert [p.refcount(int(b)) for b in a] == [2, 2, 2]
    with pytest.raises(pkv.PkvError):  # a free block cannot be shared
        p.share(np.asarray([a[0], 5], dtype=np.int32))
    assert p.refcount(int(a[0])) == 2
    with pytest.raises(pkv.PkvError):  # three drops of a block held twice
        p.release(np.asarray([a[1], a[1], a[1]], dtype=np.int32))
    assert p.refcount(int(a[1])) == 2
    p.release(np.concatenate([a, a]))
    assert p.num_free() == 6


def test_append_to_fresh_sequence():
    p = pkv.BlockPool(8, 16)
    table = np.full(4, -1, dtype=np.int32)
    nb, slots, pairs = p.append_slots(table, 0, 0, 20)
    assert nb == 2 and pairs.shape == (0, 2)
    assert slots.tolist() == [table[0] * 16 + i for i in range(16)] + \
        [table[1] * 16 + i for i in range(4)]


def test_fork_then_append_copies_only_the_shared_partial_block():
    p = pkv.BlockPool(16, 16)
    a = np.full(8, -1, dtype=np.int32)
    nb, _, _ = p.append_slots(a, 0, 0, 40)           # 40 tokens: blocks 0, 1 full, 2 partial
    assert nb == 3
    b = a.copy()
    p.share(b[:nb])                                   # fork: B shares all of A's blocks
    nb_a, slots_a, pairs_a = p.append_slots(a, nb, 40, 1)
    assert pairs_a.tolist() == [[b[2], a[2]]]         # only the partial block is copied
    assert a[0] == b[0] and a[1] == b[1] and a[2] != b[2]
    assert slots_a.tolist() == [a[2] * 16 + 8]
    assert p.refcount(int(b[2])) == 1 and p.refcount(int(a[2])) == 1
    nb_b, slots_b, pairs_b = p.append_slots(b, nb, 40, 1)
    assert pairs_b.shape == (0, 2)                    # B is now sole owner of its block
    assert slots_b.tolist() == [b[2] * 16 + 8]
    assert p.refcount(int(a[0])) == 2                 # the full prefix blocks stay shared


def test_append_at_block_boundary_needs_no_copy():
    p = pkv.BlockPool(8, 16)
    a = np.full(4, -1, dtype=np.int32)
    nb, _, _ = p.append_slots(a, 0, 0, 32)
    b = a.copy()
    p.share(b[:nb])
    nb2, slots, pairs = p.append_slots(a, nb, 32, 3)
    assert pairs.shape == (0, 2) and nb2 == 3
    assert slots.tolist() == [a[2] * 16 + i for i in range(3)]


def test_failure_changes_nothing():
    p = pkv.BlockPool(3, 16)
    a = np.full(4, -1, dtype=np.int32)
    nb, _, _ = p.append_slots(a, 0, 0, 20)            # 2 blocks
    b = a.copy()
    p.share(b[:nb])
    before = (p.num_free(), a.copy(), [p.refcount(i) for i in range(3)])
    with pytest.raises(pkv.PkvError) as e:            # needs 1 copy + 2 new, only 1 free
        p.append_slots(a, nb, 20, 40)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert p.num_free() == before[0] and np.array_equal(a, before[1])
    assert [p.refcount(i) for i in range(3)] == before[2]
    with pytest.raises(pkv.PkvError):                 # table too short for the context
        p.append_slots(a, 1, 20, 1)


def test_random_operations_keep_the_invariants():
    """Model-based: random forks, appends and releases against a python model."""
    rng = np.random.default_rng(5)
    bs, pool_n, max_blocks = 4, 64, 32
    p = pkv.BlockPool(pool_n, bs)
    seqs = []  # [table, nblocks, ctx]
    owner_count = np.zeros(pool_n, dtype=np.int64)
    for step in range(400):
        op = rng.integers(0, 4)
        if op == 0 or not seqs:                       # new sequence
            t = np.full(max_blocks, -1, dtype=np.int32)
            n = int(rng.integers(1, 12))
            try:
                nb, slots, pairs = p.append_slots(t, 0, 0, n)
            except pkv.PkvError:
                continue
            seqs.append([t, nb, n])
        elif op == 1:                                 # fork
            src = seqs[int(rng.integers(len(seqs)))]
            t = src[0].copy()
            p.share(t[: src[1]])
            seqs.append([t, src[1], src[2]])
        elif op == 2:                                 # append to a sequence
            s = seqs[int(rng.integers(len(seqs)))]
            n = int(rng.integers(1, 6))
            if s[2] + n > max_blocks * bs:
                continue
            try:
                nb, slots, pairs = p.append_slots(s[0], s[1], s[2], n)
            except pkv.PkvError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
                continue
            # every block written is now owned by this sequence alone
            for sl in slots:
                assert p.refcount(int(sl // bs)) == 1
            s[1], s[2] = nb, s[2] + n
        else:                                         # release a sequence
            s = seqs.pop(int(rng.integers(len(seqs))))
            p.release(s[0][: s[1]])
        # reference counts equal the number of tables holding each block
        owner_count[:] = 0
        for t, nb, ctx in seqs:
            for b in t[:nb]:
                owner_count[b] += 1
        assert [p.refcount(i) for i in range(pool_n)] == owner_count.tolist()
        assert p.num_free() == int((owner_count == 0).sum())
