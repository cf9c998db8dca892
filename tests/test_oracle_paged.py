"""Pins of the oracle's page allocator (oracle/paged.py).

Self-speculative decoding page (m.lqnn.cn/news/278124) §3.3: a rollback is
page-granular and the write pointer equals the sequence length, so after
every commit a sequence holds exactly the pages that cover its committed
slots; §4.5: each sequence of a batch keeps its own offsets.  A hand-worked
table fixes the order in which pages are taken and given back; random rounds
check the invariants (page count ceil(len / page), no page held twice, the
free count completes the pool).
"""
import numpy as np
import pytest

from oracle.paged import PagePool, PoolExhausted


def test_hand_table():
    # batch 2, 16 slots each, pages of 4 slots, a pool of 5 pages
    pool = PagePool(batch=2, max_ctx=16, page=4, n_pages=5)
    assert pool.max_pages == 4 and pool.free_count() == 5
    pool.ensure([6, 3])                      # seq 0: blocks 0, 1; seq 1: block 0
    assert pool.table == [[0, 1, -1, -1], [2, -1, -1, -1]]
    assert pool.free == [4, 3]
    pool.release([2, 3])                     # seq 0 keeps 1 block: page 1 goes back on top
    assert pool.table == [[0, -1, -1, -1], [2, -1, -1, -1]]
    assert pool.free == [4, 3, 1]
    pool.ensure_relative([2, 3], [5, 5])     # ends 7 and 8: page 1 again, then page 3
    assert pool.table == [[0, 1, -1, -1], [2, 3, -1, -1]]
    assert pool.free == [4]
    pool.release([7, 4])                     # seq 1 keeps 1 block: page 3 back
    assert pool.table == [[0, 1, -1, -1], [2, -1, -1, -1]]
    assert pool.free == [4, 3]
    pool.ensure([12, 4])
    assert pool.table == [[0, 1, 3, -1], [2, -1, -1, -1]]
    with pytest.raises(PoolExhausted):
        pool.ensure([16, 16])                # seq 0 takes the last page, seq 1 finds none
    assert pool.table == [[0, 1, 3, 4], [2, -1, -1, -1]]
    assert pool.free == []
    assert pool.locate(0, 13) == (4, 1) and pool.locate(1, 5) == (-1, 1)


def test_exact_page_boundaries():
    pool = PagePool(batch=1, max_ctx=256, page=64, n_pages=4)
    for n, held in [(0, 0), (1, 1), (64, 1), (65, 2), (128, 2), (129, 3), (256, 4)]:
        pool.set_lengths([n])
        assert sum(p >= 0 for p in pool.table[0]) == held, n
    pool.set_lengths([0])
    assert pool.free_count() == 4 and pool.table == [[-1] * 4]


def test_end_past_capacity_is_an_error():
    pool = PagePool(batch=1, max_ctx=100, page=64, n_pages=8)
    with pytest.raises(ValueError):
        pool.ensure([129])
    assert pool.table == [[0, 1]]            # the blocks it could address were served


def _check(pool, lens):
    held = []
    for b, n in enumerate(lens):
        need = -(-n // pool.page)
        row = pool.table[b]
        assert all(p >= 0 for p in row[:need]) and all(p < 0 for p in row[need:]), (b, n, row)
        held += row[:need]
    assert len(set(held)) == len(held)
    assert sorted(held + pool.free) == list(range(pool.n_pages))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_chain_rounds_keep_the_invariants(seed):
    rng = np.random.default_rng(seed)
    B, page, k = 4, 64, 6
    lens = [int(x) for x in rng.integers(0, 300, size=B)]
    max_ctx = 1024
    need = sum(-(-(n + 60 * (k + 1)) // page) for n in lens)
    pool = PagePool(B, max_ctx, page, need)
    pool.set_lengths(lens)
    _check(pool, lens)
    for _ in range(60):
        pool.ensure_relative(lens, [k + 1] * B)          # draft and verify write k+1 slots
        for b in range(B):
            assert all(p >= 0 for p in pool.table[b][:-(-(lens[b] + k + 1) // page)])
        acc = [int(a) for a in rng.integers(0, k + 1, size=B)]
        lens = [n + a + 1 for n, a in zip(lens, acc)]    # commit: t0 plus the accepted drafts
        pool.release(lens)
        _check(pool, lens)
        if rng.random() < 0.1:                          # a rollback of some sequences
            lens = [int(rng.integers(0, n + 1)) for n in lens]
            pool.set_lengths(lens)
            _check(pool, lens)
