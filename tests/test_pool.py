"""The page pool behind prefix sharing (host logic, no GPU): reference
counts, exhaustion, misuse, copy-on-write on append, and a randomized run
checked against the invariant that defines the pool -- a page's count is
the number of block-table entries that point to it, and a page is free
exactly when its count is 0."""
import random
import threading

import numpy as np
import pytest

import paged_kv_cache_171_gb300 as pa
from paged_kv_cache_171_gb300 import build as pa_build

EMPTY, STATE = -16, -17


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


@pytest.fixture
def pool():
    h = pa.pa_pool_create(10)
    yield h
    pa.pa_pool_destroy(h)


def test_alloc_share_release_counts(pool):
    assert pa.pa_pool_free_pages(pool) == 10
    pages = pa.pa_pool_alloc(pool, 3)
    assert len(set(pages.tolist())) == 3 and all(0 <= p < 10 for p in pages)
    assert [pa.pa_pool_refcount(pool, p) for p in pages] == [1, 1, 1]
    assert pa.pa_pool_free_pages(pool) == 7
    pa.pa_pool_share(pool, pages[:2])
    assert [pa.pa_pool_refcount(pool, p) for p in pages] == [2, 2, 1]
    pa.pa_pool_release(pool, pages)
    assert [pa.pa_pool_refcount(pool, p) for p in pages] == [1, 1, 0]
    assert pa.pa_pool_free_pages(pool) == 8
    pa.pa_pool_release(pool, [pages[0], pages[1], -1])  # unmapped entries skipped
    assert pa.pa_pool_free_pages(pool) == 10


def test_exhaustion_and_misuse_change_nothing(pool):
    with pytest.raises(pa.PAError) as e:
        pa.pa_pool_alloc(pool, 11)
    assert e.value.status == EMPTY and pa.pa_pool_free_pages(pool) == 10
    pages = pa.pa_pool_alloc(pool, 2)
    with pytest.raises(pa.PAError) as e:  # page listed twice, referenced once
        pa.pa_pool_release(pool, [pages[0], pages[0]])
    assert e.value.status == STATE and pa.pa_pool_refcount(pool, pages[0]) == 1
    free_page = next(p for p in range(10) if pa.pa_pool_refcount(pool, p) == 0)
    with pytest.raises(pa.PAError) as e:  # sharing a free page
        pa.pa_pool_share(pool, [pages[1], free_page])
    assert e.value.status == STATE and pa.pa_pool_refcount(pool, pages[1]) == 1
    with pytest.raises(pa.PAError):
        pa.pa_pool_refcount(pool, 10)


def test_prepare_append_maps_copies_or_writes_in_place(pool):
    table = np.full(4, -1, dtype=np.int32)
    # unmapped block: a fresh page, no copy
    assert pa.pa_pool_prepare_append(pool, table, 16, 0) == (-1, -1)
    assert table[0] >= 0 and pa.pa_pool_refcount(pool, table[0]) == 1
    # the only user: write in place
    assert pa.pa_pool_prepare_append(pool, table, 16, 5) == (-1, -1)
    # a fork shares the page; each writer then gets its own copy
    fork = table.copy()
    pa.pa_pool_share(pool, fork[fork >= 0])
    old = int(table[0])
    src, dst = pa.pa_pool_prepare_append(pool, fork, 16, 7)
    assert (src, dst) == (old, int(fork[0])) and dst != old
    assert pa.pa_pool_refcount(pool, old) == 1 and pa.pa_pool_refcount(pool, dst) == 1
    # the original is the last user now: in place
    assert pa.pa_pool_prepare_append(pool, table, 16, 8) == (-1, -1)
    assert int(table[0]) == old
    with pytest.raises(pa.PAError):  # position beyond the table
        pa.pa_pool_prepare_append(pool, table, 16, 64)


def test_randomized_forks_appends_and_frees_keep_the_invariant():
    n_pages, max_blocks = 64, 8
    h = pa.pa_pool_create(n_pages)
    rng = random.Random(7)
    seqs = []  # (table, length)
    try:
        for _ in range(600):
            op = rng.random()
            if op < 0.2 or not seqs:  # new sequence of a few tokens
                table = np.full(max_blocks, -1, dtype=np.int32)
                length = 0
                try:
                    for pos in range(rng.randint(1, 40)):
                        pa.pa_pool_prepare_append(h, table, 16, pos)
                        length = pos + 1
                except pa.PAError as e:
                    assert e.status == EMPTY
                seqs.append((table, length))
            elif op < 0.45:  # fork: share the whole prefix
                table, length = rng.choice(seqs)
                fork = table.copy()
                pa.pa_pool_share(h, fork[fork >= 0])
                seqs.append((fork, length))
            elif op < 0.8:  # append one token (copy-on-write when shared)
                i = rng.randrange(len(seqs))
                table, length = seqs[i]
                if length < max_blocks * 16:
                    blk = length // 16
                    before = int(table[blk])
                    shared = before >= 0 and pa.pa_pool_refcount(h, before) > 1
                    try:
                        src, dst = pa.pa_pool_prepare_append(h, table, 16, length)
                        assert (src >= 0) == shared
                        if shared:
                            assert src == before and dst == int(table[blk]) != before
                        seqs[i] = (table, length + 1)
                    except pa.PAError as e:
                        assert e.status == EMPTY and int(table[blk]) == before
            else:  # free a sequence
                table, _ = seqs.pop(rng.randrange(len(seqs)))
                pa.pa_pool_release(h, table)
            refs = np.zeros(n_pages, dtype=np.int64)
            for table, _ in seqs:
                for p in table[table >= 0]:
                    refs[p] += 1
            assert [pa.pa_pool_refcount(h, p) for p in range(n_pages)] == refs.tolist()
            assert pa.pa_pool_free_pages(h) == int((refs == 0).sum())
    finally:
        pa.pa_pool_destroy(h)


def test_concurrent_alloc_and_release_from_threads():
    h = pa.pa_pool_create(4096)
    errors = []

    def worker(seed):
        rng = random.Random(seed)
        held = []
        try:
            for _ in range(300):
                if held and rng.random() < 0.5:
                    pa.pa_pool_release(h, held.pop())
                else:
                    held.append(pa.pa_pool_alloc(h, rng.randint(1, 4)))
            for pages in held:
                pa.pa_pool_release(h, pages)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(s,)) for s in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    try:
        assert not errors, errors
        assert pa.pa_pool_free_pages(h) == 4096
        assert all(pa.pa_pool_refcount(h, p) == 0 for p in range(0, 4096, 97))
    finally:
        pa.pa_pool_destroy(h)
