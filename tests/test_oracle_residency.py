"""Pins of the oracle's residency table (HiSparse-style LRU over KV pages).

"Sparse Attention on GLM5.3 and HBM", HiSparse paragraph: KV entries live in
an LRU cache in HBM; a top-k selection that misses loads the tokens, and
eviction follows least recent use.  "Why recalling an old conversation costs
so much", "The benefit is clearly measurable": under sequential access with a
working set larger than the store, LRU reuses almost nothing (a cliff, not a
slope).

Pins: a textbook LRU cache (collections.OrderedDict) when each step touches
one page, the sequential-scan cliff, and set invariants of every step.
"""

from collections import OrderedDict

import numpy as np
import pytest

import oracle


def _touch(pages, page_size=4):
    """idx/block_table for one request that selects one token on each page."""
    pages = list(pages)
    bt = np.array([pages], np.int32)
    idx = np.array([[j * page_size for j in range(len(pages))]], np.int32)
    return idx, bt


def test_textbook_lru_single_page_steps():
    rng = np.random.default_rng(0)
    num_pages, cap = 20, 6
    res = oracle.Residency(num_pages, cap)
    lru = OrderedDict()
    for step in range(400):
        p = int(rng.integers(0, num_pages))
        idx, bt = _touch([p])
        miss, n_hit = res.step(idx, bt, 4)
        hit = p in lru
        if hit:
            lru.move_to_end(p)
        else:
            if len(lru) == cap:
                lru.popitem(last=False)
            lru[p] = True
        assert n_hit == int(hit)
        assert miss.tolist() == ([] if hit else [p])
        assert res.resident_pages().tolist() == sorted(lru)


@pytest.mark.parametrize("working_set,cap,expect_hits", [(8, 6, 0), (6, 6, None)])
def test_sequential_scan_cliff(working_set, cap, expect_hits):
    res = oracle.Residency(32, cap)
    hits = 0
    for rnd in range(5):
        for p in range(working_set):
            _, h = res.step(*_touch([p]), 4)
            hits += h
    if expect_hits is not None:
        assert hits == expect_hits  # working set larger than the store: no reuse
    else:
        assert hits == 4 * working_set  # fits: everything after the first pass hits


def test_step_invariants_random():
    rng = np.random.default_rng(1)
    num_pages, cap, page, B, k, L = 96, 24, 8, 3, 6, 200
    init = rng.choice(num_pages, size=10, replace=False)
    res = oracle.Residency(num_pages, cap, init)
    bt = rng.permutation(num_pages)[: B * 25].reshape(B, 25).astype(np.int32)
    for step in range(60):
        before = set(res.resident_pages().tolist())
        idx = np.sort(rng.choice(L, size=(B, k)), axis=1).astype(np.int32)
        idx[rng.random((B, k)) < 0.2] = -1
        A = {int(bt[b, t // page]) for b in range(B) for t in idx[b] if t >= 0}
        miss, n_hit = res.step(idx, bt, page)
        after = set(res.resident_pages().tolist())
        assert miss.tolist() == sorted(A - before)  # ascending, unique, disjoint
        assert n_hit == len(A & before) and n_hit + len(miss) == len(A)
        assert len(after) <= cap
        assert (A & before) <= after  # a step never evicts what it reads
        if len(A) <= cap:
            assert A <= after
        # slot table is a consistent bijection
        sp = res.slot_page
        assert all(res.page_slot[p] == s for s, p in enumerate(sp) if p >= 0)
        assert (res.page_slot >= 0).sum() == (sp >= 0).sum()


def test_subset_of_resident_changes_nothing():
    res = oracle.Residency(16, 8, [1, 2, 3, 4])
    miss, n_hit = res.step(*_touch([2, 4]), 4)
    assert miss.size == 0 and n_hit == 2
    assert res.resident_pages().tolist() == [1, 2, 3, 4]


def test_repeat_step_has_no_misses_and_fresh_table_misses_all():
    res = oracle.Residency(30, 10)
    pages = [7, 3, 29, 11, 0]
    miss, n_hit = res.step(*_touch(pages), 4)
    assert miss.tolist() == sorted(pages) and n_hit == 0
    miss, n_hit = res.step(*_touch(pages), 4)
    assert miss.size == 0 and n_hit == len(pages)


def test_overflow_reports_all_misses_and_keeps_hits():
    # |A| > capacity: every miss is reported; hits stay resident; admitted
    # misses are the lowest page ids, taking the least recently used slots
    res = oracle.Residency(40, 4, [0, 1])
    pages = list(range(10))
    miss, n_hit = res.step(*_touch(pages), 4)
    assert n_hit == 2 and miss.tolist() == list(range(2, 10))
    assert res.resident_pages().tolist() == [0, 1, 2, 3]


def test_victim_order_last_use_then_slot():
    res = oracle.Residency(20, 3, [5, 6, 7])  # slots 0,1,2 hold 5,6,7, last use 0
    res.step(*_touch([6]), 4)  # slot 1 used at step 1
    miss, _ = res.step(*_touch([10, 11]), 4)  # victims: slot 0 then slot 2
    assert miss.tolist() == [10, 11]
    assert res.slot_page.tolist() == [10, 6, 11]
    miss, _ = res.step(*_touch([12]), 4)  # LRU now: slot 1 (last use 1)
    assert res.slot_page.tolist() == [10, 12, 11]
