"""Admission on the page pool (pks_admission_simulate), host only: the
paged-KV worked example's capacity (83 paged vs 32 reserved requests in a
16384-slot pool), the waste landmarks of page size 1 and 512, and agreement
with the oracle's capacity functions on random pools and lengths."""

import numpy as np
import pytest

import oracle
from top_sparse_attention_pks_gb300 import build, pks

from test_oracle_paging import LENS, PAGE, RESERVE, one


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()
    oracle.build()


def test_worked_example_capacity():
    slots = one("pool_slots")
    pool = pks.Pool(slots // PAGE, PAGE)
    paged, tok_p, slots_p = pool.admission(LENS)
    naive, tok_n, slots_n = pool.admission(LENS, reserve=RESERVE)
    assert paged == one("capacity_paged") and naive == one("capacity_naive")
    assert round(paged / naive, 1) == one("capacity_ratio_1dp")
    # 16 full rounds of the five requests plus the first three fill the pool
    # exactly; the fourth (30 tokens, 32 slots) does not fit
    assert slots_p == slots and tok_p == 16 * sum(LENS) + sum(LENS[:3])
    assert slots_n == naive * RESERVE
    assert pool.free_count() == slots // PAGE  # counting only


def test_waste_landmarks():
    # page size 1: no tail waste; page size 512 = the reservation: paging and
    # reservation hold the same 2560 slots, 63.0 % of them wasted
    one_pool = pks.Pool(10000, 1)
    _, tok, slots = one_pool.admission(LENS)
    assert tok == slots
    big = pks.Pool(5, 512)
    adm_p, tok_p, slots_p = big.admission(LENS)
    adm_n, tok_n, slots_n = big.admission(LENS, reserve=512)
    assert adm_p == adm_n == 5
    assert slots_p == slots_n == one("landmark_p512_tokens")
    assert round(100 * (slots_p - tok_p) / slots_p, 1) == one("landmark_p512_waste_pct_1dp")


def test_agrees_with_oracle_on_random_cases():
    rng = np.random.default_rng(3)
    for _ in range(200):
        p = int(rng.integers(1, 300))
        pages = int(rng.integers(1, 3000))
        lens = rng.integers(0, 4000, size=int(rng.integers(1, 9))).astype(np.int32)
        if lens.max() == 0:
            lens[0] = 1
        reserve = int(rng.integers(1, 5000))
        pool = pks.Pool(pages, p)
        assert pool.admission(lens)[0] == oracle.capacity_paged(lens, p, pages * p)
        # the oracle reserves token slots, the pool whole pages: equal when
        # the reservation is a whole number of pages
        r = -(-reserve // p) * p
        assert pool.admission(lens, reserve=r)[0] == oracle.capacity_naive(lens, r, pages * p)


def test_rejects_unbounded_and_bad_lengths():
    pool = pks.Pool(8, 4)
    with pytest.raises(pks.PksError):
        pool.admission([0, 0])
    with pytest.raises(pks.PksError):
        pool.admission([3, -1])
