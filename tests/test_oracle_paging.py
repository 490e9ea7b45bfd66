"""Pins of the oracle's paging arithmetic against the "Paged KV cache" chapter.

Every expected value comes from ``golden/paged_kv_worked_example.txt``, which
restates the chapter's worked table, prose figures, landmarks, capacity and
page-sharing examples, and quiz (each with its section).
"""

from pathlib import Path

import numpy as np
import pytest

import oracle

GOLDEN = Path(__file__).parent / "golden" / "paged_kv_worked_example.txt"
KIB = 1024
TOKEN_BYTES = 128 * KIB  # "Paged KV cache": 128 KiB per token (Llama 3.1 8B shape)
MIB = 1024 * 1024


def _golden():
    rows, kv = [], {}
    for line in GOLDEN.read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0].isdigit():
            rows.append([int(x) for x in parts])
        else:
            kv[parts[0]] = [float(x) if "." in x else int(x) for x in parts[1:]]
    return rows, kv


ROWS, KV = _golden()
LENS = [r[0] for r in ROWS]
PAGE = 16
RESERVE = 512


def one(key):
    return KV[key][0]


def test_rows_pages_tail_naive():
    for length, pages, paged, fill, tail, reserve, naive_waste in ROWS:
        assert oracle.pages_for(length, PAGE) == pages
        assert oracle.pages_for(length, PAGE) * PAGE == paged
        assert oracle.tail_waste(length, PAGE) == tail
        assert PAGE - tail == fill  # tokens used in the last page
        assert reserve == RESERVE and reserve - length == naive_waste


def test_totals_and_percentages():
    pages = [oracle.pages_for(n, PAGE) for n in LENS]
    tails = [oracle.tail_waste(n, PAGE) for n in LENS]
    assert sum(LENS) == one("total_tokens")
    assert sum(pages) == one("total_pages")
    assert sum(pages) * PAGE == one("total_paged_tokens")
    assert sum(tails) == one("total_tail_waste")
    assert sum(1 for t in tails if t == 0) == one("full_last_pages")
    naive = RESERVE * len(LENS)
    assert naive == one("naive_reserved")
    assert naive - sum(LENS) == one("naive_waste")
    assert round(100 * (naive - sum(LENS)) / naive, 1) == one("naive_waste_pct_1dp")
    assert round((naive - sum(LENS)) * TOKEN_BYTES / MIB, 1) == one("naive_idle_mib_1dp")
    assert round(naive * TOKEN_BYTES / MIB, 1) == one("naive_total_mib_1dp")
    assert round(sum(pages) * PAGE * TOKEN_BYTES / MIB, 1) == one("paged_mib_1dp")
    assert round(100 * sum(tails) / (sum(pages) * PAGE), 1) == one("paged_waste_pct_1dp")
    used, waste, npages, psize, total = KV["check_rule"]
    assert used + waste == npages * psize == total
    assert sum(LENS) + sum(tails) == sum(pages) * PAGE


def test_grid_note():
    cells_per_request = RESERVE // PAGE
    assert cells_per_request * len(LENS) == one("grid_cells")
    used = sum(oracle.pages_for(n, PAGE) for n in LENS)
    assert one("grid_cells") - used == one("grid_empty_cells")


def test_landmarks():
    # page size 1: no tail anywhere
    assert sum(oracle.tail_waste(n, 1) for n in LENS) == one("landmark_p1_waste")
    # page size 512 (= the reservation): identical to naive reservation
    held = sum(oracle.pages_for(n, 512) * 512 for n in LENS)
    assert held == one("landmark_p512_tokens")
    assert round(100 * (held - sum(LENS)) / held, 1) == one("landmark_p512_waste_pct_1dp")


def test_paging_invariant_many_sizes():
    # "Paging" check rule holds at every configuration
    rng = np.random.default_rng(0)
    for _ in range(200):
        p = int(rng.integers(1, 600))
        lens = rng.integers(0, 5000, size=7)
        pages = sum(oracle.pages_for(int(n), p) for n in lens)
        tails = sum(oracle.tail_waste(int(n), p) for n in lens)
        assert int(lens.sum()) + tails == pages * p
        assert all(0 <= oracle.tail_waste(int(n), p) < p for n in lens)


def test_capacity():
    slots = one("pool_slots")
    assert 2 * 1024 ** 3 // TOKEN_BYTES == slots
    naive = oracle.capacity_naive(LENS, RESERVE, slots)
    paged = oracle.capacity_paged(LENS, PAGE, slots)
    assert naive == one("capacity_naive")
    assert paged == one("capacity_paged")
    assert round(paged / naive, 1) == one("capacity_ratio_1dp")
    per_round = sum(oracle.pages_for(n, PAGE) * PAGE for n in LENS)
    assert round(per_round / len(LENS), 1) == one("paged_mean_slots_1dp")
    rounds = slots // per_round
    assert rounds == one("rounds_full")
    left = slots - rounds * per_round
    assert left == one("slots_left_after_rounds")
    first3 = [oracle.pages_for(n, PAGE) * PAGE for n in LENS[:3]]
    assert sum(first3) == left and oracle.pages_for(LENS[3], PAGE) * PAGE == 32


def _block_table(lens, prefix_len, sharing, page=PAGE, max_pages=64, num_pages=4096,
                 free_order=None):
    group = [0 if i < sharing else -1 for i in range(len(lens))]
    return oracle.build_block_table(lens, page, max_pages, num_pages, prefix_group=group,
                                    prefix_len=prefix_len, free_order=free_order)


def test_prefix_sharing_default():
    n = one("share_default_requests")
    bt0, used0 = _block_table(LENS, 0, 0)
    bt, used = _block_table(LENS, one("share_default_prefix"), n)
    assert used0 == one("total_pages")
    assert used0 - used == one("share_default_saved_pages")
    assert used * PAGE == one("share_default_held_tokens")
    # saved pages formula of "Page sharing": (n - 1) * floor(prefix / page)
    assert (n - 1) * (one("share_default_prefix") // PAGE) == used0 - used
    # aliased pages appear in exactly the sharing rows
    shared = bt[0, : one("share_default_prefix") // PAGE]
    for r in range(1, n):
        assert (bt[r, : len(shared)] == shared).all()
    others = bt[n:][bt[n:] >= 0]
    assert not np.isin(shared, others).any()


def test_prefix_sharing_boundary():
    n = one("share_default_requests")
    _, used0 = _block_table(LENS, 0, 0)
    _, used15 = _block_table(LENS, 15, n)
    _, used16 = _block_table(LENS, 16, n)
    assert used0 - used15 == one("share_prefix15_saved")
    assert used0 - used16 == one("share_prefix16_saved")


def test_quiz():
    length, page, pages, tail = KV["quiz1"]
    assert oracle.pages_for(length, page) == pages and oracle.tail_waste(length, page) == tail
    nreq, prefix, page, saved = KV["quiz2"]
    lens = [200] * nreq
    _, used0 = _block_table(lens, 0, 0, page=page)
    _, used = _block_table(lens, prefix, nreq, page=page)
    assert used0 - used == saved


def test_block_table_fifo_and_permutation():
    lens = [403, 96, 241, 30, 176]
    bt, used = oracle.build_block_table(lens, 16, 32, 64)
    # ascending FIFO pool: pages handed out in request order, page order
    flat = np.concatenate([bt[b, : oracle.pages_for(n, 16)] for b, n in enumerate(lens)])
    assert (flat == np.arange(61)).all() and used == 61
    assert (bt[0, 26:] == -1).all()
    perm = np.random.default_rng(1).permutation(64).astype(np.int32)
    btp, _ = oracle.build_block_table(lens, 16, 32, 64, free_order=perm)
    assert (btp[bt >= 0] == perm[bt[bt >= 0]]).all()


def test_block_table_errors():
    with pytest.raises(oracle.OracleError):
        oracle.build_block_table([100], 16, 4, 64)  # needs 7 pages > max_pages
    with pytest.raises(oracle.OracleError):
        oracle.build_block_table([100, 100], 16, 8, 10)  # pool of 10 < 14 pages


def test_short_member_shares_only_its_full_pages():
    # a group member shorter than the prefix shares only the pages it fills
    lens = [100, 40, 100]  # prefix 64 tokens = 4 pages; member 1 has 2 full pages
    bt, used = oracle.build_block_table(lens, 16, 8, 64, prefix_group=[0, 0, 0], prefix_len=64)
    assert (bt[1, :2] == bt[0, :2]).all() and bt[1, 2] not in bt[0]
    assert (bt[2, :4] == bt[0, :4]).all()
    assert used == 7 + 1 + 3  # 7 + (3 - 2) + (7 - 4)
