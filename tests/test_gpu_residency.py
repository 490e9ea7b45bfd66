"""GPU parity of the residency table (miss list + LRU update) against the
oracle over multi-step sequences: miss lists, counts and the whole slot
table bit-exact after every step."""

import numpy as np
import pytest
import torch

import oracle
from top_sparse_attention_pks_gb300 import build, pks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def random_selection(rng, lens, k):
    """Seeded stand-in for a top-k output: ascending unique positions, -1 padded."""
    idx = np.full((len(lens), k), -1, np.int32)
    for b, n in enumerate(lens):
        m = min(int(n), k)
        idx[b, :m] = np.sort(rng.choice(int(n), size=m, replace=False))
    return idx


def run_sequence(num_pages, capacity, init, lens, bt, page, k, steps, seed):
    rng = np.random.default_rng(seed)
    ref = oracle.Residency(num_pages, capacity, init)
    table = pks.ResidencyTable(num_pages, capacity, init)
    bt_d = torch.from_numpy(bt).cuda()
    miss_d = torch.empty(num_pages, dtype=torch.int32, device="cuda")
    n_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    total_miss = 0
    for step in range(steps):
        idx = random_selection(rng, lens, k)
        if step % 7 == 3:
            idx = prev  # noqa: F821  (repeat a selection: hits only when it fits)
        prev = idx
        miss_ref, _ = ref.step(idx, bt, page)
        table.update(torch.from_numpy(idx).cuda(), bt_d, page, miss_d, n_d)
        torch.cuda.synchronize()
        n = int(n_d.item())
        assert n == len(miss_ref), f"step {step}: n_miss {n} != {len(miss_ref)}"
        assert (miss_d[:n].cpu().numpy() == miss_ref).all(), f"step {step}: miss list"
        assert (table.slot_page().cpu().numpy() == ref.slot_page).all(), f"step {step}"
        assert (table.page_slot().cpu().numpy() == ref.page_slot).all(), f"step {step}"
        assert (table.last_use().cpu().numpy() == ref.last_use).all(), f"step {step}"
        lu = ref.last_use
        order = table.lru_order().cpu().numpy()
        assert sorted(order.tolist()) == list(range(capacity))
        keys = [(int(lu[s]), int(s)) for s in order]
        assert keys == sorted(keys), f"step {step}: LRU order"
        total_miss += n
    assert table.step_count() == steps
    return total_miss


def test_small_sequences():
    rng = np.random.default_rng(0)
    num_pages, cap, page, k = 96, 24, 8, 6
    lens = [200, 150, 37]
    bt = np.full((3, 25), -1, np.int32)
    perm = rng.permutation(num_pages).astype(np.int32)
    off = 0
    for b, n in enumerate(lens):
        np_ = -(-n // page)
        bt[b, :np_] = perm[off: off + np_]
        off += np_
    init = rng.choice(num_pages, size=10, replace=False)
    run_sequence(num_pages, cap, init, lens, bt, page, k, steps=40, seed=1)


def test_empty_table_and_tiny_capacity():
    num_pages, page, k = 32, 4, 3
    lens = [64, 64]
    bt = np.arange(32, dtype=np.int32).reshape(2, 16)
    run_sequence(num_pages, 0, [], lens, bt, page, k, steps=5, seed=2)
    run_sequence(num_pages, 1, [], lens, bt, page, k, steps=12, seed=3)


def test_full_size_lru_workload():
    # 256 requests x 8192 tokens in 64-token pages (32768 pages), 16384 slots
    # initially holding a random half of the pages, top-1024 per request:
    # nearly every page is selected each step, so the table overflows
    from top_sparse_attention_pks_gb300.workloads import WORKLOADS, draw_host
    wl = WORKLOADS["b256_8k_lru"]
    h = draw_host(wl)
    pool = pks.Pool(wl.num_pages, wl.page_size, h["free_order"])
    bt, _ = pool.build_block_table(h["seq_lens"], wl.max_pages)
    misses = run_sequence(wl.num_pages, wl.capacity, h["initial_resident"].numpy(),
                          h["seq_lens"].numpy(), bt, wl.page_size, wl.k, steps=4, seed=4)
    assert misses > 0
