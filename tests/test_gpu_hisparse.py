"""KV cache in host memory with an LRU cache of its pages in HBM: select,
residency update, miss fetch, attention through the table.  Over several
steps with changing queries: top-k bit-exact against the oracle, every
resident slot bit-identical to its page in the host pool, and the attention
output bit-identical to pks_sparse_attention on the whole pool in HBM (the
same grid and arithmetic on the same K/V values) and within tolerance of the
oracle."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import check_attention, host, oracle_attention, oracle_topk, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import ResidentDecodeStep, SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _run(wl, capacity, n_init, steps, seed):
    t, _, bt = prepare(wl)
    host_k = t["kv_k"].cpu().pin_memory()
    host_v = t["kv_v"].cpu().pin_memory()
    rng = np.random.default_rng(seed)
    init = rng.choice(wl.num_pages, size=n_init, replace=False)
    res = ResidentDecodeStep(t, host_k, host_v, wl.k, capacity, init)
    ref_table = oracle.Residency(wl.num_pages, capacity, init)
    full = SparseDecodeStep(t, wl.k)  # K/V wholly in HBM, for the bit-identical check
    admitted_total = overflow_total = 0
    for step in range(steps):
        if step:
            t["q"].copy_(torch.randn_like(t["q"].float()).to(torch.bfloat16))
            t["q_idx"].copy_(torch.randint(-127, 128, t["q_idx"].shape, dtype=torch.int8,
                                           device="cuda"))
        out, idx = res()
        torch.cuda.synchronize()
        _, ref_idx = oracle_topk(wl, t)
        got_idx = host(idx).numpy()
        assert (got_idx == ref_idx).all(), f"step {step}: top-k"
        miss_ref, _ = ref_table.step(ref_idx, bt, wl.page_size)
        n = int(res.n_miss.item())
        assert n == len(miss_ref) and (host(res.miss[:n]).numpy() == miss_ref).all()
        # every resident page's slot holds that page's K and V
        slot_page = host(res.table.slot_page()).numpy()
        assert (slot_page == ref_table.slot_page).all()
        for s, p in enumerate(slot_page):
            if p >= 0:
                assert torch.equal(res.slot_k[s].cpu(), host_k[p]), f"step {step}: slot {s} K"
                assert torch.equal(res.slot_v[s].cpu(), host_v[p]), f"step {step}: slot {s} V"
        admitted = int((ref_table.page_slot[miss_ref] >= 0).sum()) if n else 0
        admitted_total += admitted
        overflow_total += n - admitted
        # attention through the table == attention on the whole pool in HBM
        full.topk_idx.copy_(idx)
        full.attention_only()
        torch.cuda.synchronize()
        assert torch.equal(out, full.out), f"step {step}: resident attention differs"
        check_attention(out, oracle_attention(wl, t, ref_idx), f"resident step {step}")
    return admitted_total, overflow_total


def test_all_misses_admitted():
    wl = WORKLOADS["paging_example"].replace(k=40)
    # 64 slots hold all 61 pages the requests use: every miss is admitted
    admitted, overflow = _run(wl, capacity=64, n_init=10, steps=4, seed=5)
    assert admitted > 0 and overflow == 0


def test_overflow_misses_read_from_host():
    # 61 pages in use, 12 slots: most misses are not admitted and the
    # attention reads them straight from the host pools
    wl = WORKLOADS["paging_example"].replace(k=64)
    admitted, overflow = _run(wl, capacity=12, n_init=6, steps=3, seed=6)
    assert overflow > 0


def test_b32_4k_reduced_through_the_table():
    wl = WORKLOADS["b32_4k"].replace(B=4, seq_lens=(4096, 3000, 4096, 100), num_pages=256)
    admitted, overflow = _run(wl, capacity=96, n_init=40, steps=3, seed=7)
    assert admitted > 0


def test_layers_with_the_fetch_overlapped():
    # three layers, each with its own pools, table and queries; the fetch of a
    # layer runs on a side stream under the neighbouring layers' selection and
    # attention.  Against the same layers run one call after another, the
    # oracle's residency per layer, the attention on each pool wholly in HBM
    # and the oracle's attention.
    from top_sparse_attention_pks_gb300.decoder import ResidentLayers
    wl = WORKLOADS["b32_4k"].replace(B=4, seq_lens=(4096, 3000, 4096, 100), num_pages=256)
    capacity, n_layers = 96, 3
    layers, refs, fulls, bts = [], [], [], []
    for l in range(n_layers):
        t, _, bt = prepare(wl, seed_offset=l)
        init = np.random.default_rng(40 + l).choice(wl.num_pages, size=40, replace=False)
        layers.append(dict(tensors=t, host_k=t["kv_k"].cpu().pin_memory(),
                           host_v=t["kv_v"].cpu().pin_memory(), init_pages=init))
        refs.append(oracle.Residency(wl.num_pages, capacity, init))
        fulls.append(SparseDecodeStep(t, wl.k))
        bts.append(bt)
    over = ResidentLayers(layers, wl.k, capacity)
    serial = ResidentLayers(layers, wl.k, capacity)
    admitted = 0
    for step in range(3):
        for L in layers:
            t = L["tensors"]
            t["q"].copy_(torch.randn_like(t["q"].float()).to(torch.bfloat16))
            t["q_idx"].copy_(torch.randint(-127, 128, t["q_idx"].shape, dtype=torch.int8,
                                           device="cuda"))
        got = over(overlap=True)
        ser = serial(overlap=False)
        torch.cuda.synchronize()
        for l, L in enumerate(layers):
            t = L["tensors"]
            out, idx = got[l]
            _, ref_idx = oracle_topk(wl, t)
            assert (host(idx).numpy() == ref_idx).all(), f"step {step} layer {l}: top-k"
            miss_ref, _ = refs[l].step(ref_idx, bts[l], wl.page_size)
            lay = over.layers[l]
            n = int(lay.n_miss.item())
            assert n == len(miss_ref) and (host(lay.miss[:n]).numpy() == miss_ref).all()
            admitted += int((refs[l].page_slot[miss_ref] >= 0).sum()) if n else 0
            assert torch.equal(out, ser[l][0]), f"step {step} layer {l}: overlapped != serial"
            fulls[l].topk_idx.copy_(idx)
            fulls[l].attention_only()
            torch.cuda.synchronize()
            assert torch.equal(out, fulls[l].out), f"step {step} layer {l}: != pool in HBM"
            check_attention(out, oracle_attention(wl, t, ref_idx), f"step {step} layer {l}")
    assert admitted > 0
