"""GPU parity of the decode step (indexer scan, top-k, sparse attention)
against the CPU oracle, through the C ABI.

Bar: scores, top-k indices and block tables bit-exact; attention output
within max-abs 2e-2 and relative L2 5e-3 of the fp64 oracle."""

import numpy as np
import pytest
import torch

from gpu_cases import (check_attention, host, oracle_attention, oracle_topk, prepare,
                       run_step)
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def full_check(wl, t, attn_splits=0, check_scores=True, topk_mode=0):
    step, out, idx = run_step(wl, t, attn_splits, topk_mode)
    ref_scores, ref_idx = oracle_topk(wl, t)
    if check_scores:
        sc = host(step.scores()).numpy().astype(np.int64)
        lens = host(t["seq_lens"]).numpy()
        for b, n in enumerate(lens):
            assert (sc[b, :n] == ref_scores[b, :n]).all(), f"scores differ in request {b}"
    got_idx = host(idx).numpy()
    assert (got_idx == ref_idx).all(), "top-k indices differ"
    ref = oracle_attention(wl, t, ref_idx)
    check_attention(out, ref, wl.name)
    assert step.device_error() == 0
    return step, out, got_idx


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_paging_example_config(topk_mode):
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    full_check(wl, t, topk_mode=topk_mode)


@pytest.mark.parametrize("over", [
    dict(k=1), dict(k=403), dict(k=500), dict(k=30), dict(k=31), dict(k=29),
    dict(page_size=1, num_pages=1024, max_pages=512),
    dict(page_size=512, num_pages=8, max_pages=1),
    dict(permute_pool=True),
    dict(Hi=2), dict(Hi=4), dict(Hi=8), dict(Di=128), dict(D=128),
    dict(Hq=8, Hkv=8), dict(Hq=16, Hkv=1), dict(Hq=12, Hkv=4),
    dict(Hq=128, Hkv=8, D=128), dict(Hq=40, Hkv=4),
    dict(seq_lens=(0, 1, 2, 63, 64)),
    dict(seq_lens=(512, 512, 1, 511, 500), num_pages=160),
])
def test_paging_example_variants(over):
    wl = WORKLOADS["paging_example"].replace(**over)
    t, _, _ = prepare(wl)
    full_check(wl, t)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_one_and_several_chunk_requests_together(topk_mode):
    # requests of one 4096-token top-k chunk (no request barrier in the
    # single launch) beside requests of two and three chunks, sparse and dense
    lens = (4096, 4097, 8192, 100, 12288, 300)
    wl = WORKLOADS["paging_example"].replace(
        B=len(lens), seq_lens=lens, k=300, page_size=64, num_pages=3 * 193 + 16,
        max_pages=192)
    t, _, _ = prepare(wl)
    full_check(wl, t, topk_mode=topk_mode)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_all_scores_tied(topk_mode):
    # zero indexer queries: every score is 0, selection = lowest indices
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    t["q_idx"].zero_()
    _, _, idx = full_check(wl, t, topk_mode=topk_mode)
    for b, n in enumerate(wl.seq_lens):
        expect = list(range(min(n, wl.k))) + [-1] * max(0, wl.k - n)
        assert idx[b].tolist() == expect


def test_negative_weights_and_small_range_ties():
    wl = WORKLOADS["paging_example"].replace(Hi=2)
    t, _, _ = prepare(wl)
    t["w_idx"].copy_(torch.tensor([3, -2], dtype=torch.int32))
    t["q_idx"].clamp_(-2, 2)
    t["idx_k"].clamp_(-1, 1)
    full_check(wl, t)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 1000])
def test_attention_split_counts(splits):
    wl = WORKLOADS["paging_example"].replace(k=256, seq_lens=(403, 300, 241, 30, 256),
                                             num_pages=96)
    t, _, _ = prepare(wl)
    full_check(wl, t, attn_splits=splits)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_b32_4k_reduced(topk_mode):
    wl = WORKLOADS["b32_4k"].replace(B=4, seq_lens=(4096,) * 4, num_pages=256)
    t, _, _ = prepare(wl)
    full_check(wl, t, topk_mode=topk_mode)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_ragged_prefix_reduced(topk_mode):
    wl = WORKLOADS["b64_ragged_prefix"].replace(B=16, num_pages=16 * 2048)
    t, _, bt = prepare(wl)
    # aliased prefix pages are shared by the rows of a group
    assert (bt[1, :125] == bt[0, :125]).all() or host(t["seq_lens"])[1] < 2000
    full_check(wl, t, topk_mode=topk_mode)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_128k_reduced(topk_mode):
    wl = WORKLOADS["b16_128k"].replace(B=2, seq_lens=(131072, 131072), num_pages=4096)
    t, _, _ = prepare(wl)
    full_check(wl, t, topk_mode=topk_mode)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_long_request_emit_path(topk_mode):
    # two-kernel path: a context longer than the top-k bitmap (131072 tokens)
    # goes through the chunked emit kernel, a second, short request keeps the
    # bitmap path; cooperative path: 35 chunks of one request meet at the barrier
    wl = WORKLOADS["paging_example"].replace(
        B=2, seq_lens=(140000, 5000), page_size=64, max_pages=2200, num_pages=2300, k=512,
        Di=64, D=64, Hq=8, Hkv=2)
    t, _, _ = prepare(wl)
    step, _, _ = full_check(wl, t, topk_mode=topk_mode)
    # scan + top-k (one cooperative launch, or threshold + emit) + attention + merge
    assert step.launches() == (5 if topk_mode == 1 else 4)


@pytest.mark.parametrize("topk_mode", [0, 1], ids=["coop", "two_kernel"])
def test_graph_replay_matches_eager(topk_mode):
    wl = WORKLOADS["paging_example"].replace(k=128)
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k, topk_mode=topk_mode)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)  # warm up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for trial in range(3):
        q_new, qi_new = (torch.randn_like(t["q"].float()).to(torch.bfloat16),
                         torch.randint(-127, 128, t["q_idx"].shape, dtype=torch.int8,
                                       device="cuda"))
        t["q"].copy_(q_new)
        t["q_idx"].copy_(qi_new)
        g.replay()
        torch.cuda.synchronize()
        _, ref_idx = oracle_topk(wl, t)
        assert (host(step.topk_idx).numpy() == ref_idx).all()
        check_attention(step.out, oracle_attention(wl, t, ref_idx), f"replay {trial}")


def test_attention_only_any_order_and_padding():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    rng = np.random.default_rng(0)
    idx = np.full((wl.B, wl.k), -1, np.int32)
    for b, n in enumerate(wl.seq_lens):
        m = min(n, 40)
        idx[b, rng.permutation(wl.k)[:m]] = rng.choice(n, size=m, replace=False)
    step.topk_idx.copy_(torch.from_numpy(idx))
    step.attention_only()
    torch.cuda.synchronize()
    check_attention(step.out, oracle_attention(wl, t, idx), "attention only")


def test_device_checks_report_bad_inputs():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    step()
    assert step.device_error() == 0
    # a page id outside the pool: the kernels skip it and report code 1
    t["block_table"][0, 3] = wl.num_pages + 5
    step()
    assert step.device_error() == 1
    t["block_table"][0, 3] = 3
    # a selected position past the request's length: code 2
    step()
    step.device_error()
    step.topk_idx[3, 0] = 31  # request 3 holds 30 tokens
    step.attention_only()
    assert step.device_error() == 2
    # a sequence length beyond max_pages * page_size: code 3
    t["seq_lens"][1] = wl.max_pages * wl.page_size + 1
    step()
    assert step.device_error() == 3
