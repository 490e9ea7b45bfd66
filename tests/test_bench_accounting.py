"""The benchmark's byte and FLOP accounting (no GPU).

The roofline fractions divide algorithmic bytes by measured time, so the
counts are checked here on hand-sized cases: the scan reads every cached
token's key once (aliased prefix pages once), the attention reads each
selected token's K and V rows once (unique physical rows), outputs are
written once; the sparse MLA reads one latent row per selected token and
does 2 H (d + r) + 2 H d FLOP per attended token (the MQA-mode model of
"Sparse Attention on GLM5.3 and HBM", DSA paragraphs).
"""

import numpy as np

import bench
from top_sparse_attention_pks_gb300.workloads import MLA_WORKLOADS, WORKLOADS


def test_gqa_bytes_count_unique_rows():
    wl = WORKLOADS["paging_example"].replace(B=2, seq_lens=(20, 5), k=4, Hq=4, Hkv=2, D=8, Di=16,
                                             page_size=4, max_pages=5)
    # request 1 aliases request 0's first page (a shared prefix page)
    bt = np.array([[0, 1, 2, 3, 4], [0, 5, -1, -1, -1]], np.int32)
    topk = np.array([[0, 1, 9, 19], [0, 4, -1, -1]], np.int32)
    ab = bench.algorithmic_bytes(wl, [20, 5], bt, topk)
    # scan: 20 + 5 tokens, 4 of them (page 0) shared -> 21 unique rows of Di bytes
    assert ab["scan"] == 21 * 16
    # K/V: rows {0, 1, 9, 19} of request 0 and {0 (shared with request 0), 4}
    # of request 1 -> 5 unique rows of Hkv * D * 2 B, K and V
    assert ab["kv"] == 5 * 2 * 8 * 2 * 2
    assert ab["out"] == 2 * 4 * 8 * 2
    assert ab["attended"] == 4 + 4
    assert ab["total"] == ab["scan"] + ab["kv"] + ab["out"]


def test_several_query_tokens_count_each_querys_gather():
    wl = WORKLOADS["paging_example"].replace(B=1, seq_lens=(8,), k=2, Hq=2, Hkv=1, D=4, Di=8,
                                             page_size=4, max_pages=2)
    bt = np.array([[3, 7]], np.int32)
    topk = np.array([[[0, 5], [5, 6]]], np.int32)  # [B, Nq, k]: token 5 read by both queries
    ab = bench.algorithmic_bytes(wl, [8], bt, topk)
    assert ab["scan"] == 8 * 8
    assert ab["kv"] == (2 + 2) * 1 * 4 * 2 * 2
    assert ab["out"] == 1 * 2 * 2 * 4 * 2
    assert ab["attended"] == 2 * 2


def test_mla_bytes_and_flops():
    wl = MLA_WORKLOADS["mla_paging_example"].replace(B=2, seq_lens=(10, 3), k=4, Hq=16,
                                                     page_size=4, max_pages=3, Di=64)
    bt = np.array([[0, 1, 2], [3, -1, -1]], np.int32)
    topk = np.array([[0, 1, 2, 9], [0, 2, -1, -1]], np.int32)
    ab = bench.mla_algorithmic(wl, [10, 3], bt, topk)
    assert ab["scan"] == 13 * 64
    assert ab["kv"] == 6 * 576 * 2
    assert ab["q"] == 2 * 16 * 576 * 2
    assert ab["out"] == 2 * 16 * 512 * 2
    assert ab["attended"] == 6
    assert ab["flops"] == 6 * 2 * 16 * (576 + 512)
    # the pages' intensity at d = 512, r = 64: 2H(2d + r) / ((d + r) * 2) = 1.889 H
    per_token = ab["flops"] / ab["attended"] / (576 * 2)
    assert abs(per_token / 16 - 1088 / 576) < 1e-12


def test_job_throughput_is_the_whole_job_over_the_slowest_rank():
    value, total = bench.job_throughput(2.0, 100, 1, None)
    assert total == 2.0 and value == 50.0
