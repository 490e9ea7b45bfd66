"""Several query tokens per request (n_queries = Nq): one pass over the
indexer keys scores every query, each query selects its own top-k and
attends over it.  The oracle sees B * Nq virtual requests (lengths and block
table rows repeated, queries reshaped): scores and top-k bit-exact,
attention within tolerance."""

import numpy as np
import pytest
import torch

from gpu_cases import check_attention, host, oracle_attention, oracle_topk, prepare
from top_sparse_attention_pks_gb300 import build
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _multi(wl, nq, topk_mode=0, seed=11):
    t, _, _ = prepare(wl)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    B = wl.B
    t["q"] = torch.randn((B, nq, wl.Hq, wl.D), device="cuda", generator=gen).to(torch.bfloat16)
    t["q_idx"] = torch.randint(-127, 128, (B, nq, wl.Hi, wl.Di), dtype=torch.int8, device="cuda",
                               generator=gen)
    step = SparseDecodeStep(t, wl.k, topk_mode=topk_mode)
    assert step.args.n_queries == nq
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    # the oracle's view: B * nq virtual requests
    tv = dict(t)
    tv["seq_lens"] = t["seq_lens"].repeat_interleave(nq)
    tv["block_table"] = t["block_table"].repeat_interleave(nq, dim=0)
    tv["q"] = t["q"].reshape(B * nq, wl.Hq, wl.D)
    tv["q_idx"] = t["q_idx"].reshape(B * nq, wl.Hi, wl.Di)
    wlv = wl.replace(B=B * nq)
    ref_scores, ref_idx = oracle_topk(wlv, tv)
    sc = host(step.scores()).numpy().astype(np.int64)
    lens = host(tv["seq_lens"]).numpy()
    for v, n in enumerate(lens):
        assert (sc[v, :n] == ref_scores[v, :n]).all(), f"scores of virtual request {v}"
    got = host(idx).numpy().reshape(B * nq, wl.k)
    assert (got == ref_idx).all(), "top-k"
    check_attention(out.reshape(B * nq, wl.Hq, wl.D), oracle_attention(wlv, tv, ref_idx),
                    f"{wl.name} Nq={nq}")
    return step


@pytest.mark.parametrize("nq,hi", [(2, 1), (4, 1), (8, 1), (2, 2), (4, 2), (2, 4)])
def test_paging_example_several_queries(nq, hi):
    _multi(WORKLOADS["paging_example"].replace(Hi=hi), nq)


def test_two_kernel_top_k_path():
    _multi(WORKLOADS["paging_example"].replace(k=100), 2, topk_mode=1)


def test_128k_reduced_two_queries():
    wl = WORKLOADS["b16_128k"].replace(B=2, seq_lens=(131072, 90000), num_pages=4096)
    _multi(wl, 2)


def test_selections_differ_between_queries():
    # the two queries of a request pick different tokens (they are scored
    # separately, not merged)
    step = _multi(WORKLOADS["paging_example"].replace(k=32), 2, seed=12)
    idx = host(step.topk_idx).numpy()
    assert (idx[0, 0] != idx[0, 1]).any()
