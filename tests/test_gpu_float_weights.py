"""GPU parity of the indexer with real-valued head weights.

"Sparse Attention on GLM5.3 and HBM", lightning indexer paragraph: the index
score is a weighted sum of the heads' ReLU logits.  The scan computes it in
fp32 in the oracle's convention (heads in order, each product and sum rounded
to nearest), so the scores (as fp32 values), the top-k indices and the
attention over them are compared with the oracle exactly as for integer
weights: scores and indices bit-exact, outputs within tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import check_attention, host, oracle_attention, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS, draw_float_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _oracle_f(wl, t, w_f, requests=None):
    lens = host(t["seq_lens"]).numpy()
    bt = host(t["block_table"]).numpy()
    q_idx = host(t["q_idx"]).numpy()
    w = host(w_f).numpy()
    if requests is not None:
        lens, bt, q_idx, w = lens[requests], bt[requests], q_idx[requests], w[requests]
    sc = oracle.indexer_scores_f(lens, bt, wl.page_size, q_idx, w, host(t["idx_k"]).numpy())
    return sc, oracle.topk_f(lens, sc, wl.k)


@pytest.mark.parametrize("name,signed,topk_mode", [
    ("paging_example", False, 0), ("paging_example", True, 1),
    ("b32_4k", True, 0), ("b64_ragged_prefix", False, 0), ("b64_ragged_prefix", True, 1)])
def test_float_weights_scores_topk_attention(name, signed, topk_mode):
    wl = WORKLOADS[name]
    t, _, _ = prepare(wl)
    t["w_idx_f"] = draw_float_weights(wl, "cuda", signed=signed)
    step = SparseDecodeStep(t, wl.k, topk_mode=topk_mode)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    ref_sc, ref_idx = _oracle_f(wl, t, t["w_idx_f"])
    lens = host(t["seq_lens"]).numpy()
    keys = host(step.scores()).numpy()
    got_sc = pks.float_key_to_score(keys)
    for b, n in enumerate(lens):
        np.testing.assert_array_equal(got_sc[b, :n], ref_sc[b, :n], err_msg=f"request {b}")
    assert (host(idx).numpy() == ref_idx).all(), "top-k indices differ"
    check_attention(out, oracle_attention(wl, t, ref_idx), name)


def test_integer_valued_float_weights_match_the_integer_path():
    wl = WORKLOADS["b32_4k"]
    t, _, _ = prepare(wl)
    s_int = SparseDecodeStep(t, wl.k)
    _, idx_int = s_int()
    tf = dict(t)
    tf["w_idx_f"] = torch.ones((wl.B, wl.Hi), dtype=torch.float32, device="cuda") * 3.0
    ti = dict(t)
    ti["w_idx"] = torch.full((wl.Hi,), 3, dtype=torch.int32, device="cuda")
    _, idx_i3 = SparseDecodeStep(ti, wl.k)()
    _, idx_f3 = SparseDecodeStep(tf, wl.k)()
    torch.cuda.synchronize()
    assert torch.equal(idx_i3, idx_f3)
    assert torch.equal(idx_int, idx_f3)  # uniform weights do not change the order


def test_float_weights_full_size_sampled():
    wl = WORKLOADS["b16_128k"]
    t, _, _ = prepare(wl)
    t["w_idx_f"] = draw_float_weights(wl, "cuda", signed=True)
    step = SparseDecodeStep(t, wl.k)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    req = [0, 7, 15]
    _, ref_idx = _oracle_f(wl, t, t["w_idx_f"], requests=req)
    got = host(idx).numpy()
    assert (got[req] == ref_idx).all(), "top-k indices differ"
    ref = oracle_attention(wl, t, got, requests=req)
    check_attention(out[torch.as_tensor(req, device=out.device)], ref, "b16_128k float weights")
    del t, step
    torch.cuda.empty_cache()


def test_float_weights_reject_several_query_tokens():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    a = pks.make_args(k=wl.k, w_idx_f=torch.ones((wl.B, wl.Hi), device="cuda"), **t)
    a.n_queries = 2
    import ctypes
    n = ctypes.c_size_t()
    assert pks.lib().pks_decode_workspace_size(ctypes.byref(a), ctypes.byref(n)) == -6


@pytest.mark.parametrize("topk_mode", [0, 1])
def test_all_tied_scores_take_the_lowest_tokens(topk_mode):
    # zero head weights: every token scores 0, so the top-k of a request longer
    # than k is its first k tokens
    wl = WORKLOADS["b32_4k"]
    t, _, _ = prepare(wl)
    t["w_idx"] = torch.zeros((wl.Hi,), dtype=torch.int32, device="cuda")
    step = SparseDecodeStep(t, wl.k, topk_mode=topk_mode)
    _, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    want = np.tile(np.arange(wl.k, dtype=np.int32), (wl.B, 1))
    np.testing.assert_array_equal(host(idx).numpy(), want)


def test_negative_weights_thousands_of_zero_ties_full_size():
    # weights all negative: about len/16 tokens tie at the largest score, 0
    wl = WORKLOADS["b16_128k"]
    t, _, _ = prepare(wl)
    t["w_idx_f"] = -draw_float_weights(wl, "cuda")
    step = SparseDecodeStep(t, wl.k)
    _, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    req = [0, 9]
    _, ref_idx = _oracle_f(wl, t, t["w_idx_f"], requests=req)
    assert (host(idx).numpy()[req] == ref_idx).all(), "top-k indices differ"
    del t, step
    torch.cuda.empty_cache()
