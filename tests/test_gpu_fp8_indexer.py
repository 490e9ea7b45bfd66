"""GPU checks of the FP8 (e4m3) indexer against the exact oracle.

"Sparse Attention on GLM5.3 and HBM": DSA's lightning indexer runs in FP8.
The scan takes each head's dot product on the tensor core with fp32
accumulation in the hardware's order, so its scores are compared with the
exact scores within a rounding bound (2^-16 of the sum of the absolute
products, weights included: about 256 times the fp32 unit roundoff per
accumulated term); the selection is checked two ways: bit-exact against the
oracle's top-k run on the GPU's own fp32 scores (the select logic), and valid
against the exact scores (no unselected token scores more than a selected one
by more than twice the bound).  Attention over the selection as usual.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import check_attention, host, oracle_attention, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import (WORKLOADS, draw_float_weights,
                                                      draw_fp8_indexer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _bound(t, w, lens, bt, P, requests):
    """2^-16 * sum_h |w_h| * sum_d |q_hd k_d| for every token of the requests."""
    kf = t["idx_k"].view(torch.float8_e4m3fn).double().abs()
    qf = t["q_idx"].view(torch.float8_e4m3fn).double().abs()
    out = []
    for b in requests:
        n = int(lens[b])
        tok = torch.arange(n, device=kf.device)
        pages = torch.as_tensor(bt[b], device=kf.device).long()[tok // P]
        rows = kf[pages, tok % P]                      # [n, Di]
        s = (rows @ qf[b].T) @ torch.as_tensor(np.abs(w[b]), device=kf.device, dtype=torch.float64)
        out.append(s.cpu().numpy() * 2.0 ** -16)
    return out


@pytest.mark.parametrize("name,signed,requests", [
    ("paging_example", False, None), ("b32_4k", True, None), ("b64_ragged_prefix", False, None),
    ("b16_128k", True, [0, 11])])
def test_fp8_scores_selection_attention(name, signed, requests):
    wl = WORKLOADS[name]
    t, _, _ = prepare(wl)
    t["q_idx"], t["idx_k"] = draw_fp8_indexer(wl, "cuda")
    t["w_idx_f"] = draw_float_weights(wl, "cuda", signed=signed)
    t["idx_fp8"] = True
    step = SparseDecodeStep(t, wl.k)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    req = list(range(wl.B)) if requests is None else requests
    lens = host(t["seq_lens"]).numpy()
    bt = host(t["block_table"]).numpy()
    w = host(t["w_idx_f"]).numpy()
    g = pks.float_key_to_score(host(step.scores()).numpy())[req]
    got_idx = host(idx).numpy()
    exact = oracle.indexer_scores_fp8(lens[req], bt[req], wl.page_size, host(t["q_idx"])[req],
                                      w[req], host(t["idx_k"]))
    bounds = _bound(t, w, lens, bt, wl.page_size, req)
    for i, b in enumerate(req):
        n = int(lens[b])
        err = np.abs(g[i, :n].astype(np.float64) - exact[i, :n])
        assert (err <= bounds[i] + 1e-30).all(), f"request {b}: score error above the bound"
    # the select logic is exact on the GPU's own scores
    np.testing.assert_array_equal(got_idx[req], oracle.topk_f(lens[req], g, wl.k))
    # and the selection is valid for the exact scores
    for i, b in enumerate(req):
        n = int(lens[b])
        if n <= wl.k:
            continue
        sel = np.zeros(n, bool)
        sel[got_idx[b][got_idx[b] >= 0]] = True
        slack = 2 * bounds[i].max()
        assert exact[i, :n][sel].min() >= exact[i, :n][~sel].max() - slack, f"request {b}"
    ref = oracle_attention(wl, t, got_idx, requests=None if requests is None else req)
    o = out if requests is None else out[torch.as_tensor(req, device=out.device)]
    check_attention(o, ref, name)
    del t, step
    torch.cuda.empty_cache()


def test_fp8_needs_real_weights():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    a = pks.make_args(k=wl.k, idx_fp8=True, **t)
    import ctypes
    assert pks.lib().pks_decode_workspace_size(ctypes.byref(a), ctypes.byref(ctypes.c_size_t())) == -1
