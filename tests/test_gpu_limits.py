"""Parity at the limits the C ABI accepts: the largest batch (4096 requests),
the largest k (65536, with a request just above and one exactly at it), a
1.5M-token request (367 top-k chunks meeting at one barrier), and an empty
batch.  Top-k bit-exact, attention within tolerance."""

import numpy as np
import pytest
import torch

from gpu_cases import check_attention, host, oracle_attention, oracle_topk, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _check(wl, t, **kw):
    step = SparseDecodeStep(t, wl.k, **kw)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    _, ref_idx = oracle_topk(wl, t)
    assert (host(idx).numpy() == ref_idx).all(), "top-k"
    return step, out, ref_idx


def test_largest_batch():
    rng = np.random.default_rng(21)
    lens = tuple(int(x) for x in rng.integers(0, 200, size=4096))
    wl = WORKLOADS["paging_example"].replace(B=4096, seq_lens=lens, k=48, page_size=16,
                                             max_pages=13, num_pages=4096 * 13)
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    step.out.fill_(float("nan"))  # every output must be written, empty requests too
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    _, ref_idx = oracle_topk(wl, t)
    assert (host(idx).numpy() == ref_idx).all(), "top-k"
    req = list(range(0, 4096, 97)) + [4095]
    o = out[torch.as_tensor(req, device=out.device)]
    check_attention(o, oracle_attention(wl, t, ref_idx, requests=req), "B = 4096")
    # requests of length 0 (spread over the whole batch) get zero outputs
    empty = [b for b, n in enumerate(lens) if n == 0]
    assert any(b >= 256 for b in empty)
    assert (out[torch.as_tensor(empty, device=out.device)].float() == 0).all()


def test_largest_k():
    wl = WORKLOADS["paging_example"].replace(
        B=3, seq_lens=(70000, 65536, 1000), k=65536, page_size=64, max_pages=1100,
        num_pages=3 * 1100, Di=64, D=64, Hq=4, Hkv=1)
    t, _, _ = prepare(wl)
    step, out, ref_idx = _check(wl, t)
    assert (ref_idx[1] == np.arange(65536)).all()  # exactly k tokens: dense
    check_attention(out, oracle_attention(wl, t, ref_idx), "k = 65536")


def test_one_and_a_half_million_token_request():
    n = 1_500_000
    wl = WORKLOADS["paging_example"].replace(
        B=1, seq_lens=(n,), k=2048, page_size=64, max_pages=-(-n // 64),
        num_pages=-(-n // 64) + 100, Di=64, D=64, Hq=8, Hkv=2, Hi=2)
    t, _, _ = prepare(wl)
    step, out, ref_idx = _check(wl, t)
    assert step.launches() == 4  # one cooperative top-k launch for 367 chunks
    check_attention(out, oracle_attention(wl, t, ref_idx), "1.5M tokens")


def test_empty_batch_launches_nothing():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    t0 = {k: (v[:0] if k in ("seq_lens", "block_table", "q", "q_idx") else v) for k, v in t.items()}
    step = SparseDecodeStep(t0, wl.k)
    assert step.launches() == 0
    step()  # no device work, no error
    torch.cuda.synchronize()
    assert step.device_error() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_real_weights_at_the_limits(fp8):
    """fp32 keys (real head weights, and FP8 e4m3 inputs) through the largest k
    and a 1.5M-token request: the selection is bit-exact against the oracle's
    top-k on the kernel's own scores (and, with int8 inputs, on the oracle's)."""
    import oracle
    from top_sparse_attention_pks_gb300.workloads import draw_float_weights, draw_fp8_indexer
    n = 1_500_000
    wl = WORKLOADS["paging_example"].replace(
        B=3, seq_lens=(n, 70000, 1000), k=65536, page_size=64, max_pages=-(-n // 64),
        num_pages=-(-n // 64) + 1200 + 20, Di=64, D=64, Hq=4, Hkv=1, Hi=2)
    t, _, _ = prepare(wl)
    if fp8:
        t["q_idx"], t["idx_k"] = draw_fp8_indexer(wl, "cuda")
        t["idx_fp8"] = True
    t["w_idx_f"] = draw_float_weights(wl, "cuda", signed=True)
    step = SparseDecodeStep(t, wl.k)
    _, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    lens = host(t["seq_lens"]).numpy()
    got_sc = pks.float_key_to_score(host(step.scores()).numpy())
    got = host(idx).numpy()
    np.testing.assert_array_equal(got, oracle.topk_f(lens, got_sc, wl.k))
    if not fp8:
        ref_sc = oracle.indexer_scores_f(lens, host(t["block_table"]).numpy(), wl.page_size,
                                         host(t["q_idx"]).numpy(), host(t["w_idx_f"]).numpy(),
                                         host(t["idx_k"]).numpy())
        for b, m in enumerate(lens):
            np.testing.assert_array_equal(got_sc[b, :m], ref_sc[b, :m])
    del t, step
    torch.cuda.empty_cache()
