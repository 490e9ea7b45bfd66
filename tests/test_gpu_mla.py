"""GPU parity of the sparse MLA in MQA mode (tcgen05 kernel) against the oracle.

"Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraphs:
the sparse MLA runs in MQA mode over the top-k tokens, one latent row of
d + r = 512 + 64 values per token shared by H query heads.  Outputs (bf16 in,
fp32 accumulation, bf16 probabilities in the second product) within the
decode step's tolerance of the fp64 oracle; top-k indices of the full DSA step
bit-exact.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import check_attention, host
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import MlaAttention, MlaDecodeStep
from top_sparse_attention_pks_gb300.workloads import (MLA_LATENT, MLA_WORKLOADS, draw_host,
                                                      draw_mla_tensors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _prepare(wl, seed_offset=0):
    h = draw_host(wl)
    pool = pks.Pool(wl.num_pages, wl.page_size, h["free_order"])
    bt, _ = pool.build_block_table(h["seq_lens"], wl.max_pages, h["prefix_group"], wl.prefix_len)
    pool.close()
    t = draw_mla_tensors(wl, "cuda", seed_offset)
    t["seq_lens"] = h["seq_lens"].cuda()
    t["block_table"] = torch.from_numpy(bt).cuda()
    return t


def _oracle_mla(t, idx, page_size, requests=None, scale=None, q=None):
    """Oracle MLA on the selected rows only: the host gathers each request's
    selected latent rows into a compact pool of one-token pages."""
    bt = host(t["block_table"]).numpy().astype(np.int64)
    lens = host(t["seq_lens"]).numpy()
    q = host(t["q"] if q is None else q)
    idx = np.asarray(idx)
    if requests is not None:
        requests = np.asarray(requests)
        bt, lens, q, idx = bt[requests], lens[requests], q[requests], idx[requests]
    B, k = idx.shape
    max_len = int(max(1, idx.max() + 1)) if idx.size else 1
    rows, bt_c = [], np.full((B, max_len), -1, np.int32)
    for b in range(B):
        sel = idx[b][idx[b] >= 0]
        assert (sel < lens[b]).all()
        phys = bt[b, sel // page_size] * page_size + sel % page_size
        bt_c[b, sel] = np.arange(len(rows), len(rows) + len(sel), dtype=np.int32)
        rows.extend(phys.tolist())
    kv = t["kv"]
    dk = kv.shape[-1]
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=kv.device)
    pool = host(kv.reshape(-1, dk).index_select(0, r)).reshape(-1, 1, dk)
    if len(rows) == 0:
        pool = torch.zeros((1, 1, dk), dtype=torch.bfloat16)
    return oracle.mla_sparse_attention(bt_c, 1, idx, q, pool, MLA_LATENT, scale)


def _random_lists(rng, lens, k, holes=True):
    """Per request min(k, len) distinct tokens at random positions of a k-list,
    -1 elsewhere (when holes); else the tokens first, -1 after."""
    idx = np.full((len(lens), k), -1, np.int32)
    for b, n in enumerate(lens):
        m = min(k, int(n))
        sel = rng.choice(int(n), size=m, replace=False).astype(np.int32) if m else []
        pos = np.sort(rng.choice(k, size=m, replace=False)) if holes else np.arange(m)
        idx[b, pos] = sel
    return idx


@pytest.mark.parametrize("H", [128, 64, 24])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_mla_random_lists(H, splits):
    wl = MLA_WORKLOADS["mla_paging_example"]
    t = _prepare(wl)
    q = t["q"][:, :H].contiguous()
    rng = np.random.default_rng(H * 10 + splits)
    k = 96  # three tiles of 32 and lists with holes
    idx = _random_lists(rng, host(t["seq_lens"]).numpy(), k)
    idx_d = torch.from_numpy(idx).cuda()
    att = MlaAttention(t["seq_lens"], t["block_table"], idx_d, q, t["kv"], splits=splits)
    out = att()
    torch.cuda.synchronize()
    assert att.device_error() == 0
    ref = _oracle_mla(t, idx, wl.page_size, q=q)
    check_attention(out, ref, f"H={H} splits={splits}")


def test_mla_long_lists_many_tiles_and_scale():
    """k = 2048 positions in 32 tiles over 2 splits; a non-default softmax scale
    large enough that the running max moves several times (O rescaled in TMEM)."""
    wl = MLA_WORKLOADS["mla_paging_example"].replace(seq_lens=(3000, 2500), B=2, num_pages=400,
                                                     max_pages=200)
    t = _prepare(wl)
    rng = np.random.default_rng(7)
    idx = _random_lists(rng, [3000, 2500], 2048, holes=False)
    idx_d = torch.from_numpy(idx).cuda()
    for scale in (0.0, 0.35):
        att = MlaAttention(t["seq_lens"], t["block_table"], idx_d, t["q"], t["kv"],
                           sm_scale=scale, splits=2)
        out = att()
        torch.cuda.synchronize()
        ref = _oracle_mla(t, idx, wl.page_size, scale=scale or None)
        check_attention(out, ref, f"scale={scale}")


def test_mla_more_tiles_than_one_cta_holds():
    """k = 4096 positions (64 tiles) with splits = 1: the library raises the
    split count so that no CTA takes more than 32 tiles, and the partials of
    the raised splits are merged as usual."""
    wl = MLA_WORKLOADS["mla_paging_example"].replace(seq_lens=(5000, 4500), B=2, num_pages=700,
                                                     max_pages=320)
    t = _prepare(wl)
    rng = np.random.default_rng(8)
    idx = _random_lists(rng, [5000, 4500], 4096)
    idx_d = torch.from_numpy(idx).cuda()
    att = MlaAttention(t["seq_lens"], t["block_table"], idx_d, t["q"], t["kv"], splits=1)
    out = att()
    torch.cuda.synchronize()
    assert att.device_error() == 0
    check_attention(out, _oracle_mla(t, idx, wl.page_size), "k = 4096, splits 1 -> 2")


def test_mla_decode_step_paging_example():
    wl = MLA_WORKLOADS["mla_paging_example"]
    t = _prepare(wl)
    step = MlaDecodeStep(t, wl.k)
    out, idx = step()
    torch.cuda.synchronize()
    lens = host(t["seq_lens"]).numpy()
    scores = oracle.indexer_scores(lens, host(t["block_table"]).numpy(), wl.page_size,
                                   host(t["q_idx"]).numpy(), host(t["w_idx"]).numpy(),
                                   host(t["idx_k"]).numpy())
    ref_idx = oracle.topk(lens, scores, wl.k)
    assert (host(idx).numpy() == ref_idx).all(), "top-k indices differ"
    check_attention(out, _oracle_mla(t, ref_idx, wl.page_size), "mla decode step")
    assert step.attention.device_error() == 0


def test_mla_empty_requests_and_device_checks():
    wl = MLA_WORKLOADS["mla_paging_example"].replace(seq_lens=(0, 40, 100), B=3)
    t = _prepare(wl)
    idx = np.full((3, 64), -1, np.int32)
    idx[1, :40] = np.arange(40)
    idx[2, :5] = [1, 2, 3, 99, 100]  # 100 is past the request's length: skipped, flagged
    att = MlaAttention(t["seq_lens"], t["block_table"], torch.from_numpy(idx).cuda(), t["q"],
                       t["kv"], splits=1)
    out = att()
    torch.cuda.synchronize()
    assert att.device_error() == 2
    assert att.device_error() == 0  # cleared by the read
    o = out.float()
    assert torch.isfinite(o).all()
    assert not o[0].any(), "a request with no token gets zeros"
    ok = idx.copy()
    ok[2, 4] = -1
    check_attention(out[1:], _oracle_mla(t, ok, wl.page_size, requests=[1, 2]), "checks")


def test_mla_rejects_bad_shapes():
    wl = MLA_WORKLOADS["mla_paging_example"]
    t = _prepare(wl)
    idx = torch.full((wl.B, 64), -1, dtype=torch.int32, device="cuda")
    att = MlaAttention(t["seq_lens"], t["block_table"], idx, t["q"], t["kv"])
    a = att.args
    a.H = 129
    with pytest.raises(pks.PksError, match="INVALID"):
        pks.pks_mla_sparse_attention(a)
    a.H, a.d_rope = 128, 32
    with pytest.raises(pks.PksError, match="UNSUPPORTED"):
        pks.pks_mla_sparse_attention(a)
    a.d_rope, a.workspace_bytes = 64, 0
    with pytest.raises(pks.PksError, match="WORKSPACE"):
        pks.pks_mla_sparse_attention(a)


# requests compared at full size (the oracle's MLA is 128 heads x 2048 rows each)
FULL_SAMPLED = {"mla_b16_128k": [0, 5, 15], "mla_b64_32k_h64": [0, 17, 63]}


@pytest.mark.parametrize("name", ["mla_b16_128k", "mla_b64_32k_h64"])
def test_mla_full_size(name):
    wl = MLA_WORKLOADS[name]
    t = _prepare(wl)
    step = MlaDecodeStep(t, wl.k)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.attention.device_error() == 0
    req = FULL_SAMPLED[name]
    lens = host(t["seq_lens"]).numpy()[req]
    bt = host(t["block_table"]).numpy()[req]
    scores = oracle.indexer_scores(lens, bt, wl.page_size, host(t["q_idx"]).numpy()[req],
                                   host(t["w_idx"]).numpy(), host(t["idx_k"]).numpy())
    ref_idx = oracle.topk(lens, scores, wl.k)
    got = host(idx).numpy()[req]
    assert (got == ref_idx).all(), "top-k indices differ"
    ref = _oracle_mla(t, host(idx).numpy(), wl.page_size, requests=req)
    check_attention(out[torch.as_tensor(req, device=out.device)], ref, name)
    del t, step
    torch.cuda.empty_cache()


def test_dsa_step_fp8_indexer_real_weights_mla():
    """The full DSA step: FP8 e4m3 indexer with real head weights, top-k, sparse
    MLA.  Top-k exact against the oracle run on the GPU's own scores' order is
    covered by the FP8 tests; here the MLA over the step's selection."""
    from top_sparse_attention_pks_gb300.workloads import draw_float_weights, draw_fp8_indexer
    wl = MLA_WORKLOADS["mla_paging_example"]
    t = _prepare(wl)
    t["q_idx"], t["idx_k"] = draw_fp8_indexer(wl, "cuda")
    t["w_idx_f"] = draw_float_weights(wl, "cuda", signed=True)
    t["idx_fp8"] = True
    step = MlaDecodeStep(t, wl.k)
    out, idx = step()
    torch.cuda.synchronize()
    got = host(idx).numpy()
    lens = host(t["seq_lens"]).numpy()
    exact = oracle.indexer_scores_fp8(lens, host(t["block_table"]).numpy(), wl.page_size,
                                      host(t["q_idx"]), host(t["w_idx_f"]).numpy(),
                                      host(t["idx_k"]))
    for b, n in enumerate(lens):
        sel = got[b][got[b] >= 0]
        assert len(sel) == min(n, wl.k) and (np.diff(sel) > 0).all()
        if n > wl.k:  # the exact top scores are selected up to fp32 rounding
            unsel = np.setdiff1d(np.arange(n), sel)
            assert exact[b, sel].min() >= exact[b, unsel].max() - 1e-3 * np.abs(exact[b, :n]).max()
    check_attention(out, _oracle_mla(t, got, wl.page_size), "dsa step")


@pytest.mark.parametrize("page_size", [1, 64])
def test_mla_page_sizes(page_size):
    lens = (403, 96, 241, 30, 176)
    npages = sum(-(-n // page_size) for n in lens) + 3
    wl = MLA_WORKLOADS["mla_paging_example"].replace(
        page_size=page_size, num_pages=npages, max_pages=-(-max(lens) // page_size))
    t = _prepare(wl)
    rng = np.random.default_rng(page_size)
    idx = _random_lists(rng, lens, 80)
    att = MlaAttention(t["seq_lens"], t["block_table"], torch.from_numpy(idx).cuda(), t["q"],
                       t["kv"])
    out = att()
    torch.cuda.synchronize()
    assert att.device_error() == 0
    check_attention(out, _oracle_mla(t, idx, page_size), f"page_size={page_size}")


def test_mla_one_head_one_token_and_one_split():
    wl = MLA_WORKLOADS["mla_paging_example"]
    t = _prepare(wl)
    q1 = t["q"][:, :1].contiguous()
    idx = np.full((wl.B, 1), -1, np.int32)
    idx[:, 0] = [5, 0, 240, 29, 100]
    att = MlaAttention(t["seq_lens"], t["block_table"], torch.from_numpy(idx).cuda(), q1, t["kv"])
    out = att()
    torch.cuda.synchronize()
    # one selected token: the output is its latent row (to bf16 rounding)
    check_attention(out, _oracle_mla(t, idx, wl.page_size, q=q1), "one head, one token")
    # every request's whole list in one CTA pair (splits = 1), 2048 positions
    wl2 = MLA_WORKLOADS["mla_paging_example"].replace(seq_lens=(3000,), B=1, num_pages=200,
                                                      max_pages=190)
    t2 = _prepare(wl2)
    idx2 = _random_lists(np.random.default_rng(3), [3000], 2048, holes=False)
    att2 = MlaAttention(t2["seq_lens"], t2["block_table"], torch.from_numpy(idx2).cuda(), t2["q"],
                        t2["kv"], splits=1)
    out2 = att2()
    torch.cuda.synchronize()
    check_attention(out2, _oracle_mla(t2, idx2, wl2.page_size), "one split, 32 tiles")


@pytest.mark.parametrize("splits", [1, 2])
def test_mla_more_ctas_than_sms(splits):
    """96 requests, one or two splits each: 192 or 384 CTAs of 230 KB, so later
    waves allocate tensor memory after earlier ones have freed it (with two
    splits the merge kernel follows, launched as a programmatic dependent)."""
    lens = tuple(int(x) for x in np.random.default_rng(9).integers(1, 300, size=96))
    npages = sum(-(-n // 16) for n in lens)
    wl = MLA_WORKLOADS["mla_paging_example"].replace(
        B=96, seq_lens=lens, num_pages=npages, max_pages=-(-max(lens) // 16))
    t = _prepare(wl)
    idx = _random_lists(np.random.default_rng(10), lens, 128)
    att = MlaAttention(t["seq_lens"], t["block_table"], torch.from_numpy(idx).cuda(), t["q"],
                       t["kv"], splits=splits)
    for _ in range(2):
        out = att()
    torch.cuda.synchronize()
    assert att.device_error() == 0
    check_attention(out, _oracle_mla(t, idx, wl.page_size), "96 requests")
