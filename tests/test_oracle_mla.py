"""Pins of the oracle's sparse MLA in MQA mode.

"Sparse Attention on GLM5.3 and HBM", DeepSeek Sparse Attention paragraphs:
the sparse MLA runs in MQA mode, so every token keeps one latent row of
d + r values (latent d = 512, RoPE r = 64 in the pages' DeepSeek V3.2
configuration) that all query heads share; attention scores use the whole
row and the output is a weighted sum of the latent part.

Pins: a library dense attention (torch, float64, value width d) for k >= len,
the reduction to the already pinned GQA oracle with one KV head, closed forms
for one token and for a zero query, the RoPE part entering the scores but not
the values, the scale argument, and paging invariance.
"""

import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _contiguous(rng, lens, page, H, d, r):
    max_pages = -(-max(lens) // page)
    bt = np.full((len(lens), max_pages), -1, np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        npg = -(-n // page)
        bt[b, :npg] = np.arange(nxt, nxt + npg)
        nxt += npg
    kv = _bf16(rng.standard_normal((nxt, page, d + r)))
    q = _bf16(rng.standard_normal((len(lens), H, d + r)))
    return bt, kv, q


def _dense_idx(lens, k):
    idx = np.full((len(lens), k), -1, np.int32)
    for b, n in enumerate(lens):
        idx[b, :n] = np.arange(n)
    return idx


@pytest.mark.parametrize("H,d,r", [(16, 64, 16), (8, 512, 64), (3, 32, 0)])
def test_dense_matches_library_sdpa(H, d, r):
    rng = np.random.default_rng(1)
    lens, page = [29, 64, 3], 16
    bt, kv, q = _contiguous(rng, lens, page, H, d, r)
    scale = 0.37 / np.sqrt(d + r)
    out = oracle.mla_sparse_attention(bt, page, _dense_idx(lens, 64), q, kv, d, scale)
    flat = kv.double().reshape(-1, d + r)
    off = 0
    for b, n in enumerate(lens):
        rows = flat[off: off + -(-n // page) * page][:n]
        off += -(-n // page) * page
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double()[None], rows[None], rows[None, :, :d], scale=float(scale))[0]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_reduces_to_gqa_oracle_with_one_kv_head():
    """With scale 1/sqrt(d + r) the MLA is the GQA oracle with Hkv = 1, K = V =
    the latent row, output truncated to the first d values."""
    rng = np.random.default_rng(2)
    lens, page, H, d, r, k = [50, 17, 33], 8, 12, 48, 16, 20
    bt, kv, q = _contiguous(rng, lens, page, H, d, r)
    idx = np.full((3, k), -1, np.int32)
    for b, n in enumerate(lens):
        sel = np.sort(rng.choice(n, size=min(n, k), replace=False))
        idx[b, :len(sel)] = sel
    got = oracle.mla_sparse_attention(bt, page, idx, q, kv, d)
    pool = kv.reshape(kv.shape[0], page, 1, d + r)
    ref = oracle.sparse_attention(bt, page, idx, q, pool, pool)[:, :, :d]
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_single_token_returns_its_latent():
    rng = np.random.default_rng(3)
    bt, kv, q = _contiguous(rng, [40], 8, 4, 32, 8)
    idx = np.array([[-1, 13, -1]], np.int32)
    out = oracle.mla_sparse_attention(bt, 8, idx, q, kv, 32)
    want = kv.double().reshape(-1, 40)[13, :32].numpy()
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], want)


def test_zero_query_averages_latents():
    rng = np.random.default_rng(4)
    bt, kv, q = _contiguous(rng, [21], 4, 2, 16, 8)
    q = torch.zeros_like(q)
    sel = [0, 5, 6, 20]
    idx = np.array([sel + [-1]], np.int32)
    out = oracle.mla_sparse_attention(bt, 4, idx, q, kv, 16)
    want = kv.double().reshape(-1, 24)[sel, :16].mean(0).numpy()
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-15)


def test_rope_part_enters_scores_not_values():
    rng = np.random.default_rng(5)
    d, r = 16, 8
    bt, kv, q = _contiguous(rng, [30], 8, 3, d, r)
    idx = _dense_idx([30], 32)
    base = oracle.mla_sparse_attention(bt, 8, idx, q, kv, d)
    # query with a zero RoPE part: the keys' RoPE values do not matter
    q0 = q.clone()
    q0[..., d:] = 0
    kv2 = kv.clone()
    kv2[..., d:] = _bf16(rng.standard_normal(kv2[..., d:].shape))
    np.testing.assert_array_equal(oracle.mla_sparse_attention(bt, 8, idx, q0, kv, d),
                                  oracle.mla_sparse_attention(bt, 8, idx, q0, kv2, d))
    # with a RoPE query they do
    assert np.abs(oracle.mla_sparse_attention(bt, 8, idx, q, kv2, d) - base).max() > 1e-3


def test_scale_argument():
    rng = np.random.default_rng(6)
    bt, kv, q = _contiguous(rng, [19], 4, 2, 8, 8)
    idx = _dense_idx([19], 19)
    default = oracle.mla_sparse_attention(bt, 4, idx, q, kv, 8)
    np.testing.assert_array_equal(default,
                                  oracle.mla_sparse_attention(bt, 4, idx, q, kv, 8, 0.25))
    assert np.abs(oracle.mla_sparse_attention(bt, 4, idx, q, kv, 8, 0.5) - default).max() > 1e-3


def test_paging_invariance_and_empty_selection():
    rng = np.random.default_rng(7)
    d, r, n = 16, 8, 37
    bt1, kv1, q = _contiguous(rng, [n], 1, 2, d, r)  # page size 1
    # the same tokens in pages of 8, pages placed in reverse pool order
    npg = -(-n // 8)
    kv8 = torch.zeros((npg, 8, d + r), dtype=torch.bfloat16)
    flat = kv1.reshape(-1, d + r)
    bt8 = np.array([[npg - 1 - p for p in range(npg)]], np.int32)
    for t in range(n):
        kv8[bt8[0, t // 8], t % 8] = flat[t]
    idx = np.array([[2, 3, 11, 36, -1]], np.int32)
    np.testing.assert_array_equal(oracle.mla_sparse_attention(bt1, 1, idx, q, kv1, d),
                                  oracle.mla_sparse_attention(bt8, 8, idx, q, kv8, d))
    none = np.full((1, 5), -1, np.int32)
    assert not oracle.mla_sparse_attention(bt8, 8, none, q, kv8, d).any()
