"""Pins of the oracle's sparse attention.

"Sparse Attention on GLM5.3 and HBM": scaled dot-product attention runs over
only the selected top-k tokens (introduction and DSA paragraph); with k at
least the context length it is ordinary dense attention.  K/V are read through
the block table of the "Paged KV cache" chapter (section "Paging").

Pins: a library dense attention (torch, float64) for k >= len, closed forms
for one token and for a zero query, the GQA head mapping, order and paging
invariance.
"""

import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)


def _contiguous_case(rng, lens, page, Hq, Hkv, D):
    """Pool whose pages hold each request's tokens in order (identity table)."""
    max_pages = -(-max(lens) // page)
    bt = np.full((len(lens), max_pages), -1, np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        npg = -(-n // page)
        bt[b, :npg] = np.arange(nxt, nxt + npg)
        nxt += npg
    kv_k = _bf16(rng.standard_normal((nxt, page, Hkv, D)))
    kv_v = _bf16(rng.standard_normal((nxt, page, Hkv, D)))
    q = _bf16(rng.standard_normal((len(lens), Hq, D)))
    return bt, kv_k, kv_v, q


def _dense_idx(lens, k):
    idx = np.full((len(lens), k), -1, np.int32)
    for b, n in enumerate(lens):
        idx[b, :n] = np.arange(n)
    return idx


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 64), (4, 4, 16), (6, 1, 32)])
def test_dense_matches_library_sdpa(Hq, Hkv, D):
    rng = np.random.default_rng(0)
    lens, page = [37, 5, 64], 16
    bt, kv_k, kv_v, q = _contiguous_case(rng, lens, page, Hq, Hkv, D)
    k = 64
    out = oracle.sparse_attention(bt, page, _dense_idx(lens, k), q, kv_k, kv_v)
    flat_k = kv_k.double().reshape(-1, Hkv, D)
    flat_v = kv_v.double().reshape(-1, Hkv, D)
    off = 0
    for b, n in enumerate(lens):
        K = flat_k[off: off + n].permute(1, 0, 2)  # [Hkv, n, D]
        V = flat_v[off: off + n].permute(1, 0, 2)
        rep = Hq // Hkv
        K = K.repeat_interleave(rep, dim=0)
        V = V.repeat_interleave(rep, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[b].double().unsqueeze(1), K, V).squeeze(1)
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)
        off += -(-n // page) * page


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    lens, page = [40], 8
    bt, kv_k, kv_v, q = _contiguous_case(rng, lens, page, 4, 2, 16)
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 3] = 29
    out = oracle.sparse_attention(bt, page, idx, q, kv_k, kv_v)
    v = kv_v.double().reshape(-1, 2, 16)[29]
    for h in range(4):
        assert (out[0, h] == v[h // 2].numpy()).all()


def test_zero_query_averages_values():
    rng = np.random.default_rng(2)
    lens, page = [50], 16
    bt, kv_k, kv_v, _ = _contiguous_case(rng, lens, page, 2, 1, 32)
    q = torch.zeros((1, 2, 32), dtype=torch.bfloat16)
    sel = [0, 7, 8, 33, 49]
    idx = np.array([sel + [-1] * 3], np.int32)
    out = oracle.sparse_attention(bt, page, idx, q, kv_k, kv_v)
    v = kv_v.double().reshape(-1, 1, 32)[sel, 0].mean(0).numpy()
    np.testing.assert_allclose(out[0, 0], v, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out[0, 1], v, rtol=1e-14, atol=1e-15)


def test_gqa_groups_are_contiguous():
    # kv head j holds the constant value j + 1: query head h must see h // G + 1
    Hq, Hkv, D, page = 6, 3, 8, 4
    kv_k = torch.randn((2, page, Hkv, D)).to(torch.bfloat16)
    kv_v = torch.zeros((2, page, Hkv, D))
    for j in range(Hkv):
        kv_v[:, :, j, :] = j + 1
    kv_v = kv_v.to(torch.bfloat16)
    q = torch.randn((1, Hq, D)).to(torch.bfloat16)
    bt = np.array([[0, 1]], np.int32)
    out = oracle.sparse_attention(bt, page, np.array([[0, 5, 6]], np.int32), q, kv_k, kv_v)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // (Hq // Hkv) + 1, rtol=1e-15)


def test_empty_selection_gives_zero():
    rng = np.random.default_rng(3)
    bt, kv_k, kv_v, q = _contiguous_case(rng, [10], 4, 2, 1, 8)
    out = oracle.sparse_attention(bt, 4, np.full((1, 4), -1, np.int32), q, kv_k, kv_v)
    assert (out == 0).all()


def test_order_and_padding_invariance():
    rng = np.random.default_rng(4)
    bt, kv_k, kv_v, q = _contiguous_case(rng, [64], 16, 4, 2, 32)
    sel = np.array([1, 5, 6, 40, 63, 20], np.int32)
    a = oracle.sparse_attention(bt, 16, sel[None], q, kv_k, kv_v)
    mixed = np.array([[-1, 63, 20, -1, 1, 40, 6, 5, -1]], np.int32)
    b = oracle.sparse_attention(bt, 16, mixed, q, kv_k, kv_v)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_paging_invariance():
    # identical logical K/V under page sizes 1/16/64/512 and permuted pools
    rng = np.random.default_rng(5)
    lens, Hq, Hkv, D, k = [300, 41], 4, 2, 16, 32
    logical_k = [rng.standard_normal((n, Hkv, D)) for n in lens]
    logical_v = [rng.standard_normal((n, Hkv, D)) for n in lens]
    q = _bf16(rng.standard_normal((2, Hq, D)))
    idx = np.stack([np.sort(rng.choice(n, size=min(n, k), replace=False)) for n in lens])
    idx = idx.astype(np.int32)
    ref = None
    for page in (1, 16, 64, 512):
        max_pages = -(-max(lens) // page)
        num_pages = sum(-(-n // page) for n in lens) + 2
        perm = rng.permutation(num_pages).astype(np.int32)
        bt, _ = oracle.build_block_table(lens, page, max_pages, num_pages, free_order=perm)
        pk = np.zeros((num_pages, page, Hkv, D), np.float32)
        pv = np.zeros((num_pages, page, Hkv, D), np.float32)
        for b, n in enumerate(lens):
            for t in range(n):
                pk[bt[b, t // page], t % page] = logical_k[b][t]
                pv[bt[b, t // page], t % page] = logical_v[b][t]
        out = oracle.sparse_attention(bt, page, idx, q, _bf16(pk), _bf16(pv))
        if ref is None:
            ref = out
        assert (out == ref).all()
