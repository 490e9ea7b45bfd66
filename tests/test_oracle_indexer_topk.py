"""Pins of the oracle's indexer scores and top-k selection.

The lightning indexer of "Sparse Attention on GLM5.3 and HBM" (DeepSeek Sparse
Attention paragraph): per indexer head a query-key dot product, a ReLU, then a
weighted sum over heads; the top-K tokens by that score are shared by all
attention heads, and a query with fewer than K tokens stays dense.  Ties go to
the lower token index (the ordering fixed for bit-exact comparison).

The pins are closed forms and brute force, never the oracle's own formula.
"""

import numpy as np
import pytest

import oracle


def _pool(rng, num_pages, page, di):
    return rng.integers(-127, 128, size=(num_pages, page, di), dtype=np.int8)


def _identity_table(lens, page, max_pages):
    """Block table that lays each request's pages out contiguously, in order."""
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        np_ = -(-n // page)
        bt[b, :np_] = np.arange(nxt, nxt + np_)
        nxt += np_
    return bt, nxt


def _logical_keys(pool, lens, page):
    """Logical keys of each request under the identity table (pool order)."""
    flat = pool.reshape(-1, pool.shape[-1])
    out, off = [], 0
    for n in lens:
        out.append(flat[off: off + n])
        off += -(-n // page) * page
    return out


def test_unit_query_picks_a_key_column():
    rng = np.random.default_rng(0)
    page, di, lens = 8, 32, [37, 8, 1]
    bt, used = _identity_table(lens, page, 8)
    pool = _pool(rng, used, page, di)
    keys = _logical_keys(pool, lens, page)
    for i in (0, 5, 31):
        for c in (1, 3):
            q = np.zeros((len(lens), 1, di), dtype=np.int8)
            q[:, 0, i] = c
            s = oracle.indexer_scores(lens, bt, page, q, np.ones(1, np.int32), pool)
            for b, n in enumerate(lens):
                expect = c * np.maximum(keys[b][:, i].astype(np.int64), 0)
                assert (s[b, :n] == expect).all()


def test_opposite_heads_give_absolute_dot():
    # relu(x) + relu(-x) = |x|: a dropped ReLU would give 0 here
    rng = np.random.default_rng(1)
    page, di, lens = 16, 64, [100, 33]
    bt, used = _identity_table(lens, page, 8)
    pool = _pool(rng, used, page, di)
    keys = _logical_keys(pool, lens, page)
    qh = rng.integers(-127, 128, size=(len(lens), di), dtype=np.int8)
    q = np.stack([qh, -qh], axis=1)
    s = oracle.indexer_scores(lens, bt, page, q, np.ones(2, np.int32), pool)
    for b, n in enumerate(lens):
        dot = keys[b].astype(np.int64) @ qh[b].astype(np.int64)
        assert (s[b, :n] == np.abs(dot)).all()


def test_head_weights_pair_with_their_heads():
    rng = np.random.default_rng(2)
    page, di, lens = 4, 16, [30]
    bt, used = _identity_table(lens, page, 8)
    pool = _pool(rng, used, page, di)
    keys = _logical_keys(pool, lens, page)[0].astype(np.int64)
    q = np.zeros((1, 3, di), dtype=np.int8)
    q[0, 0, 2] = 1
    q[0, 1, 7] = 1
    q[0, 2, 9] = 1
    s = oracle.indexer_scores(lens, bt, page, q, np.array([5, 0, -2], np.int32), pool)
    expect = 5 * np.maximum(keys[:, 2], 0) - 2 * np.maximum(keys[:, 9], 0)
    assert (s[0, :30] == expect).all()


def test_self_key_gives_squared_norm():
    di, page = 32, 4
    q = np.random.default_rng(3).integers(-127, 128, size=(1, 1, di), dtype=np.int8)
    pool = np.zeros((1, page, di), dtype=np.int8)
    pool[0, 2] = q[0, 0]
    bt = np.array([[0]], dtype=np.int32)
    s = oracle.indexer_scores([4], bt, page, q, np.ones(1, np.int32), pool)
    assert s[0, 2] == int((q.astype(np.int64) ** 2).sum())
    assert (s[0, [0, 1, 3]] == 0).all()


def test_scores_invariant_under_paging():
    # the same logical keys under several page sizes and permuted pools
    rng = np.random.default_rng(4)
    di, lens = 32, [130, 64, 7]
    logical = [rng.integers(-127, 128, size=(n, di), dtype=np.int8) for n in lens]
    q = rng.integers(-127, 128, size=(len(lens), 2, di), dtype=np.int8)
    w = np.array([1, 2], np.int32)
    ref = None
    for page in (1, 4, 16, 64, 256):
        max_pages = -(-max(lens) // page)
        num_pages = sum(-(-n // page) for n in lens) + 3
        perm = rng.permutation(num_pages).astype(np.int32)
        bt, _ = oracle.build_block_table(lens, page, max_pages, num_pages, free_order=perm)
        pool = rng.integers(-127, 128, size=(num_pages, page, di), dtype=np.int8)
        for b, n in enumerate(lens):
            for t in range(n):
                pool[bt[b, t // page], t % page] = logical[b][t]
        s = oracle.indexer_scores(lens, bt, page, q, w, pool, ld=max(lens))
        if ref is None:
            ref = s
        assert (s == ref).all()


def _brute_topk(scores_row, n, k):
    order = sorted(range(n), key=lambda t: (-int(scores_row[t]), t))
    chosen = sorted(order[:k]) if n > k else list(range(n))
    return chosen + [-1] * (k - len(chosen))


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    B, L = 6, 90
    lens = rng.integers(0, L + 1, size=B).astype(np.int32)
    lens[0] = L
    hi = [3, 10, 1000][seed % 3]  # small ranges force many ties
    scores = rng.integers(-hi, hi, size=(B, L)).astype(np.int64)
    for k in (1, 5, 17, 89, 90, 128):
        got = oracle.topk(lens, scores, k)
        for b in range(B):
            assert got[b].tolist() == _brute_topk(scores[b], int(lens[b]), k)


def test_topk_dense_and_all_ties():
    lens = np.array([10, 3, 0], np.int32)
    scores = np.zeros((3, 10), np.int64)
    got = oracle.topk(lens, scores, 4)
    assert got[0].tolist() == [0, 1, 2, 3]  # all tied: lowest indices
    assert got[1].tolist() == [0, 1, 2, -1]  # dense: fewer than k tokens
    assert got[2].tolist() == [-1] * 4
    got = oracle.topk(lens, scores, 10)
    assert got[0].tolist() == list(range(10))


def test_topk_extreme_values():
    s = np.array([[2**31 - 1, -2**31, 0, 2**31 - 1, -1]], np.int64)
    assert oracle.topk([5], s, 2)[0].tolist() == [0, 3]
    assert oracle.topk([5], s, 4)[0].tolist() == [0, 2, 3, 4]
