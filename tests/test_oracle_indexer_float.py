"""Pins of the oracle's indexer with real-valued head weights.

"Sparse Attention on GLM5.3 and HBM", lightning indexer paragraph: a token's
index score is a weighted sum of the query heads' ReLU logits, and the top-K
tokens by that score are kept (dense below K).  With real weights the score
is a floating-point sum whose value depends on the order of the additions;
the pages fix none, so both sides follow one convention: fp32, heads in
order, each product and sum rounded to nearest on its own.

Pins: integer-valued weights reproduce the exact integer oracle (scores and
selection); scaling the weights by a power of two scales the scores exactly
and keeps the selection; the fp32 score lies within the rounding bound of the
float64 definition; the head order is the stated one (a case where another
order gives another value); equal scores go to the lower token, -0 equals +0;
negative weights.
"""

import numpy as np
import pytest

import oracle


def _case(rng, lens, page=8, Hi=4, Di=32):
    max_pages = -(-max(lens) // page)
    bt = np.full((len(lens), max_pages), -1, np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        npg = -(-n // page)
        bt[b, :npg] = np.arange(nxt, nxt + npg)
        nxt += npg
    idx_k = rng.integers(-127, 128, size=(nxt, page, Di), dtype=np.int8)
    q_idx = rng.integers(-127, 128, size=(len(lens), Hi, Di), dtype=np.int8)
    return np.asarray(lens, np.int32), bt, q_idx, idx_k


@pytest.mark.parametrize("Hi", [1, 4, 8])
def test_integer_weights_reproduce_the_integer_oracle(Hi):
    rng = np.random.default_rng(Hi)
    lens, bt, q, ik = _case(rng, [300, 41, 129], Hi=Hi)
    w_int = rng.integers(0, 4, size=Hi).astype(np.int32)
    wf = np.tile(w_int.astype(np.float32), (3, 1))
    si = oracle.indexer_scores(lens, bt, 8, q, w_int, ik)
    sf = oracle.indexer_scores_f(lens, bt, 8, q, wf, ik)
    # integer sums below 2^24 are exact in fp32
    assert np.abs(si).max() < 2 ** 24
    np.testing.assert_array_equal(sf.astype(np.int64), si)
    np.testing.assert_array_equal(oracle.topk_f(lens, sf, 64), oracle.topk(lens, si, 64))


def test_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(3)
    lens, bt, q, ik = _case(rng, [200, 77])
    wf = rng.standard_normal((2, 4)).astype(np.float32)
    s1 = oracle.indexer_scores_f(lens, bt, 8, q, wf, ik)
    s8 = oracle.indexer_scores_f(lens, bt, 8, q, wf * np.float32(8), ik)
    np.testing.assert_array_equal(s8, s1 * np.float32(8))
    np.testing.assert_array_equal(oracle.topk_f(lens, s1, 32), oracle.topk_f(lens, s8, 32))


def test_within_rounding_of_the_float64_definition():
    rng = np.random.default_rng(4)
    lens, bt, q, ik = _case(rng, [150], Hi=8, Di=64)
    wf = (rng.standard_normal((1, 8)) * 3).astype(np.float32)
    sf = oracle.indexer_scores_f(lens, bt, 8, q, wf, ik)[0, :150].astype(np.float64)
    keys = ik.reshape(-1, 64).astype(np.int64)[:150]
    dots = np.maximum(keys @ q[0].astype(np.int64).T, 0).astype(np.float64)  # [150, 8]
    terms = dots * wf[0].astype(np.float64)
    exact = terms.sum(1)
    # 8 products and 8 sums, each within half an ulp of its result
    bound = 16 * np.finfo(np.float32).eps * np.abs(terms).sum(1)
    assert (np.abs(sf - exact) <= bound).all()


def test_heads_are_summed_in_order():
    # one key, three heads whose weighted logits are 2^25, 1, -2^25: in head
    # order (2^25 + 1) rounds to 2^25 and the score is 0 (exact value 1)
    Di = 4
    key = np.array([[[1, 0, 0, 0]]], np.int8)
    q = np.array([[[1, 0, 0, 0], [1, 0, 0, 0], [1, 0, 0, 0]]], np.int8)
    wf = np.array([[2.0 ** 25, 1.0, -(2.0 ** 25)]], np.float32)
    bt = np.array([[0]], np.int32)
    s = oracle.indexer_scores_f(np.array([1], np.int32), bt, 1, q, wf, key.reshape(1, 1, Di))
    assert s[0, 0] == 0.0
    wf2 = np.array([[2.0 ** 25, -(2.0 ** 25), 1.0]], np.float32)
    s2 = oracle.indexer_scores_f(np.array([1], np.int32), bt, 1, q, wf2, key.reshape(1, 1, Di))
    assert s2[0, 0] == 1.0


def test_ties_go_to_the_lower_token_and_signed_zeros_are_equal():
    lens = np.array([6], np.int32)
    sc = np.array([[1.5, -0.0, 2.0, 0.0, 1.5, 2.0, 9, 9]], np.float32)
    # top-4: the two 2.0s (tokens 2, 5), the 1.5s (0, 4)
    np.testing.assert_array_equal(oracle.topk_f(lens, sc, 4), [[0, 2, 4, 5]])
    # top-5 adds the lower of the two zeros: token 1 (-0) before token 3 (+0)
    np.testing.assert_array_equal(oracle.topk_f(lens, sc, 5), [[0, 1, 2, 4, 5]])


def test_negative_weights_select_the_largest_signed_scores():
    rng = np.random.default_rng(5)
    lens, bt, q, ik = _case(rng, [90], Hi=2)
    wf = np.array([[-1.0, -0.5]], np.float32)
    sf = oracle.indexer_scores_f(lens, bt, 8, q, wf, ik)
    assert (sf[0, :90] <= 0).all()
    sel = oracle.topk_f(lens, sf, 10)[0]
    order = sorted(range(90), key=lambda t: (-float(sf[0, t]), t))[:10]
    np.testing.assert_array_equal(sel, sorted(order))
