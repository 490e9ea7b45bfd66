"""Pins of the oracle's FP8 (e4m3) indexer.

"Sparse Attention on GLM5.3 and HBM": DSA's lightning indexer runs in FP8
with a weighted sum of the heads' ReLU logits.  The oracle computes each dot
product exactly (e4m3 values are integer multiples of 2^-9) and the weighted
sum in float64; it is the exact reference the GPU's fp32 tensor-core scores
are held against within a rounding bound.

Pins: every finite e4m3 code decodes as torch's float8_e4m3fn; the exact dot
equals a float64 matmul of the decoded values (exact in float64 here); inputs
whose e4m3 values are small integers give the integer oracle's scores; NaN
codes are rejected.
"""

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_codes_decode_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    for c in codes:
        got = oracle.e4m3_value(int(c))
        if np.isnan(ref[c]):
            assert np.isnan(got)
        else:
            assert got == ref[c], hex(c)


def _pool(rng, lens, page, Hi, Di, scale):
    max_pages = -(-max(lens) // page)
    bt = np.full((len(lens), max_pages), -1, np.int32)
    nxt = 0
    for b, n in enumerate(lens):
        npg = -(-n // page)
        bt[b, :npg] = np.arange(nxt, nxt + npg)
        nxt += npg
    f8 = torch.float8_e4m3fn
    k = (torch.from_numpy(rng.standard_normal((nxt, page, Di))) * scale).clamp(-448, 448).to(f8)
    q = (torch.from_numpy(rng.standard_normal((len(lens), Hi, Di))) * scale).clamp(-448, 448).to(f8)
    return np.asarray(lens, np.int32), bt, q, k


def test_exact_dot_equals_float64_matmul():
    rng = np.random.default_rng(0)
    lens, bt, q, k = _pool(rng, [40], 8, 1, 128, 30.0)
    s = oracle.indexer_scores_fp8(lens, bt, 8, q, np.ones((1, 1), np.float32), k)
    kd = k.double().reshape(-1, 128)[:40]
    ref = torch.clamp(kd @ q.double()[0, 0], min=0).numpy()
    np.testing.assert_array_equal(s[0, :40], ref)


def test_small_integer_values_match_the_integer_oracle():
    # codes of the integers -16..16 are exact; the fp8 oracle with integer
    # weights then equals the int8 oracle on the same values
    rng = np.random.default_rng(1)
    Hi, Di, page = 4, 64, 8
    lens = np.array([100, 33], np.int32)
    max_pages = 13
    bt = np.full((2, max_pages), -1, np.int32)
    bt[0, :13] = np.arange(13)
    bt[1, :5] = np.arange(13, 18)
    ki = rng.integers(-16, 17, size=(18, page, Di)).astype(np.int8)
    qi = rng.integers(-16, 17, size=(2, Hi, Di)).astype(np.int8)
    w = np.array([1, 2, 0, 3], np.int32)
    f8 = torch.float8_e4m3fn
    kf = torch.from_numpy(ki.astype(np.float32)).to(f8)
    qf = torch.from_numpy(qi.astype(np.float32)).to(f8)
    s8 = oracle.indexer_scores_fp8(lens, bt, page, qf, np.tile(w.astype(np.float32), (2, 1)), kf)
    si = oracle.indexer_scores(lens, bt, page, qi, w, ki)
    np.testing.assert_array_equal(s8, si.astype(np.float64))


def test_nan_codes_are_rejected():
    lens = np.array([1], np.int32)
    bt = np.array([[0]], np.int32)
    q = np.full((1, 1, 4), 0x38, np.uint8)  # 1.0
    k = np.array([[[0x38, 0x7F, 0, 0]]], np.uint8)  # NaN in the key
    with pytest.raises(oracle.OracleError):
        oracle.indexer_scores_fp8(lens, bt, 1, q, np.ones((1, 1), np.float32), k)
