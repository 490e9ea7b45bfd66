"""Shared set-up for the GPU parity tests: seeded inputs on the device, the
product's decode step, and the oracle's answer on host copies of the same
inputs.  No expected value here comes from the CUDA path."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from top_sparse_attention_pks_gb300 import pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import Workload, draw_host, draw_tensors

# attention tolerance of the decode step (bf16 in, fp32 accumulate) against the
# fp64 oracle
MAX_ABS = 2e-2
REL_L2 = 5e-3


def prepare(wl: Workload, device="cuda", seed_offset=0, tensors_on=None):
    """Device inputs for ``wl`` plus host-side draws; block table from the product
    allocator (itself checked against the oracle's in the host tests)."""
    h = draw_host(wl)
    pool = pks.Pool(wl.num_pages, wl.page_size, h["free_order"])
    bt, used = pool.build_block_table(h["seq_lens"], wl.max_pages, h["prefix_group"],
                                      wl.prefix_len)
    pool.close()
    t = draw_tensors(wl, tensors_on or device, seed_offset)
    t = {k: v.to(device) for k, v in t.items()}
    t["seq_lens"] = h["seq_lens"].to(device)
    t["block_table"] = torch.from_numpy(bt).to(device)
    return t, h, bt


def host(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu()


def oracle_topk(wl, t, requests=None):
    """Oracle scores (int64) and top-k for all requests or a subset."""
    lens = host(t["seq_lens"]).numpy()
    bt = host(t["block_table"]).numpy()
    q_idx = host(t["q_idx"]).numpy()
    if requests is not None:
        lens, bt, q_idx = lens[requests], bt[requests], q_idx[requests]
    idx_k = host(t["idx_k"]).numpy()
    scores = oracle.indexer_scores(lens, bt, wl.page_size, q_idx, host(t["w_idx"]).numpy(),
                                   idx_k)
    return scores, oracle.topk(lens, scores, wl.k)


def oracle_attention(wl, t, idx, requests=None):
    """Oracle attention for the given selection (all requests or a subset).

    Only the K/V rows the selection reads leave the device: the host gathers
    them into a compact pool of one-token pages (row j of request b's block
    row is the j-th selected token), and the oracle runs on that pool with
    page_size 1.  The physical row of each token is found on the host from
    the real block table."""
    bt = host(t["block_table"]).numpy().astype(np.int64)
    lens = host(t["seq_lens"]).numpy()
    q = host(t["q"])
    idx = np.asarray(idx)
    if requests is not None:
        requests = np.asarray(requests)
        bt, lens, q, idx = bt[requests], lens[requests], q[requests], idx[requests]
    P = wl.page_size
    B, k = idx.shape
    max_len = int(max(1, idx.max() + 1)) if idx.size else 1
    rows, bt_c = [], np.full((B, max_len), -1, np.int32)
    for b in range(B):
        sel = idx[b][idx[b] >= 0]
        assert (sel < lens[b]).all(), "selection beyond the request's length"
        phys = bt[b, sel // P] * P + sel % P
        bt_c[b, sel] = np.arange(len(rows), len(rows) + len(sel), dtype=np.int32)
        rows.extend(phys.tolist())
    dev = t["kv_k"].device
    Hkv, D = t["kv_k"].shape[2], t["kv_k"].shape[3]
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=dev)
    kk = host(t["kv_k"].reshape(-1, Hkv, D).index_select(0, r)).reshape(-1, 1, Hkv, D)
    vv = host(t["kv_v"].reshape(-1, Hkv, D).index_select(0, r)).reshape(-1, 1, Hkv, D)
    if len(rows) == 0:
        kk = torch.zeros((1, 1, Hkv, D), dtype=torch.bfloat16)
        vv = torch.zeros((1, 1, Hkv, D), dtype=torch.bfloat16)
    return oracle.sparse_attention(bt_c, 1, idx, q, kk, vv)


def check_attention(got: torch.Tensor, ref: np.ndarray, what=""):
    g = got.double().cpu().numpy()
    err = np.abs(g - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.sqrt((ref ** 2).sum()))
    rel = float(np.sqrt(((g - ref) ** 2).sum()) / denom) if denom > 0 else max_abs
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    assert max_abs <= MAX_ABS, f"{what}: max abs error {max_abs:.3e} > {MAX_ABS}"
    assert rel <= REL_L2, f"{what}: relative L2 error {rel:.3e} > {REL_L2}"
    return max_abs, rel


def run_step(wl, t, attn_splits=0, topk_mode=0):
    step = SparseDecodeStep(t, wl.k, attn_splits=attn_splits, topk_mode=topk_mode)
    out, idx = step()
    torch.cuda.synchronize()
    return step, out, idx
