"""The bounded device-side waits give up, report device error 5 and leave the
GPU usable.

Two waits exist: the top-k request barrier (the cooperative selection's CTAs
of one request meet there) and the mbarrier waits of the sparse MLA kernel's
warps.  Each test makes its wait run out without faking the GPU: the barrier
counter of one request starts at -1, so it needs one arrival more than the
request's CTAs make; the MLA waits get a budget of 100 clock cycles, far below
the time their copies and MMAs take.  Then the same work runs again and must
match the oracle."""

import numpy as np
import pytest
import torch

import oracle
from gpu_cases import check_attention, host, oracle_attention, oracle_topk, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import MlaAttention, SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import (MLA_LATENT, MLA_WORKLOADS, WORKLOADS,
                                                      draw_mla_tensors)

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # device error word: a bounded wait ran out


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def test_topk_barrier_wait_runs_out_and_the_step_recovers():
    # two requests of 3 and 2 chunks: the single cooperative top-k launch
    wl = WORKLOADS["paging_example"].replace(B=2, seq_lens=(10000, 7000), num_pages=1100,
                                             max_pages=640, k=64)
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k, wait_limit=100000)
    assert step.launches() == 4  # scan, cooperative top-k, attention, merge
    off = pks.pks_decode_barrier_offset(step.args)
    counters = step.workspace[off: off + 4 * wl.B].view(torch.int32)
    counters[0] = -1  # request 0's barrier now needs one more arrival than it gets
    torch.cuda.synchronize()
    _, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == TIMEOUT
    # request 1 passed its own barrier: its selection is complete and exact
    _, ref_idx = oracle_topk(wl, t)
    assert (host(idx).numpy()[1] == ref_idx[1]).all()
    # a re-initialised workspace gives the exact step again
    pks.pks_decode_workspace_init(step.args)
    out, idx = step()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    got = host(idx).numpy()
    assert (got == ref_idx).all()
    check_attention(out, oracle_attention(wl, t, ref_idx), "after the time-out")


def test_mla_mbarrier_waits_run_out_and_the_kernel_recovers():
    wl = WORKLOADS["paging_example"]
    mwl = MLA_WORKLOADS["mla_paging_example"]
    t, h, bt = prepare(wl)
    _, ref_idx = oracle_topk(wl, t)
    mt = draw_mla_tensors(mwl, "cpu")
    mbt = np.full((wl.B, mwl.max_pages), -1, np.int32)
    mbt[:, : bt.shape[1]] = bt
    dev = t["q"].device
    args = (t["seq_lens"], torch.from_numpy(mbt).to(dev), torch.from_numpy(ref_idx).to(dev),
            mt["q"].to(dev), mt["kv"].to(dev))
    short = MlaAttention(*args, splits=2, wait_limit=100)
    short()
    torch.cuda.synchronize()
    assert short.device_error() == TIMEOUT
    # the tensor memory was released and the GPU is usable: a default budget
    # gives the right answer on the same device
    full = MlaAttention(*args, splits=2)
    out = full()
    torch.cuda.synchronize()
    assert full.device_error() == 0
    ref = oracle.mla_sparse_attention(mbt, mwl.page_size, ref_idx, mt["q"], mt["kv"], MLA_LATENT)
    check_attention(out, ref, "MLA after the time-out")
