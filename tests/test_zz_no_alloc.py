"""pks_sparse_attention_static: attention with the library's fixed device
scratch instead of a caller workspace.  Compared through the C ABI with
pks_sparse_attention (same arguments, same grid) on two calls in a row, and
with the oracle.  Collected last so that it also runs after every other test;
it sets up its own inputs and passes alone in a fresh process too."""

import numpy as np
import pytest
import torch

from gpu_cases import MAX_ABS, REL_L2, check_attention, oracle_attention, prepare
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.decoder import SparseDecodeStep
from top_sparse_attention_pks_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def _compare(a: torch.Tensor, b: torch.Tensor, what: str):
    x, y = a.double(), b.double()
    max_abs = float((x - y).abs().max())
    rel = float((x - y).norm() / y.norm())
    assert torch.isfinite(x).all(), what
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: {max_abs:.3e} / {rel:.3e}"


CASES = {
    "paging_example": dict(),
    "paging_example_gqa16": dict(Hq=16, Hkv=1, k=200),
    "b32_4k_reduced": dict(B=4, seq_lens=(4096, 4000, 1, 0), num_pages=256),
}


@pytest.mark.parametrize("case", list(CASES))
def test_static_scratch_matches_workspace_entry_point(case):
    base = "b32_4k" if case.startswith("b32") else "paging_example"
    wl = WORKLOADS[base].replace(**CASES[case])
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    step()  # the step's own top-k selection feeds both attention calls
    torch.cuda.synchronize()
    idx = step.topk_idx.cpu().numpy()

    step.attention_only()  # existing entry point, caller workspace
    torch.cuda.synchronize()
    ref = step.out.clone()

    args = pks.make_args(k=wl.k, topk_idx=step.topk_idx, out=step.out, **t)  # no workspace
    pks.pks_sparse_attention_static(args)  # first call: per-device set-up
    torch.cuda.synchronize()
    _compare(step.out, ref, f"{case}: call 1")
    free_before = torch.cuda.mem_get_info()[0]
    for call in (2, 3):
        step.out.fill_(float("nan"))
        pks.pks_sparse_attention_static(args)
        torch.cuda.synchronize()
        _compare(step.out, ref, f"{case}: call {call}")
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed across calls"
    check_attention(step.out, oracle_attention(wl, t, idx), f"{case}: oracle")


def test_static_scratch_rejects_shapes_beyond_its_size():
    wl = WORKLOADS["paging_example"]
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    step()
    torch.cuda.synchronize()
    before = step.out.clone()
    # 1024 attention CTAs x 8 query heads x (64 + 2) floats fit; 1024 CTAs of
    # a 64-head, D=128 request group do not: 8 MiB < (1024 + 1) * 64 * 130 * 4
    wl2 = WORKLOADS["paging_example"].replace(Hq=64, Hkv=8, D=128, B=1, seq_lens=(403,))
    t2, _, _ = prepare(wl2)
    out2 = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    idx2 = torch.full((1, wl2.k), -1, dtype=torch.int32, device="cuda")
    args = pks.make_args(k=wl2.k, topk_idx=idx2, out=out2, attn_splits=1024, **t2)
    with pytest.raises(pks.PksError) as ei:
        pks.pks_sparse_attention_static(args)
    assert ei.value.code == -8
    torch.cuda.synchronize()
    assert torch.equal(out2, torch.zeros_like(out2)), "a rejected call wrote output"
    # a call that fits still works after the rejection
    args_ok = pks.make_args(k=wl.k, topk_idx=step.topk_idx, out=step.out, **t)
    pks.pks_sparse_attention_static(args_ok)
    torch.cuda.synchronize()
    _compare(step.out, before, "after rejection")


def test_static_call_with_smaller_batch_keeps_workspace_path_working():
    """The two entry points share one attention kernel and its shared-memory
    limit, which grows with the batch.  A static call with a smaller batch
    between two workspace calls with a larger one must not lower that limit:
    the second workspace call has to launch and match the oracle."""
    wl = WORKLOADS["b32_4k"].replace(B=6, seq_lens=(4096, 3000, 4096, 17, 2500, 4096),
                                     num_pages=512)
    t, _, _ = prepare(wl)
    step = SparseDecodeStep(t, wl.k)
    step()  # workspace path at B = 6
    torch.cuda.synchronize()
    idx = step.topk_idx.cpu().numpy()
    ref = oracle_attention(wl, t, idx)
    check_attention(step.out, ref, "workspace call before the static one")

    wl1 = wl.replace(B=1, seq_lens=(4096,))
    t1, _, _ = prepare(wl1)
    step1 = SparseDecodeStep(t1, wl1.k)
    step1()
    torch.cuda.synchronize()
    out1 = torch.full_like(step1.out, float("nan"))
    args1 = pks.make_args(k=wl1.k, topk_idx=step1.topk_idx, out=out1, **t1)
    pks.pks_sparse_attention_static(args1)  # same D and head group, smaller batch
    torch.cuda.synchronize()
    check_attention(out1, oracle_attention(wl1, t1, step1.topk_idx.cpu().numpy()),
                    "static call with one request")

    step.out.fill_(float("nan"))
    step()  # workspace path at B = 6 again: the limit it needs is still set
    torch.cuda.synchronize()
    assert (step.topk_idx.cpu().numpy() == idx).all()
    check_attention(step.out, ref, "workspace call after the static one")
