"""C-ABI checks that need no GPU: exported symbols, the host page allocator
and block-table builder (compared with the oracle), argument validation and
workspace sizing."""

import re
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from top_sparse_attention_pks_gb300 import build, pks
from top_sparse_attention_pks_gb300.workloads import WORKLOADS, draw_host

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_library()


def declared_functions():
    text = (ROOT / "include" / "pks.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pks_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert "pks_decode_step" in names and "pks_residency_update" in names
    L = pks.lib()
    for n in names:
        assert hasattr(L, n), f"libpks.so does not export {n}"


def test_status_strings():
    L = pks.lib()
    for code in range(-7, 1):
        assert L.pks_status_str(code).decode() not in ("", "unknown status")


def test_pool_fifo_and_free():
    pool = pks.Pool(8, 16)
    assert pool.alloc(3).tolist() == [0, 1, 2]
    pool.free([1])
    assert pool.alloc(5).tolist() == [3, 4, 5, 6, 7]
    assert pool.alloc(1).tolist() == [1]  # freed pages go to the back
    with pytest.raises(pks.PksError) as e:
        pool.alloc(1)
    assert e.value.code == -2
    assert pool.free_count() == 0
    with pytest.raises(pks.PksError):
        pool.free([9])  # out of range
    pool.free([0, 2])
    with pytest.raises(pks.PksError):
        pool.free([0])  # already free
    with pytest.raises(pks.PksError):
        pool.free([3, 3])  # repeated
    assert pool.free_count() == 2


def test_pool_rejects_bad_permutation():
    with pytest.raises(pks.PksError):
        pks.Pool(4, 16, free_order=[0, 1, 1, 3])


def _compare_tables(wl, **over):
    wl = wl.replace(**over) if over else wl
    h = draw_host(wl)
    ref_bt, ref_used = oracle.build_block_table(
        h["seq_lens"], wl.page_size, wl.max_pages, wl.num_pages,
        prefix_group=h["prefix_group"], prefix_len=wl.prefix_len, free_order=h["free_order"])
    pool = pks.Pool(wl.num_pages, wl.page_size, h["free_order"])
    bt, used = pool.build_block_table(h["seq_lens"], wl.max_pages, h["prefix_group"],
                                      wl.prefix_len)
    assert used == ref_used
    assert (bt == ref_bt).all()
    assert pool.free_count() == wl.num_pages - used
    return bt, used


@pytest.mark.parametrize("name", ["paging_example", "b32_4k", "b64_ragged_prefix", "b16_128k",
                                  "b256_8k_lru"])
def test_block_table_matches_oracle(name):
    bt, used = _compare_tables(WORKLOADS[name])
    if name == "b64_ragged_prefix":
        wl = WORKLOADS[name]
        lens = draw_host(wl)["seq_lens"].numpy()
        full = sum(-(-int(n) // wl.page_size) for n in lens)
        assert full - used > 0  # prefix aliasing saved pages


def test_block_table_prefix_example():
    # "Page sharing": the first three requests share 64 tokens -> 8 pages saved
    lens, group = [403, 96, 241, 30, 176], [0, 0, 0, -1, -1]
    ref_bt, ref_used = oracle.build_block_table(lens, 16, 32, 64, prefix_group=group,
                                                prefix_len=64)
    pool = pks.Pool(64, 16)
    bt, used = pool.build_block_table(lens, 32, group, 64)
    assert (bt == ref_bt).all() and used == ref_used == 61 - 8


def test_block_table_rollback_on_oom():
    pool = pks.Pool(10, 16)
    with pytest.raises(pks.PksError) as e:
        pool.build_block_table([100, 100], 8)  # needs 14 pages
    assert e.value.code == -2
    assert pool.free_count() == 10
    assert pool.alloc(10).tolist() == list(range(10))  # order restored? (FIFO back)


def test_block_table_invalid():
    pool = pks.Pool(64, 16)
    with pytest.raises(pks.PksError) as e:
        pool.build_block_table([100], 4)  # 7 pages > max_pages
    assert e.value.code == -1
    with pytest.raises(pks.PksError):
        pool.build_block_table([-1], 4)


def test_capacity_with_product_allocator():
    # "How many users": a 16384-token pool in 16-token pages admits 83 of the
    # example requests arriving cyclically
    lens = [403, 96, 241, 30, 176]
    pool = pks.Pool(16384 // 16, 16)
    admitted = 0
    while True:
        n = -(-lens[admitted % 5] // 16)
        try:
            pool.alloc(n)
        except pks.PksError as e:
            assert e.code == -2
            break
        admitted += 1
    assert admitted == oracle.capacity_paged(lens, 16, 16384) == 83


def _cpu_args(**over):
    wl = WORKLOADS["paging_example"]
    B, P = wl.B, wl.page_size
    t = dict(
        seq_lens=torch.zeros(B, dtype=torch.int32),
        block_table=torch.zeros((B, wl.max_pages), dtype=torch.int32),
        q=torch.zeros((B, wl.Hq, wl.D), dtype=torch.bfloat16),
        q_idx=torch.zeros((B, wl.Hi, wl.Di), dtype=torch.int8),
        w_idx=torch.ones(wl.Hi, dtype=torch.int32),
        kv_k=torch.zeros((wl.num_pages, P, wl.Hkv, wl.D), dtype=torch.bfloat16),
        kv_v=torch.zeros((wl.num_pages, P, wl.Hkv, wl.D), dtype=torch.bfloat16),
        idx_k=torch.zeros((wl.num_pages, P, wl.Di), dtype=torch.int8),
    )
    a = pks.make_args(k=wl.k, topk_idx=torch.zeros((B, wl.k), dtype=torch.int32),
                      out=torch.zeros((B, wl.Hq, wl.D), dtype=torch.bfloat16), **t)
    for key, v in over.items():
        setattr(a, key, v)
    return a


def test_workspace_size_and_validation_without_gpu():
    a = _cpu_args()
    n = pks.pks_decode_workspace_size(a)
    assert n > 0 and n % 256 == 0
    L = pks.lib()
    import ctypes
    # no workspace -> PKS_ERR_WORKSPACE, before any device work
    assert L.pks_decode_step(ctypes.byref(a), None) == -7
    cases = [dict(Hq=6, Hkv=4), dict(k=0), dict(page_size=0), dict(B=-1),
             dict(reserved=(ctypes.c_int32 * 1)(1)), dict(wait_limit=-1), dict(topk_mode=2), dict(topk_mode=-1), dict(n_queries=-1), dict(attn_splits=-2),
             dict(attn_splits=1025)]
    for c in cases:
        assert L.pks_decode_workspace_size(ctypes.byref(_cpu_args(**c)),
                                           ctypes.byref(ctypes.c_size_t())) == -1, c
    unsupported = [dict(D=96), dict(Di=32), dict(Hi=3), dict(Hq=64, Hkv=2), dict(B=5000),
                   dict(k=70000), dict(n_queries=3), dict(Hi=4, n_queries=4),
                   dict(B=1025, n_queries=4)]
    for c in unsupported:
        assert L.pks_decode_workspace_size(ctypes.byref(_cpu_args(**c)),
                                           ctypes.byref(ctypes.c_size_t())) == -6, c
    # null pointers are rejected
    assert L.pks_decode_step(ctypes.byref(_cpu_args(q=None)), None) == -1
    assert L.pks_indexer_scores(ctypes.byref(_cpu_args(idx_k=None)), None, 512, None) == -1


def test_static_attention_rejects_oversized_shapes_on_host():
    # the allocation-free attention checks its fixed scratch before any CUDA
    # call: 4096 requests x 64 heads x 130 floats of partials exceed 8 MiB
    import ctypes
    a = _cpu_args()
    a.B, a.Hq, a.Hkv, a.D = 4096, 64, 8, 128
    assert pks.lib().pks_sparse_attention_static(ctypes.byref(a), None) == -8
    assert pks.lib().pks_status_str(-8).decode().startswith("shapes need more scratch")


def test_workspace_size_scales_with_batch():
    small = pks.pks_decode_workspace_size(_cpu_args())
    a = _cpu_args(B=50)
    assert pks.pks_decode_workspace_size(a) > small


def test_residency_layout_on_host():
    n = pks.pks_residency_state_bytes(32768, 16384)
    off = pks.pks_residency_offsets(32768, 16384)
    assert off["page_slot"] >= 64 and all(v % 256 == 0 for v in off.values())
    assert off["slot_page"] >= off["page_slot"] + 4 * 32768
    assert n >= off["lru_order"] + 4 * 16384
    with pytest.raises(pks.PksError):
        pks.pks_residency_state_bytes(0, 4)


def _mla_cpu_args(**over):
    import ctypes
    a = pks.pks_mla_args()
    a.B, a.H, a.d_latent, a.d_rope = 16, 128, 512, 64
    a.page_size, a.max_pages, a.num_pages, a.k = 64, 2048, 32768, 2048
    for key, v in over.items():
        setattr(a, key, v)
    return a


def test_mla_workspace_and_validation_without_gpu():
    import ctypes
    L = pks.lib()
    n = ctypes.c_size_t()
    assert L.pks_mla_workspace_size(ctypes.byref(_mla_cpu_args(splits=1)), ctypes.byref(n)) == 0
    one = n.value
    assert L.pks_mla_workspace_size(ctypes.byref(_mla_cpu_args(splits=4)), ctypes.byref(n)) == 0
    # four splits: (m, l) and 512 fp32 partial values per (request, split, head)
    assert n.value >= one + 16 * 4 * 128 * (8 + 512 * 4)
    # no workspace -> PKS_ERR_WORKSPACE, before any device work
    assert L.pks_mla_sparse_attention(ctypes.byref(_mla_cpu_args(B=0, splits=2)), None) == -7
    for c in [dict(H=0), dict(H=129), dict(k=0), dict(B=-1), dict(splits=65), dict(trim=2),
              dict(sm_scale=-1.0), dict(wait_limit=-1), dict(page_size=0)]:
        assert L.pks_mla_workspace_size(ctypes.byref(_mla_cpu_args(**c)), ctypes.byref(n)) == -1, c
    for c in [dict(d_latent=256), dict(d_rope=32)]:
        assert L.pks_mla_workspace_size(ctypes.byref(_mla_cpu_args(**c)), ctypes.byref(n)) == -6, c
    # null device pointers with B > 0
    a = _mla_cpu_args()
    assert L.pks_mla_sparse_attention(ctypes.byref(a), None) == -1


def test_mla_split_count_keeps_each_cta_within_32_tiles():
    # k = 4096: 64 tiles of 64 tokens; one split would give a CTA 64 tiles, so
    # the library raises it to two (the workspace then holds two splits'
    # partials, exactly as with splits = 2); k = 2048 keeps one split (no
    # partials at all)
    import ctypes
    L = pks.lib()
    n = ctypes.c_size_t()
    sizes = {}
    for k, splits in [(4096, 1), (4096, 2), (4096, 3), (2048, 1)]:
        assert L.pks_mla_workspace_size(ctypes.byref(_mla_cpu_args(k=k, splits=splits)),
                                        ctypes.byref(n)) == 0
        sizes[(k, splits)] = n.value
    assert sizes[(4096, 1)] == sizes[(4096, 2)]
    assert sizes[(4096, 3)] > sizes[(4096, 2)]
    assert sizes[(2048, 1)] < sizes[(4096, 2)]


def test_stage_copy_argument_errors():
    # rejected on the host, before any launch
    INVALID = -1
    L = pks.lib()
    R = pks.pks_copy_range
    arr = (R * 9)()
    for i in range(9):
        arr[i] = R(16, 32, 16)
    assert L.pks_stage_copy(None, 1, None) == INVALID
    assert L.pks_stage_copy(arr, 0, None) == INVALID
    assert L.pks_stage_copy(arr, pks.PKS_STAGE_MAX_RANGES + 1, None) == INVALID
    arr[1] = R(None, 32, 16)
    assert L.pks_stage_copy(arr, 2, None) == INVALID
    arr[1] = R(16, None, 16)
    assert L.pks_stage_copy(arr, 2, None) == INVALID
    assert pks.PKS_STAGE_MAX_RANGES == 8


def test_barrier_offset_lies_in_the_control_block():
    import ctypes
    a = _cpu_args()
    total = pks.pks_decode_workspace_size(a)
    off = pks.pks_decode_barrier_offset(a)
    assert off % 256 == 0 and 0 < off < total
    # the counters follow the per-request score histograms (2048 int32 each)
    assert off >= 2048 * 4 * a.B
    L = pks.lib()
    assert L.pks_decode_barrier_offset(ctypes.byref(a), None) == -1
    assert L.pks_decode_barrier_offset(ctypes.byref(_cpu_args(k=0)),
                                       ctypes.byref(ctypes.c_size_t())) == -1
