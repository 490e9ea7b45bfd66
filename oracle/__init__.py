"""CPU oracle for the sparse decode step - TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The product library never imports it.  The arithmetic lives in
``pks_oracle.c`` (plain C, int64 and double precision); this module compiles it
with the host C compiler and marshals numpy arrays to it through ctypes.

Parity status of each function (what pins it, in ``tests/test_oracle_*.py``):

* pages_for / tail_waste / build_block_table / capacity_* - pinned by the
  worked example, landmarks, quiz and capacity figures of the "Paged KV cache"
  chapter (``tests/golden/paged_kv_worked_example.txt``).
* indexer_scores - pinned by closed forms (unit query vectors, q and -q heads
  giving |q.k|), weight scaling, and invariance under page permutation.
* topk - pinned by a brute-force library sort on small inputs and the dense
  and all-ties special cases.
* sparse_attention - pinned by a library dense attention (k >= len), the
  single-token and zero-query closed forms, and paging invariance.
* residency_* - pinned by a textbook LRU cache (one page per step), the
  sequential-scan cliff, and set invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pks_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"
_lib = None


def build(force: bool = False) -> Path:
    """Compile ``pks_oracle.c`` into ``oracle/_build/liboracle.so``."""
    _BUILD.mkdir(exist_ok=True)
    if (not force and _LIB_PATH.exists()
            and _LIB_PATH.stat().st_mtime >= max(_SRC.stat().st_mtime,
                                                  (_HERE / "pks_oracle.h").stat().st_mtime)):
        return _LIB_PATH
    tmp = _LIB_PATH.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra",
           "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(str(build()))
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


def _declare(L):
    L.orc_pages_for.argtypes = [_I64, _I64]
    L.orc_pages_for.restype = _I64
    L.orc_tail_waste.argtypes = [_I64, _I64]
    L.orc_tail_waste.restype = _I64
    L.orc_build_block_table.argtypes = [_I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P]
    L.orc_build_block_table.restype = ctypes.c_int
    L.orc_capacity_paged.argtypes = [_I32, _P, _I32, _I64]
    L.orc_capacity_paged.restype = _I64
    L.orc_capacity_naive.argtypes = [_I32, _P, _I32, _I64]
    L.orc_capacity_naive.restype = _I64
    L.orc_indexer_scores.argtypes = [_I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64]
    L.orc_indexer_scores.restype = ctypes.c_int
    L.orc_topk.argtypes = [_I32, _P, _P, _I64, _I32, _P]
    L.orc_topk.restype = ctypes.c_int
    L.orc_sparse_attention.argtypes = [_I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P,
                                       _P, _P, _P]
    L.orc_sparse_attention.restype = ctypes.c_int
    L.orc_indexer_scores_f.argtypes = [_I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P,
                                       _I64]
    L.orc_indexer_scores_f.restype = ctypes.c_int
    L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_value.restype = ctypes.c_double
    L.orc_indexer_scores_fp8.argtypes = [_I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P,
                                         _I64]
    L.orc_indexer_scores_fp8.restype = ctypes.c_int
    L.orc_topk_f.argtypes = [_I32, _P, _P, _I64, _I32, _P]
    L.orc_topk_f.restype = ctypes.c_int
    L.orc_mla_sparse_attention.argtypes = [_I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P,
                                           _P, _P, ctypes.c_double, _P]
    L.orc_mla_sparse_attention.restype = ctypes.c_int
    L.orc_residency_init.argtypes = [_I32, _I32, _I32, _P, _P, _P, _P, _P]
    L.orc_residency_init.restype = ctypes.c_int
    L.orc_residency_step.argtypes = [_I32, _I32, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P,
                                     _P, _P, _P, _P]
    L.orc_residency_step.restype = ctypes.c_int
    L.orc_set_threads.argtypes = [ctypes.c_int]
    L.orc_set_threads.restype = ctypes.c_int


def _arr(x, dtype):
    """Contiguous numpy array of ``dtype`` (accepts numpy arrays, lists, CPU torch tensors)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            x = t.view(torch.int16).numpy().view(np.uint16)
        else:
            x = t.numpy()
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != dtype:
        if dtype == np.uint16 and a.dtype != np.uint16:
            raise TypeError("bf16 inputs must be given as bf16 tensors or uint16 bit patterns")
        a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def set_threads(n: int = 0) -> int:
    return lib().orc_set_threads(int(n))


def pages_for(length: int, page_size: int) -> int:
    return lib().orc_pages_for(int(length), int(page_size))


def tail_waste(length: int, page_size: int) -> int:
    return lib().orc_tail_waste(int(length), int(page_size))


def build_block_table(seq_lens, page_size, max_pages, num_pages, prefix_group=None,
                      prefix_len=0, free_order=None):
    """Returns ``(block_table int32 [B, max_pages], pages_used)``; raises on failure."""
    lens = _arr(seq_lens, np.int32)
    B = lens.shape[0]
    grp = _arr(prefix_group, np.int32)
    fo = _arr(free_order, np.int32)
    bt = np.empty((B, max_pages), dtype=np.int32)
    used = np.zeros(1, dtype=np.int32)
    rc = lib().orc_build_block_table(B, _ptr(lens), _ptr(grp), int(prefix_len), int(page_size),
                                     int(max_pages), int(num_pages), _ptr(fo), _ptr(bt),
                                     _ptr(used))
    if rc != 0:
        raise OracleError(f"build_block_table failed with code {rc}")
    return bt, int(used[0])


def capacity_paged(lens, page_size, slots) -> int:
    a = _arr(lens, np.int32)
    return lib().orc_capacity_paged(a.shape[0], _ptr(a), int(page_size), int(slots))


def capacity_naive(lens, reserve, slots) -> int:
    a = _arr(lens, np.int32)
    return lib().orc_capacity_naive(a.shape[0], _ptr(a), int(reserve), int(slots))


def indexer_scores(seq_lens, block_table, page_size, q_idx, w_idx, idx_k, ld=None):
    """int64 scores [B, ld] (entries at t >= len_b are 0)."""
    lens = _arr(seq_lens, np.int32)
    bt = _arr(block_table, np.int32)
    qi = _arr(q_idx, np.int8)
    w = _arr(w_idx, np.int32)
    ik = _arr(idx_k, np.int8)
    B, Hi, Di = qi.shape
    assert ik.shape[-1] == Di
    max_pages = bt.shape[1]
    if ld is None:
        ld = max_pages * page_size
    out = np.zeros((B, ld), dtype=np.int64)
    _check(lib().orc_indexer_scores(B, _ptr(lens), _ptr(bt), max_pages, int(page_size), Hi, Di,
                                    _ptr(qi), _ptr(w), _ptr(ik), _ptr(out), int(ld)),
           "indexer_scores")
    return out


def indexer_scores_f(seq_lens, block_table, page_size, q_idx, w_f, idx_k, ld=None):
    """Float-weighted indexer scores: float32 [B, ld] (fp32, heads in order)."""
    lens = _arr(seq_lens, np.int32)
    bt = _arr(block_table, np.int32)
    qi = _arr(q_idx, np.int8)
    wf = _arr(w_f, np.float32)
    ik = _arr(idx_k, np.int8)
    B, Hi, Di = qi.shape
    assert wf.shape == (B, Hi)
    if ld is None:
        ld = int(bt.shape[1]) * int(page_size)
    out = np.zeros((B, ld), dtype=np.float32)
    _check(lib().orc_indexer_scores_f(B, _ptr(lens), _ptr(bt), bt.shape[1], int(page_size), Hi,
                                      Di, _ptr(qi), _ptr(wf), _ptr(ik), _ptr(out), int(ld)),
           "indexer_scores_f")
    return out


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code) & 0xFF)


def _bytes(x):
    """uint8 view of int8 / uint8 / float8 tensors or arrays."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        return t.numpy()
    a = np.ascontiguousarray(np.asarray(x))
    return a.view(np.uint8) if a.dtype != np.uint8 else a


def indexer_scores_fp8(seq_lens, block_table, page_size, q_idx, w_f, idx_k, ld=None):
    """Exact FP8 e4m3 indexer scores (float64 [B, ld])."""
    lens = _arr(seq_lens, np.int32)
    bt = _arr(block_table, np.int32)
    qi = _bytes(q_idx)
    ik = _bytes(idx_k)
    wf = _arr(w_f, np.float32)
    B, Hi, Di = qi.shape
    if ld is None:
        ld = int(bt.shape[1]) * int(page_size)
    out = np.zeros((B, ld), dtype=np.float64)
    _check(lib().orc_indexer_scores_fp8(B, _ptr(lens), _ptr(bt), bt.shape[1], int(page_size), Hi,
                                        Di, _ptr(qi), _ptr(wf), _ptr(ik), _ptr(out), int(ld)),
           "indexer_scores_fp8")
    return out


def topk_f(seq_lens, scores, k):
    lens = _arr(seq_lens, np.int32)
    sc = _arr(scores, np.float32)
    B = lens.shape[0]
    out = np.empty((B, k), dtype=np.int32)
    _check(lib().orc_topk_f(B, _ptr(lens), _ptr(sc), sc.shape[1], int(k), _ptr(out)), "topk_f")
    return out


def topk(seq_lens, scores, k):
    lens = _arr(seq_lens, np.int32)
    sc = _arr(scores, np.int64)
    B = lens.shape[0]
    out = np.empty((B, k), dtype=np.int32)
    _check(lib().orc_topk(B, _ptr(lens), _ptr(sc), sc.shape[1], int(k), _ptr(out)), "topk")
    return out


def sparse_attention(block_table, page_size, idx, q, kv_k, kv_v):
    """double [B, Hq, D]."""
    bt = _arr(block_table, np.int32)
    ix = _arr(idx, np.int32)
    qa = _arr(q, np.uint16)
    ka = _arr(kv_k, np.uint16)
    va = _arr(kv_v, np.uint16)
    B, Hq, D = qa.shape
    Hkv = ka.shape[2]
    assert ka.shape[3] == D and va.shape == ka.shape
    out = np.empty((B, Hq, D), dtype=np.float64)
    _check(lib().orc_sparse_attention(B, _ptr(bt), bt.shape[1], int(page_size), Hq, Hkv, D,
                                      ix.shape[1], _ptr(ix), _ptr(qa), _ptr(ka), _ptr(va),
                                      _ptr(out)), "sparse_attention")
    return out


def mla_sparse_attention(block_table, page_size, idx, q, kv, d, scale=None):
    """Sparse MLA in MQA mode: q [B, H, d + r], kv pool [num_pages, page_size, d + r]
    (bf16); scale defaults to 1 / sqrt(d + r).  double [B, H, d]."""
    bt = _arr(block_table, np.int32)
    ix = _arr(idx, np.int32)
    qa = _arr(q, np.uint16)
    ka = _arr(kv, np.uint16)
    B, H, dk = qa.shape
    assert ka.shape[-1] == dk and 0 < d <= dk
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    out = np.empty((B, H, d), dtype=np.float64)
    _check(lib().orc_mla_sparse_attention(B, _ptr(bt), bt.shape[1], int(page_size), H, int(d),
                                          dk - int(d), ix.shape[1], _ptr(ix), _ptr(qa),
                                          _ptr(ka), float(scale), _ptr(out)),
           "mla_sparse_attention")
    return out


def decode_step(seq_lens, block_table, page_size, k, q, q_idx, w_idx, kv_k, kv_v, idx_k):
    """The whole step: (scores int64, top-k int32 [B, k], out double [B, Hq, D])."""
    scores = indexer_scores(seq_lens, block_table, page_size, q_idx, w_idx, idx_k)
    idx = topk(seq_lens, scores, k)
    out = sparse_attention(block_table, page_size, idx, q, kv_k, kv_v)
    return scores, idx, out


class Residency:
    """Host-side residency table (HiSparse-style LRU over KV pages)."""

    def __init__(self, num_pages: int, capacity: int, initial_pages=()):
        self.num_pages = int(num_pages)
        self.capacity = int(capacity)
        self.page_slot = np.empty(self.num_pages, dtype=np.int32)
        self.slot_page = np.empty(self.capacity, dtype=np.int32)
        self.last_use = np.empty(self.capacity, dtype=np.int32)
        self.step_no = np.zeros(1, dtype=np.int32)
        init = _arr(np.asarray(initial_pages, dtype=np.int32), np.int32)
        _check(lib().orc_residency_init(self.num_pages, self.capacity, init.shape[0], _ptr(init),
                                        _ptr(self.page_slot), _ptr(self.slot_page),
                                        _ptr(self.last_use), _ptr(self.step_no)),
               "residency_init")

    def step(self, idx, block_table, page_size):
        """Returns ``(miss_list int32 [n_miss], n_hit)``."""
        ix = _arr(idx, np.int32)
        bt = _arr(block_table, np.int32)
        B, k = ix.shape
        miss = np.empty(max(self.num_pages, 1), dtype=np.int32)
        n_miss = np.zeros(1, dtype=np.int32)
        n_hit = np.zeros(1, dtype=np.int32)
        _check(lib().orc_residency_step(self.num_pages, self.capacity, _ptr(self.page_slot),
                                        _ptr(self.slot_page), _ptr(self.last_use),
                                        _ptr(self.step_no), B, k, int(page_size), bt.shape[1],
                                        _ptr(ix), _ptr(bt), _ptr(miss), _ptr(n_miss),
                                        _ptr(n_hit)), "residency_step")
        return miss[: int(n_miss[0])].copy(), int(n_hit[0])

    def resident_pages(self):
        return np.sort(self.slot_page[self.slot_page >= 0])
