"""Python binding of libpks (ctypes): argument marshalling only.

Every function here forwards to the C entry point of the same name in
``include/pks.h``; all computation runs in the library's CUDA kernels (device
functions) or its host code (page allocator, block tables).  torch provides
device memory and streams.  There is no fallback: if ``libpks.so`` is missing
the first call raises.
"""

from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional, Sequence

import numpy as np
import torch

_LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libpks.so"
_lib = None

PKS_OK = 0
STATUS_NAMES = {
    0: "PKS_OK", -1: "PKS_ERR_INVALID", -2: "PKS_ERR_OOM", -3: "PKS_ERR_CUDA",
    -4: "PKS_ERR_TIMEOUT", -5: "PKS_ERR_DEVICE_CHECK", -6: "PKS_ERR_UNSUPPORTED",
    -7: "PKS_ERR_WORKSPACE",
    -8: "PKS_ERR_TOO_LARGE",
}


class PksError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        name = STATUS_NAMES.get(self.code, str(self.code))
        msg = lib().pks_status_str(self.code).decode()
        super().__init__(f"{where}: {name} ({msg})")


class pks_decode_args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("D", ctypes.c_int32), ("Hi", ctypes.c_int32), ("Di", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("k", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w_idx", ctypes.c_void_p),
        ("kv_k", ctypes.c_void_p), ("kv_v", ctypes.c_void_p), ("idx_k", ctypes.c_void_p),
        ("topk_idx", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("attn_splits", ctypes.c_int32), ("topk_mode", ctypes.c_int32),
        ("n_queries", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1),
        ("w_idx_f", ctypes.c_void_p), ("idx_fp8", ctypes.c_int32), ("wait_limit", ctypes.c_int32),
    ]


class pks_mla_args(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("d_latent", ctypes.c_int32),
        ("d_rope", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("k", ctypes.c_int32),
        ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("topk_idx", ctypes.c_void_p), ("q", ctypes.c_void_p), ("kv", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t), ("sm_scale", ctypes.c_float),
        ("trim", ctypes.c_int32), ("splits", ctypes.c_int32), ("wait_limit", ctypes.c_int32),
    ]


def library_path() -> Path:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded libpks.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "top_sparse_attention_pks_gb300.build.build_library()")
        L = ctypes.CDLL(str(_LIB_PATH))
        _declare(L)
        _lib = L
    return _lib


class pks_copy_range(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


PKS_STAGE_MAX_RANGES = 8

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_ST = ctypes.c_int32
_PARGS = ctypes.POINTER(pks_decode_args)


def _declare(L):
    L.pks_status_str.argtypes = [_I32]
    L.pks_status_str.restype = ctypes.c_char_p
    L.pks_pool_create.argtypes = [_I32, _I32, _P, ctypes.POINTER(_P)]
    L.pks_pool_create.restype = _ST
    L.pks_pool_destroy.argtypes = [_P]
    L.pks_pool_destroy.restype = None
    L.pks_pool_free_count.argtypes = [_P, _P]
    L.pks_pool_free_count.restype = _ST
    L.pks_alloc_pages.argtypes = [_P, _I32, _P]
    L.pks_alloc_pages.restype = _ST
    L.pks_free_pages.argtypes = [_P, _I32, _P]
    L.pks_free_pages.restype = _ST
    L.pks_admission_simulate.argtypes = [_P, _I32, _P, _I32, _P, _P, _P]
    L.pks_admission_simulate.restype = _ST
    L.pks_build_block_table.argtypes = [_P, _I32, _P, _P, _I32, _I32, _P, _P]
    L.pks_build_block_table.restype = _ST
    L.pks_decode_workspace_size.argtypes = [_PARGS, ctypes.POINTER(ctypes.c_size_t)]
    L.pks_decode_workspace_size.restype = _ST
    L.pks_decode_workspace_init.argtypes = [_PARGS, _P]
    L.pks_decode_workspace_init.restype = _ST
    L.pks_decode_step.argtypes = [_PARGS, _P]
    L.pks_decode_step.restype = _ST
    L.pks_sparse_attention_static.argtypes = [_PARGS, _P]
    L.pks_sparse_attention_static.restype = _ST
    L.pks_decode_select.argtypes = [_PARGS, _P]
    L.pks_decode_select.restype = _ST
    L.pks_sparse_attention_resident.argtypes = [_PARGS, _P, _I32, _P, _P, _P]
    L.pks_sparse_attention_resident.restype = _ST
    L.pks_residency_fetch.argtypes = [_P, _I32, _I32, _P, _P, _P, _P, _P, _P, ctypes.c_int64, _P]
    L.pks_residency_fetch.restype = _ST
    L.pks_decode_launches.argtypes = [_PARGS, _P]
    L.pks_decode_launches.restype = _ST
    L.pks_decode_step_timed.argtypes = [_PARGS, _P, _P]
    L.pks_decode_step_timed.restype = _ST
    L.pks_indexer_scores.argtypes = [_PARGS, _P, ctypes.c_int64, _P]
    L.pks_indexer_scores.restype = _ST
    L.pks_sparse_attention.argtypes = [_PARGS, _P]
    L.pks_sparse_attention.restype = _ST
    L.pks_decode_barrier_offset.argtypes = [_PARGS, ctypes.POINTER(ctypes.c_size_t)]
    L.pks_decode_barrier_offset.restype = _ST
    L.pks_decode_device_error.argtypes = [_PARGS, _P, _P]
    L.pks_decode_device_error.restype = _ST
    L.pks_residency_state_bytes.argtypes = [_I32, _I32, ctypes.POINTER(ctypes.c_size_t)]
    L.pks_residency_state_bytes.restype = _ST
    L.pks_residency_offsets.argtypes = [_I32, _I32] + [ctypes.POINTER(ctypes.c_size_t)] * 4
    L.pks_residency_offsets.restype = _ST
    L.pks_residency_init.argtypes = [_P, _I32, _I32, _I32, _P, _P]
    L.pks_residency_init.restype = _ST
    L.pks_residency_update.argtypes = [_P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P,
                                       _P]
    L.pks_residency_update.restype = _ST
    L.pks_stage_copy.argtypes = [ctypes.POINTER(pks_copy_range), _I32, _P]
    L.pks_stage_copy.restype = _ST

    _PM = ctypes.POINTER(pks_mla_args)
    L.pks_mla_workspace_size.argtypes = [_PM, ctypes.POINTER(ctypes.c_size_t)]
    L.pks_mla_workspace_size.restype = _ST
    L.pks_mla_sparse_attention.argtypes = [_PM, _P]
    L.pks_mla_sparse_attention.restype = _ST
    L.pks_mla_device_error.argtypes = [_PM, ctypes.POINTER(ctypes.c_int32), _P]
    L.pks_mla_device_error.restype = _ST


def _check(code: int, where: str):
    if code != PKS_OK:
        raise PksError(code, where)


def _stream(stream) -> Optional[int]:
    if stream is None:
        if torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dptr(t: Optional[torch.Tensor], dtype, name: str) -> Optional[int]:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host_i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


# ----------------------------------------------------------- page pool ---

def pks_pool_create(num_pages: int, page_size: int, free_order=None) -> int:
    fo = None if free_order is None else _host_i32(free_order)
    h = ctypes.c_void_p()
    _check(lib().pks_pool_create(int(num_pages), int(page_size),
                                 None if fo is None else fo.ctypes.data, ctypes.byref(h)),
           "pks_pool_create")
    return h.value


def pks_pool_destroy(pool: int) -> None:
    lib().pks_pool_destroy(pool)


def pks_pool_free_count(pool: int) -> int:
    out = ctypes.c_int32()
    _check(lib().pks_pool_free_count(pool, ctypes.addressof(out)), "pks_pool_free_count")
    return out.value


def pks_alloc_pages(pool: int, n: int) -> np.ndarray:
    out = np.empty(max(int(n), 1), dtype=np.int32)
    _check(lib().pks_alloc_pages(pool, int(n), out.ctypes.data), "pks_alloc_pages")
    return out[: int(n)]


def pks_free_pages(pool: int, ids) -> None:
    a = _host_i32(ids)
    _check(lib().pks_free_pages(pool, a.shape[0], a.ctypes.data), "pks_free_pages")


def pks_build_block_table(pool: int, seq_lens, max_pages: int, prefix_group=None,
                          prefix_len: int = 0):
    """Returns ``(block_table int32 [B, max_pages] host array, pages_used)``."""
    lens = _host_i32(seq_lens)
    grp = None if prefix_group is None else _host_i32(prefix_group)
    B = lens.shape[0]
    bt = np.empty((B, int(max_pages)), dtype=np.int32)
    used = ctypes.c_int32()
    _check(lib().pks_build_block_table(pool, B, lens.ctypes.data,
                                       None if grp is None else grp.ctypes.data,
                                       int(prefix_len), int(max_pages), bt.ctypes.data,
                                       ctypes.addressof(used)), "pks_build_block_table")
    return bt, used.value


def pks_admission_simulate(pool: int, lens, reserve: int = 0):
    """``(admitted, tokens, slots)`` of cyclic admission on the pool's free pages
    (reserve 0: paging; reserve > 0: every request reserves that many tokens)."""
    a = _host_i32(lens)
    adm, tok, slots = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().pks_admission_simulate(pool, a.shape[0], a.ctypes.data, int(reserve),
                                        ctypes.addressof(adm), ctypes.addressof(tok),
                                        ctypes.addressof(slots)), "pks_admission_simulate")
    return adm.value, tok.value, slots.value


class Pool:
    """Owning wrapper of a host page pool handle."""

    def __init__(self, num_pages: int, page_size: int, free_order=None):
        self.handle = pks_pool_create(num_pages, page_size, free_order)

    def alloc(self, n: int) -> np.ndarray:
        return pks_alloc_pages(self.handle, n)

    def free(self, ids) -> None:
        pks_free_pages(self.handle, ids)

    def free_count(self) -> int:
        return pks_pool_free_count(self.handle)

    def build_block_table(self, seq_lens, max_pages, prefix_group=None, prefix_len=0):
        return pks_build_block_table(self.handle, seq_lens, max_pages, prefix_group, prefix_len)

    def admission(self, lens, reserve: int = 0):
        return pks_admission_simulate(self.handle, lens, reserve)

    def close(self):
        if self.handle:
            pks_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------- decode step ---

def make_args(*, seq_lens, block_table, q, q_idx, w_idx, kv_k, kv_v, idx_k, k: int,
              topk_idx=None, out=None, workspace=None, attn_splits: int = 0,
              topk_mode: int = 0, num_pages: Optional[int] = None,
              w_idx_f=None, idx_fp8: bool = False, wait_limit: int = 0) -> pks_decode_args:
    """Fill a ``pks_decode_args`` from tensors (shapes are read off the tensors).

    ``q`` is [B, Hq, D], or [B, Nq, Hq, D] for Nq query tokens per request (then
    ``q_idx`` is [B, Nq, Hi, Di], ``topk_idx`` [B, Nq, k], ``out`` [B, Nq, Hq, D])."""
    a = pks_decode_args()
    if q.dim() == 4:
        B, Nq, Hq, D = q.shape
        if q_idx.dim() != 4 or q_idx.shape[:2] != q.shape[:2]:
            raise ValueError("q_idx must be [B, Nq, Hi, Di] like q")
        _, _, Hi, Di = q_idx.shape
        a.n_queries = int(Nq)
    else:
        B, Hq, D = q.shape
        _, Hi, Di = q_idx.shape
    npages, P, Hkv, D2 = kv_k.shape
    if D2 != D or tuple(kv_v.shape) != tuple(kv_k.shape):
        raise ValueError("kv_k / kv_v / q shapes disagree")
    if tuple(idx_k.shape) != (npages, P, Di):
        raise ValueError("idx_k must be [num_pages, page_size, Di]")
    a.B, a.Hq, a.Hkv, a.D, a.Hi, a.Di = int(B), int(Hq), int(Hkv), int(D), int(Hi), int(Di)
    a.page_size = int(P)
    a.max_pages = int(block_table.shape[1])
    a.num_pages = int(npages if num_pages is None else num_pages)
    a.k = int(k)
    a.seq_lens = _dptr(seq_lens, torch.int32, "seq_lens")
    a.block_table = _dptr(block_table, torch.int32, "block_table")
    a.q = _dptr(q, torch.bfloat16, "q")
    if q_idx.dtype != torch.int8:  # FP8 e4m3 tensors: their bit patterns
        q_idx = q_idx.view(torch.int8)
    if idx_k.dtype != torch.int8:
        idx_k = idx_k.view(torch.int8)
    a.q_idx = _dptr(q_idx, torch.int8, "q_idx")
    a.w_idx = _dptr(w_idx, torch.int32, "w_idx")
    a.kv_k = _dptr(kv_k, torch.bfloat16, "kv_k")
    a.kv_v = _dptr(kv_v, torch.bfloat16, "kv_v")
    a.idx_k = _dptr(idx_k, torch.int8, "idx_k")
    a.topk_idx = _dptr(topk_idx, torch.int32, "topk_idx")
    a.out = _dptr(out, torch.bfloat16, "out")
    if workspace is not None:
        a.workspace = _dptr(workspace, torch.uint8, "workspace")
        a.workspace_bytes = workspace.numel()
    a.attn_splits = int(attn_splits)
    a.topk_mode = int(topk_mode)
    a.w_idx_f = _dptr(w_idx_f, torch.float32, "w_idx_f")
    a.idx_fp8 = 1 if idx_fp8 else 0
    a.wait_limit = int(wait_limit)
    return a


def float_key_to_score(keys: np.ndarray) -> np.ndarray:
    """The fp32 scores behind the int32 keys the scan writes with real weights."""
    k = np.asarray(keys, dtype=np.int32)
    bits = np.where(k >= 0, k, k ^ np.int32(0x7fffffff))
    return bits.astype(np.int32).view(np.float32)


def pks_decode_workspace_size(args: pks_decode_args) -> int:
    n = ctypes.c_size_t()
    _check(lib().pks_decode_workspace_size(ctypes.byref(args), ctypes.byref(n)),
           "pks_decode_workspace_size")
    return n.value


def pks_decode_workspace_init(args: pks_decode_args, stream=None) -> None:
    _check(lib().pks_decode_workspace_init(ctypes.byref(args), _stream(stream)),
           "pks_decode_workspace_init")


def pks_decode_launches(args: pks_decode_args) -> int:
    """Kernels one pks_decode_step with these shapes enqueues on the current device."""
    n = ctypes.c_int32()
    _check(lib().pks_decode_launches(ctypes.byref(args), ctypes.byref(n)), "pks_decode_launches")
    return n.value


def pks_decode_select(args: pks_decode_args, stream=None) -> None:
    """Scan and top-k only (writes args.topk_idx)."""
    _check(lib().pks_decode_select(ctypes.byref(args), _stream(stream)), "pks_decode_select")


def pks_sparse_attention_resident(args: pks_decode_args, state: torch.Tensor, capacity: int,
                                  slot_k: torch.Tensor, slot_v: torch.Tensor,
                                  stream=None) -> None:
    """Attention with K/V through the residency table (args' K/V = host pools)."""
    _check(lib().pks_sparse_attention_resident(
        ctypes.byref(args), _dptr(state, torch.uint8, "state"), int(capacity),
        _dptr(slot_k, torch.bfloat16, "slot_k"), _dptr(slot_v, torch.bfloat16, "slot_v"),
        _stream(stream)), "pks_sparse_attention_resident")


def pks_residency_fetch(state: torch.Tensor, num_pages: int, capacity: int,
                        miss_list: torch.Tensor, n_miss: torch.Tensor, host_k: torch.Tensor,
                        host_v: torch.Tensor, slot_k: torch.Tensor, slot_v: torch.Tensor,
                        page_bytes: int, stream=None) -> None:
    """Copy the admitted misses of the last residency step into their slots."""
    _check(lib().pks_residency_fetch(
        _dptr(state, torch.uint8, "state"), int(num_pages), int(capacity),
        _dptr(miss_list, torch.int32, "miss_list"), _dptr(n_miss, torch.int32, "n_miss"),
        _dptr(host_k, torch.bfloat16, "host_k"), _dptr(host_v, torch.bfloat16, "host_v"),
        _dptr(slot_k, torch.bfloat16, "slot_k"), _dptr(slot_v, torch.bfloat16, "slot_v"),
        int(page_bytes), _stream(stream)), "pks_residency_fetch")


def pks_stage_copy(pairs: Sequence, stream=None) -> None:
    """One launch copying each (dst, src) pair of equally sized tensors (device
    or page-locked host memory), in order of the pairs; at most
    PKS_STAGE_MAX_RANGES pairs."""
    n = len(pairs)
    arr = (pks_copy_range * max(1, n))()
    for i, (dst, src) in enumerate(pairs):
        nb = dst.numel() * dst.element_size()
        if src.numel() * src.element_size() != nb:
            raise ValueError(f"pks_stage_copy: pair {i} sizes differ")
        if nb == 0:  # nothing to move (empty tensors are never page-locked)
            arr[i] = pks_copy_range(None, None, 0)
            continue
        if not (dst.is_contiguous() and src.is_contiguous()):
            raise ValueError(f"pks_stage_copy: pair {i} not contiguous")
        if (dst.device.type == "cpu" and not dst.is_pinned()) or \
                (src.device.type == "cpu" and not src.is_pinned()):
            raise ValueError(f"pks_stage_copy: pair {i} host tensor not page-locked")
        arr[i] = pks_copy_range(dst.data_ptr(), src.data_ptr(), nb)
    _check(lib().pks_stage_copy(arr, n, _stream(stream)), "pks_stage_copy")


def pks_decode_step(args: pks_decode_args, stream=None) -> None:
    _check(lib().pks_decode_step(ctypes.byref(args), _stream(stream)), "pks_decode_step")


def pks_decode_step_timed(args: pks_decode_args, events: Sequence, stream=None) -> None:
    """``events``: four torch.cuda.Event (or None) recorded at the stage boundaries."""
    arr = (ctypes.c_void_p * 4)()
    for i, e in enumerate(events):
        arr[i] = None if e is None else e.cuda_event
    _check(lib().pks_decode_step_timed(ctypes.byref(args), _stream(stream), arr),
           "pks_decode_step_timed")


def pks_indexer_scores(args: pks_decode_args, scores: torch.Tensor, stream=None) -> None:
    ld = scores.shape[1]
    _check(lib().pks_indexer_scores(ctypes.byref(args), _dptr(scores, torch.int32, "scores"),
                                    int(ld), _stream(stream)), "pks_indexer_scores")


def pks_sparse_attention(args: pks_decode_args, stream=None) -> None:
    _check(lib().pks_sparse_attention(ctypes.byref(args), _stream(stream)),
           "pks_sparse_attention")


def pks_sparse_attention_static(args: pks_decode_args, stream=None) -> None:
    """Attention over args.topk_idx with the library's fixed device scratch (no workspace)."""
    _check(lib().pks_sparse_attention_static(ctypes.byref(args), _stream(stream)),
           "pks_sparse_attention_static")


def pks_decode_barrier_offset(args: pks_decode_args) -> int:
    """Byte offset of the top-k request barriers' arrival counters in the workspace."""
    n = ctypes.c_size_t()
    _check(lib().pks_decode_barrier_offset(ctypes.byref(args), ctypes.byref(n)),
           "pks_decode_barrier_offset")
    return n.value


def pks_decode_device_error(args: pks_decode_args, stream=None) -> int:
    code = ctypes.c_int32()
    _check(lib().pks_decode_device_error(ctypes.byref(args), ctypes.addressof(code),
                                         _stream(stream)), "pks_decode_device_error")
    return code.value


# ------------------------------------------------------------ residency ---

def pks_residency_state_bytes(num_pages: int, capacity: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().pks_residency_state_bytes(int(num_pages), int(capacity), ctypes.byref(n)),
           "pks_residency_state_bytes")
    return n.value


def pks_residency_offsets(num_pages: int, capacity: int) -> dict:
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().pks_residency_offsets(int(num_pages), int(capacity), *map(ctypes.byref, v)),
           "pks_residency_offsets")
    return dict(zip(("page_slot", "slot_page", "last_use", "lru_order"), (x.value for x in v)))


def pks_residency_init(state: torch.Tensor, num_pages: int, capacity: int, init_pages=(),
                       stream=None) -> None:
    pages = _host_i32(init_pages).reshape(-1)
    _check(lib().pks_residency_init(_dptr(state, torch.uint8, "state"), int(num_pages),
                                    int(capacity), pages.shape[0],
                                    pages.ctypes.data if pages.size else None, _stream(stream)),
           "pks_residency_init")


def pks_residency_update(state: torch.Tensor, num_pages: int, capacity: int, page_size: int,
                         topk_idx: torch.Tensor, block_table: torch.Tensor,
                         miss_list: torch.Tensor, n_miss: torch.Tensor, stream=None) -> None:
    B, k = topk_idx.shape
    _check(lib().pks_residency_update(
        _dptr(state, torch.uint8, "state"), int(num_pages), int(capacity), int(B), int(k),
        int(page_size), int(block_table.shape[1]), _dptr(topk_idx, torch.int32, "topk_idx"),
        _dptr(block_table, torch.int32, "block_table"),
        _dptr(miss_list, torch.int32, "miss_list"), _dptr(n_miss, torch.int32, "n_miss"),
        _stream(stream)), "pks_residency_update")


class ResidencyTable:
    """A residency state buffer in device memory (torch-allocated)."""

    def __init__(self, num_pages: int, capacity: int, init_pages=(), device="cuda", stream=None):
        self.num_pages, self.capacity = int(num_pages), int(capacity)
        nbytes = pks_residency_state_bytes(num_pages, capacity)
        self.state = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.offsets = pks_residency_offsets(num_pages, capacity)
        pks_residency_init(self.state, num_pages, capacity, init_pages, stream)

    def update(self, topk_idx, block_table, page_size, miss_list, n_miss, stream=None):
        pks_residency_update(self.state, self.num_pages, self.capacity, page_size, topk_idx,
                             block_table, miss_list, n_miss, stream)

    def fetch(self, miss_list, n_miss, host_k, host_v, slot_k, slot_v, stream=None):
        """Copy the admitted misses of the last update from the host pools into their slots."""
        page_bytes = host_k[0].numel() * host_k.element_size()
        pks_residency_fetch(self.state, self.num_pages, self.capacity, miss_list, n_miss, host_k,
                            host_v, slot_k, slot_v, page_bytes, stream)

    def _i32(self, name, n):
        off = self.offsets[name]
        return self.state[off: off + 4 * n].view(torch.int32)

    def page_slot(self):
        return self._i32("page_slot", self.num_pages)

    def slot_page(self):
        return self._i32("slot_page", self.capacity)

    def last_use(self):
        return self._i32("last_use", self.capacity)

    def lru_order(self):
        return self._i32("lru_order", self.capacity)

    def step_count(self) -> int:
        return int(self.state[:16].view(torch.int32)[2].item())


# ---------------------------------------------------------------- sparse MLA


def make_mla_args(*, seq_lens, block_table, topk_idx, q, kv, out=None, workspace=None,
                  sm_scale: float = 0.0, trim: bool = False, splits: int = 0,
                  d_latent: int = 512, num_pages: Optional[int] = None,
                  wait_limit: int = 0) -> pks_mla_args:
    """Fill a ``pks_mla_args``: q [B, H, d + r], kv [num_pages, page_size, d + r],
    topk_idx [B, k], out [B, H, d] (bf16 / int32 tensors on the device)."""
    a = pks_mla_args()
    B, H, dk = q.shape
    npages, P, dk2 = kv.shape
    if dk2 != dk or dk <= d_latent:
        raise ValueError("q and kv must both be [..., d + r] with r > 0")
    a.B, a.H, a.d_latent, a.d_rope = int(B), int(H), int(d_latent), int(dk - d_latent)
    a.page_size, a.max_pages = int(P), int(block_table.shape[1])
    a.num_pages = int(npages if num_pages is None else num_pages)
    a.k = int(topk_idx.shape[-1])
    a.seq_lens = _dptr(seq_lens, torch.int32, "seq_lens")
    a.block_table = _dptr(block_table, torch.int32, "block_table")
    a.topk_idx = _dptr(topk_idx, torch.int32, "topk_idx")
    a.q = _dptr(q, torch.bfloat16, "q")
    a.kv = _dptr(kv, torch.bfloat16, "kv")
    a.out = _dptr(out, torch.bfloat16, "out")
    if workspace is not None:
        a.workspace = _dptr(workspace, torch.uint8, "workspace")
        a.workspace_bytes = workspace.numel()
    a.sm_scale = float(sm_scale)
    a.trim = 1 if trim else 0
    a.splits = int(splits)
    a.wait_limit = int(wait_limit)
    return a


def pks_mla_workspace_size(args: pks_mla_args) -> int:
    n = ctypes.c_size_t()
    _check(lib().pks_mla_workspace_size(ctypes.byref(args), ctypes.byref(n)),
           "pks_mla_workspace_size")
    return n.value


def pks_mla_sparse_attention(args: pks_mla_args, stream=None) -> None:
    _check(lib().pks_mla_sparse_attention(ctypes.byref(args), _stream(stream)),
           "pks_mla_sparse_attention")


def pks_mla_device_error(args: pks_mla_args, stream=None) -> int:
    code = ctypes.c_int32()
    _check(lib().pks_mla_device_error(ctypes.byref(args), ctypes.byref(code), _stream(stream)),
           "pks_mla_device_error")
    return code.value
