"""Owning wrapper around one decode-step shape: outputs, workspace, arguments."""

from __future__ import annotations

import torch

from . import pks


class SparseDecodeStep:
    """Device tensors of one batch plus the output, top-k and workspace buffers.

    ``tensors`` holds device tensors named like the C arguments: seq_lens,
    block_table, q, q_idx, w_idx, kv_k, kv_v, idx_k.  Calling the object runs
    ``pks_decode_step`` on ``stream`` (default: torch's current stream).
    """

    def __init__(self, tensors: dict, k: int, attn_splits: int = 0, topk_mode: int = 0,
                 stream=None, wait_limit: int = 0):
        t = dict(tensors)
        q = t["q"]
        dev = q.device
        self.tensors = t
        self.k = int(k)
        # q: [B, Hq, D], or [B, Nq, Hq, D] with Nq query tokens per request
        self.out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        self.topk_idx = torch.empty(tuple(q.shape[:-2]) + (self.k,), dtype=torch.int32, device=dev)
        probe = pks.make_args(k=self.k, topk_idx=self.topk_idx, out=self.out,
                              attn_splits=attn_splits, topk_mode=topk_mode,
                              wait_limit=wait_limit, **t)
        nbytes = pks.pks_decode_workspace_size(probe)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        if self.workspace.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")
        self.args = pks.make_args(k=self.k, topk_idx=self.topk_idx, out=self.out,
                                  workspace=self.workspace, attn_splits=attn_splits,
                                  topk_mode=topk_mode, wait_limit=wait_limit, **t)
        pks.pks_decode_workspace_init(self.args, stream)

    def __call__(self, stream=None):
        pks.pks_decode_step(self.args, stream)
        return self.out, self.topk_idx

    def timed(self, events, stream=None):
        pks.pks_decode_step_timed(self.args, events, stream)

    def attention_only(self, stream=None):
        pks.pks_sparse_attention(self.args, stream)

    def scores(self, stream=None) -> torch.Tensor:
        B = self.args.B * max(1, self.args.n_queries)  # one row per query token
        ld = self.args.max_pages * self.args.page_size
        out = torch.zeros((B, ld), dtype=torch.int32, device=self.out.device)
        pks.pks_indexer_scores(self.args, out, stream)
        return out

    def launches(self) -> int:
        """Kernels one step enqueues on the current device."""
        return pks.pks_decode_launches(self.args)

    def device_error(self, stream=None) -> int:
        return pks.pks_decode_device_error(self.args, stream)


class ResidentDecodeStep:
    """The decode step with the KV cache in host memory and an LRU cache of
    its pages in HBM: select (scan + top-k), residency update (miss list),
    fetch of the admitted misses into their slots, attention through the
    table.  ``host_k`` / ``host_v`` are device-accessible (pinned) host tensors
    [num_pages, P, Hkv, D]; ``tensors`` holds the other inputs on the device.
    The slots start with ``init_pages`` (copied in here, as a loader would)."""

    def __init__(self, tensors: dict, host_k: torch.Tensor, host_v: torch.Tensor, k: int,
                 capacity: int, init_pages=(), stream=None):
        t = dict(tensors)
        t["kv_k"], t["kv_v"] = host_k, host_v
        self.step = SparseDecodeStep(t, k, stream=stream)
        self.args = self.step.args
        dev = t["q"].device
        num_pages = host_k.shape[0]
        self.capacity = int(capacity)
        self.slot_k = torch.empty((max(1, capacity),) + tuple(host_k.shape[1:]),
                                  dtype=torch.bfloat16, device=dev)
        self.slot_v = torch.empty_like(self.slot_k)
        self.table = pks.ResidencyTable(num_pages, capacity, init_pages, device=dev, stream=stream)
        init = sorted(set(int(p) for p in init_pages))
        if init:
            idx = torch.tensor(init, dtype=torch.long)
            self.slot_k[: len(init)].copy_(host_k.index_select(0, idx))
            self.slot_v[: len(init)].copy_(host_v.index_select(0, idx))
        self.host_k, self.host_v = host_k, host_v
        self.block_table = t["block_table"]
        self.page_size = host_k.shape[1]
        self.miss = torch.empty(num_pages, dtype=torch.int32, device=dev)
        self.n_miss = torch.zeros(1, dtype=torch.int32, device=dev)

    # the step's four calls, in order
    def select(self, stream=None):
        pks.pks_decode_select(self.args, stream)

    def update(self, stream=None):
        self.table.update(self.step.topk_idx, self.block_table, self.page_size, self.miss,
                          self.n_miss, stream)

    def fetch(self, stream=None):
        self.table.fetch(self.miss, self.n_miss, self.host_k, self.host_v, self.slot_k,
                         self.slot_v, stream)

    def attend(self, stream=None):
        pks.pks_sparse_attention_resident(self.args, self.table.state, self.capacity, self.slot_k,
                                          self.slot_v, stream)

    def __call__(self, stream=None):
        self.select(stream)
        self.update(stream)
        self.fetch(stream)
        self.attend(stream)
        return self.step.out, self.step.topk_idx


class ResidentLayers:
    """Several layers of the decode step through HBM residency tables, the
    miss fetch overlapped layer by layer ("Sparse Attention on GLM5.3 and
    HBM", HiSparse paragraph: the KV cache lives in host memory, an LRU cache
    of it in HBM, misses of the top-k are loaded, the loads overlapped across
    layers).  Every layer has its own KV pools in pinned host memory, its own
    slot table and slot pools, and its own inputs (``tensors`` per layer).

    With ``overlap`` the fetch of layer l runs on a side stream: it waits for
    layer l's residency update (an event) and runs while the main stream
    selects layer l+1 and attends layer l-1; layer l's attention waits for its
    own fetch (a second event).  Without it the four calls of every layer run
    one after the other on the main stream.  Both orders compute the same
    values: each layer's fetch writes only that layer's slots, which only that
    layer's attention reads."""

    def __init__(self, layers: list, k: int, capacity: int, stream=None):
        # layers: dicts with "tensors" (device inputs), "host_k", "host_v"
        # (pinned [num_pages, P, Hkv, D]) and "init_pages"
        self.layers = [ResidentDecodeStep(L["tensors"], L["host_k"], L["host_v"], k, capacity,
                                          L["init_pages"], stream=stream) for L in layers]
        dev = layers[0]["tensors"]["q"].device
        self.side = torch.cuda.Stream(device=dev)
        n = len(self.layers)
        self.updated = [torch.cuda.Event() for _ in range(n)]
        self.fetched = [torch.cuda.Event() for _ in range(n)]

    def __call__(self, stream=None, overlap: bool = True):
        main = stream if stream is not None else torch.cuda.current_stream()
        if not overlap:
            for L in self.layers:
                L(main)
            return [(L.step.out, L.step.topk_idx) for L in self.layers]
        side = self.side
        n = len(self.layers)
        for l in range(n + 1):
            if l < n:
                L = self.layers[l]
                L.select(main)
                L.update(main)
                self.updated[l].record(main)
                side.wait_event(self.updated[l])
                L.fetch(side)
                self.fetched[l].record(side)
            if l > 0:  # the previous layer's attention, once its own fetch is done
                main.wait_event(self.fetched[l - 1])
                self.layers[l - 1].attend(main)
        return [(L.step.out, L.step.topk_idx) for L in self.layers]


class MlaAttention:
    """Sparse MLA in MQA mode over given selections: ``pks_mla_sparse_attention``
    with its own output and workspace.  q [B, H, d + r], kv [num_pages, P, d + r]
    (bf16), topk_idx [B, k] (int32), d = 512 latent values."""

    def __init__(self, seq_lens, block_table, topk_idx, q, kv, sm_scale: float = 0.0,
                 trim: bool = False, splits: int = 0, stream=None, wait_limit: int = 0):
        dev = q.device
        self.out = torch.empty((q.shape[0], q.shape[1], 512), dtype=torch.bfloat16, device=dev)
        probe = pks.make_mla_args(seq_lens=seq_lens, block_table=block_table, topk_idx=topk_idx,
                                  q=q, kv=kv, out=self.out, sm_scale=sm_scale, trim=trim,
                                  splits=splits)
        nbytes = pks.pks_mla_workspace_size(probe)
        self.workspace = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.args = pks.make_mla_args(seq_lens=seq_lens, block_table=block_table,
                                      topk_idx=topk_idx, q=q, kv=kv, out=self.out,
                                      workspace=self.workspace, sm_scale=sm_scale, trim=trim,
                                      splits=splits, wait_limit=wait_limit)
        self._keep = (seq_lens, block_table, topk_idx, q, kv)

    def __call__(self, stream=None):
        pks.pks_mla_sparse_attention(self.args, stream)
        return self.out

    def device_error(self, stream=None) -> int:
        return pks.pks_mla_device_error(self.args, stream)


class MlaDecodeStep:
    """The DSA decode step with MLA attention: indexer scan and top-k
    (``pks_decode_select``), then the sparse MLA over the selected tokens.
    ``tensors``: seq_lens, block_table, q_idx, w_idx, idx_k as for the GQA
    step, plus q [B, H, d + r] and kv [num_pages, P, d + r] (bf16)."""

    def __init__(self, tensors: dict, k: int, topk_mode: int = 0, splits: int = 0,
                 sm_scale: float = 0.0, stream=None):
        t = dict(tensors)
        q, kv = t["q"], t["kv"]
        dev = q.device
        B = q.shape[0]
        self.k = int(k)
        self.topk_idx = torch.empty((B, self.k), dtype=torch.int32, device=dev)
        # selection arguments: the indexer and top-k fields of pks_decode_args
        # (the GQA attention fields stay unset; select does not read them)
        a = pks.pks_decode_args()
        npages, P, _ = kv.shape
        _, Hi, Di = t["q_idx"].shape
        a.B, a.Hq, a.Hkv, a.D, a.Hi, a.Di = int(B), 1, 1, 64, int(Hi), int(Di)
        a.page_size, a.max_pages = int(P), int(t["block_table"].shape[1])
        a.num_pages, a.k = int(npages), self.k
        a.seq_lens = pks._dptr(t["seq_lens"], torch.int32, "seq_lens")
        a.block_table = pks._dptr(t["block_table"], torch.int32, "block_table")
        a.q_idx = pks._dptr(t["q_idx"], torch.int8, "q_idx")
        a.w_idx = pks._dptr(t.get("w_idx"), torch.int32, "w_idx")
        a.idx_k = pks._dptr(t["idx_k"], torch.int8, "idx_k")
        a.topk_idx = pks._dptr(self.topk_idx, torch.int32, "topk_idx")
        a.topk_mode = int(topk_mode)
        # real-valued head weights and FP8 e4m3 queries/keys (DSA's indexer)
        if t.get("w_idx_f") is not None:
            a.w_idx_f = pks._dptr(t["w_idx_f"], torch.float32, "w_idx_f")
        a.idx_fp8 = 1 if t.get("idx_fp8") else 0
        nbytes = pks.pks_decode_workspace_size(a)
        self.select_workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        a.workspace = self.select_workspace.data_ptr()
        a.workspace_bytes = self.select_workspace.numel()
        pks.pks_decode_workspace_init(a, stream)
        self.select_args = a
        self.attention = MlaAttention(t["seq_lens"], t["block_table"], self.topk_idx, q, kv,
                                      sm_scale=sm_scale, trim=True, splits=splits)
        self.out = self.attention.out
        self.tensors = t

    def select(self, stream=None):
        pks.pks_decode_select(self.select_args, stream)
        return self.topk_idx

    def __call__(self, stream=None):
        pks.pks_decode_select(self.select_args, stream)
        pks.pks_mla_sparse_attention(self.attention.args, stream)
        return self.out, self.topk_idx
