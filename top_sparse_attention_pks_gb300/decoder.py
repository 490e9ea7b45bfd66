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
                 stream=None):
        t = dict(tensors)
        q = t["q"]
        dev = q.device
        self.tensors = t
        self.k = int(k)
        # q: [B, Hq, D], or [B, Nq, Hq, D] with Nq query tokens per request
        self.out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        self.topk_idx = torch.empty(tuple(q.shape[:-2]) + (self.k,), dtype=torch.int32, device=dev)
        probe = pks.make_args(k=self.k, topk_idx=self.topk_idx, out=self.out,
                              attn_splits=attn_splits, topk_mode=topk_mode, **t)
        nbytes = pks.pks_decode_workspace_size(probe)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        if self.workspace.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")
        self.args = pks.make_args(k=self.k, topk_idx=self.topk_idx, out=self.out,
                                  workspace=self.workspace, attn_splits=attn_splits,
                                  topk_mode=topk_mode, **t)
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

    def __call__(self, stream=None):
        pks.pks_decode_select(self.args, stream)
        self.table.update(self.step.topk_idx, self.block_table, self.page_size, self.miss,
                          self.n_miss, stream)
        self.table.fetch(self.miss, self.n_miss, self.host_k, self.host_v, self.slot_k,
                         self.slot_v, stream)
        pks.pks_sparse_attention_resident(self.args, self.table.state, self.capacity, self.slot_k,
                                          self.slot_v, stream)
        return self.step.out, self.step.topk_idx
