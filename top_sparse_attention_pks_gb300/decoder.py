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
        B, Hq, D = q.shape
        dev = q.device
        self.tensors = t
        self.k = int(k)
        self.out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
        self.topk_idx = torch.empty((B, self.k), dtype=torch.int32, device=dev)
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
        B = self.args.B
        ld = self.args.max_pages * self.args.page_size
        out = torch.zeros((B, ld), dtype=torch.int32, device=self.out.device)
        pks.pks_indexer_scores(self.args, out, stream)
        return out

    def launches(self) -> int:
        """Kernels one step enqueues on the current device."""
        return pks.pks_decode_launches(self.args)

    def device_error(self, stream=None) -> int:
        return pks.pks_decode_device_error(self.args, stream)
