"""Top-k sparse attention decode over a paged KV cache, native to GB300 (sm_103a).

The compute path is ``libpks.so`` (C ABI, ``include/pks.h``): CUDA kernels for
the int8 indexer scan, the exact top-k selection, the paged sparse attention
and the HBM residency table, plus a host page allocator.  ``pks`` is its
ctypes binding; ``decoder`` holds a convenience wrapper that owns the output
and workspace tensors of one batch shape.
"""

from . import pks  # noqa: F401  (loads libpks.so lazily, on first call)
from .pks import (PksError, Pool, ResidencyTable, make_args, pks_alloc_pages,  # noqa: F401
                  pks_build_block_table, pks_decode_device_error, pks_decode_step,
                  pks_decode_step_timed, pks_decode_workspace_init, pks_decode_workspace_size,
                  pks_free_pages, pks_indexer_scores, pks_pool_create, pks_pool_destroy,
                  pks_pool_free_count, pks_residency_init, pks_residency_offsets,
                  pks_residency_state_bytes, pks_residency_update, pks_sparse_attention)
