"""pkd: batch decode attention over a paged KV cache for GB300 (sm_103a).

``BatchDecodePagedKV`` mirrors FlashInfer's BatchDecodeWithPagedKVCacheWrapper plan()/run();
the work happens in ``_build/libpkd.so`` (hand-written CUDA kernels behind a C ABI declared
in ``include/pkd.h``).  Build it with ``paged_kv_decode_23_gb300.build.build()``.
"""
from ._lib import PkdError, LIB_PATH  # noqa: F401
from .decode import (BatchDecodePagedKV, BatchMLAPagedAttention,  # noqa: F401
                     CUDAGraphBatchDecodePagedKV, check_page_table, graph_workspace_bytes,
                     mla_graph_workspace_bytes, mla_plan_host, noalloc_check_status, plan_host,
                     workspace_bytes)

__all__ = ["BatchDecodePagedKV", "BatchMLAPagedAttention", "CUDAGraphBatchDecodePagedKV",
           "PkdError", "check_page_table", "graph_workspace_bytes", "mla_graph_workspace_bytes",
           "mla_plan_host", "noalloc_check_status", "plan_host", "workspace_bytes"]
