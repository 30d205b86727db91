"""Paged KV-cache write and paged decode attention for one GB300 (sm_103a).

A thin Python binding over the C ABI of ``include/pkv.h`` (``libpkv.so``,
built in-tree by ``paged_kv_cache_67_gb300.build``).  The functions carry the
C names and only marshal torch tensors into pointers and sizes: every step of
the computation runs in the library's CUDA kernels.  There is no CPU
fallback; if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    FLAG_APPEND_MISMATCH,
    FLAG_BLOCK_OUT_OF_RANGE,
    FLAG_CONTEXT_NEGATIVE,
    FLAG_CONTEXT_OVER_HINT,
    FLAG_CONTEXT_TOO_LONG,
    FLAG_QUERY_LEN,
    FLAG_QUERY_OVER_HINT,
    FLAG_SLOT_OUT_OF_RANGE,
    FLAG_TIMEOUT,
    PKV_ERR_OUT_OF_BLOCKS,
    BlockManager,
    PkvError,
    PreparedCall,
    DecodeWorkspace,
    exported_symbols,
    library_path,
    load_library,
    KERNEL_AUTO,
    KERNEL_CUDA_CORE,
    KERNEL_TC,
    KERNEL_WIDE,
    pkv_decode_attention,
    pkv_decode_attention_with_kernel,
    pkv_decode_attention_xpacked,
    pkv_decode_plan,
    pkv_decode_workspace_size,
    pkv_copy_async,
    pkv_hbm_copy,
    pkv_hbm_gather_read,
    pkv_hbm_gather_read_pair,
    pkv_fp32_fma_peak,
    FMA_THREADS,
    FMA_CHAINS,
    pkv_prefill_attention,
    pkv_status_string,
    pkv_version,
    pkv_write,
    pkv_write_decode_attention,
    pkv_write_xpacked,
    prepare_copy_async,
    prepare_decode_attention,
    prepare_write_decode_attention,
)
