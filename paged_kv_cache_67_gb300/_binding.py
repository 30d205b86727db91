"""ctypes binding of libpkv.so: argument marshalling only.

Each function takes torch tensors, checks the shapes/dtypes/devices needed
to fill the C arguments, and calls the C entry point of the same name on the
caller's current CUDA stream (or the given one).  Status codes other than
PKV_OK raise PkvError.  Memory is the caller's: nothing here allocates on
the call path (DecodeWorkspace is a one-off helper that allocates the
workspace buffer with torch, zero-filled).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libpkv.so")
_INCLUDE = os.path.join(os.path.dirname(_PKG), "include")

PKV_F32, PKV_BF16, PKV_F16 = 0, 1, 2
_DT = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.float16: PKV_F16}

FLAG_SLOT_OUT_OF_RANGE = 0x1
FLAG_BLOCK_OUT_OF_RANGE = 0x2
FLAG_CONTEXT_TOO_LONG = 0x4
FLAG_CONTEXT_NEGATIVE = 0x8
FLAG_CONTEXT_OVER_HINT = 0x10
FLAG_TIMEOUT = 0x20
FLAG_APPEND_MISMATCH = 0x40
FLAG_QUERY_LEN = 0x80
FLAG_QUERY_OVER_HINT = 0x100

_lock = threading.Lock()
_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({pkv_status_string(status)})")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libpkv.so (raises if it has not been built: no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m paged_kv_cache_67_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, c_int, c_size = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.pkv_write.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, c_int, c_int, c_int,
                                  c_int, vp, vp]
        lib.pkv_write.restype = c_int
        lib.pkv_decode_workspace_size.argtypes = [c_int] * 8
        lib.pkv_decode_workspace_size.restype = c_size
        lib.pkv_decode_plan.argtypes = [c_int] * 10 + [ctypes.POINTER(c_int), ctypes.POINTER(c_int)]
        lib.pkv_decode_plan.restype = c_int
        lib.pkv_decode_attention.argtypes = [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                             c_int, c_int, i64, ctypes.c_float, c_int, c_int,
                                             c_int, vp, c_size, vp, vp]
        lib.pkv_decode_attention.restype = c_int
        lib.pkv_decode_attention_with_kernel.argtypes = [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int,
                                                         c_int, c_int, c_int, i64, ctypes.c_float,
                                                         c_int, c_int, c_int, vp, c_size, vp, c_int,
                                                         vp]
        lib.pkv_decode_attention_with_kernel.restype = c_int
        lib.pkv_write_decode_attention.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp,
                                                   c_int, c_int, c_int, c_int, c_int, c_int, i64,
                                                   ctypes.c_float, c_int, c_int, c_int, vp, c_size,
                                                   vp, vp]
        lib.pkv_write_decode_attention.restype = c_int
        lib.pkv_write_xpacked.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, c_int, c_int, c_int,
                                          c_int, vp, vp]
        lib.pkv_write_xpacked.restype = c_int
        lib.pkv_decode_attention_xpacked.argtypes = lib.pkv_decode_attention.argtypes
        lib.pkv_decode_attention_xpacked.restype = c_int
        lib.pkv_prefill_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, c_int, i64, c_int, c_int,
                                              c_int, c_int, c_int, i64, ctypes.c_float, c_int, c_int,
                                              vp, vp]
        lib.pkv_prefill_attention.restype = c_int
        P = ctypes.POINTER
        lib.pkv_bm_create.argtypes = [i64, c_int, c_int, P(vp)]
        lib.pkv_bm_create.restype = c_int
        lib.pkv_bm_destroy.argtypes = [vp]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_add_sequence.argtypes = [vp, i64, vp, i64, vp, P(i64)]
        lib.pkv_bm_add_sequence.restype = c_int
        lib.pkv_bm_append_tokens.argtypes = [vp, vp, vp, c_int, vp]
        lib.pkv_bm_append_tokens.restype = c_int
        lib.pkv_bm_free_sequence.argtypes = [vp, i64]
        lib.pkv_bm_free_sequence.restype = c_int
        lib.pkv_bm_build_batch.argtypes = [vp, vp, c_int, c_int, ctypes.c_int32, vp, vp]
        lib.pkv_bm_build_batch.restype = c_int
        lib.pkv_bm_sequence_info.argtypes = [vp, i64, P(i64), P(c_int), vp, c_int]
        lib.pkv_bm_sequence_info.restype = c_int
        lib.pkv_bm_stats.argtypes = [vp, P(i64), P(i64), P(i64)]
        lib.pkv_bm_stats.restype = None
        lib.pkv_bm_block_refcount.argtypes = [vp, i64]
        lib.pkv_bm_block_refcount.restype = c_int
        lib.pkv_hbm_copy.argtypes = [vp, vp, c_size, vp]
        lib.pkv_hbm_copy.restype = c_int
        lib.pkv_copy_async.argtypes = [vp, vp, c_size, vp]
        lib.pkv_copy_async.restype = c_int
        lib.pkv_hbm_gather_read.argtypes = [vp, vp, i64, i64, i64, vp, vp]
        lib.pkv_hbm_gather_read.restype = c_int
        lib.pkv_hbm_gather_read_pair.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
        lib.pkv_hbm_gather_read_pair.restype = c_int
        lib.pkv_fp32_fma_peak.argtypes = [vp, c_int, c_int, ctypes.c_float, ctypes.c_float,
                                          ctypes.c_float, c_int, vp]
        lib.pkv_fp32_fma_peak.restype = c_int
        lib.pkv_status_string.argtypes = [c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def exported_symbols() -> list[str]:
    """Names of the entry points the headers under include/ declare (PKV_API)."""
    names = []
    for h in sorted(os.listdir(_INCLUDE)):
        if h.endswith(".h"):
            with open(os.path.join(_INCLUDE, h)) as f:
                names += re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", f.read())
    return names


def pkv_status_string(status: int) -> str:
    return load_library().pkv_status_string(status).decode()


def pkv_version() -> str:
    return load_library().pkv_version().decode()


def _stream_handle(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str):
    if status != 0:
        raise PkvError(status, what)


def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def pkv_write(k_cache, v_cache, k, v, slot_mapping, err_flags=None, stream=None) -> None:
    """write_kv in place: k_cache/v_cache [num_blocks, bs, KVH, D]; k, v
    [T, KVH, D] (each token's row contiguous; the token stride may be
    larger); slot_mapping [T] int64 with negative = padding."""
    lib = load_library()
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape, "caches must be [nb, bs, KVH, D]")
    nb, bs, kvh, d = k_cache.shape
    _require(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    _require(k.dim() == 3 and v.shape == k.shape and k.shape[1:] == (kvh, d), "k, v must be [T, KVH, D]")
    _require(k.stride(2) == 1 and k.stride(1) == d and v.stride(2) == 1 and v.stride(1) == d,
             "each token's [KVH, D] row must be contiguous")
    _require(k.dtype == v.dtype == k_cache.dtype == v_cache.dtype and k.dtype in _DT, "dtype mismatch")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
             and slot_mapping.numel() == k.shape[0], "slot_mapping must be contiguous int64 [T]")
    dev = k_cache.device
    _require(dev.type == "cuda" and all(t.device == dev for t in (v_cache, k, v, slot_mapping)),
             "all tensors must be on the same CUDA device")
    T = k.shape[0]
    _check(lib.pkv_write(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), _ptr(slot_mapping), T,
                         k.stride(0) if T > 0 else kvh * d, v.stride(0) if T > 0 else kvh * d, nb,
                         bs, kvh, d, _DT[k.dtype], _ptr(err_flags), _stream_handle(stream, dev)),
           "pkv_write")


def pkv_decode_workspace_size(B, H, num_kv_heads, head_dim, block_size, max_blocks,
                              max_context_len=0, partition_size=0) -> int:
    return int(load_library().pkv_decode_workspace_size(B, H, num_kv_heads, head_dim, block_size,
                                                        max_blocks, max_context_len, partition_size))


def pkv_decode_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks, max_context_len=0,
                    partition_size=0, dtype=torch.bfloat16, num_sms=152):
    """(partition_size, max_partitions, kernel) the library would use
    (kernel 2 = wide-group tcgen05, 1 = TMA/tensor-core, 0 = CUDA-core); host only."""
    mp, kern = ctypes.c_int(0), ctypes.c_int(0)
    P = load_library().pkv_decode_plan(B, H, num_kv_heads, head_dim, block_size, max_blocks,
                                       max_context_len, partition_size, _DT[dtype], num_sms,
                                       ctypes.byref(mp), ctypes.byref(kern))
    return P, mp.value, kern.value


class DecodeWorkspace:
    """A zero-filled device workspace sized for pkv_decode_attention."""

    def __init__(self, B, H, num_kv_heads, head_dim, block_size, max_blocks, max_context_len=0,
                 partition_size=0, device="cuda"):
        self.nbytes = pkv_decode_workspace_size(B, H, num_kv_heads, head_dim, block_size,
                                                max_blocks, max_context_len, partition_size)
        self.buffer = torch.zeros(max(self.nbytes, 256), dtype=torch.uint8, device=device)


def _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens):
    _require(q.dim() == 3 and out.shape == q.shape, "q and out must be [B, H, D]")
    B, H, D = q.shape
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape and k_cache.shape[3] == D,
             "caches must be [nb, bs, KVH, D]")
    for t in (out, q, k_cache, v_cache, block_tables, context_lens):
        _require(t.is_contiguous(), "tensors must be contiguous")
    _require(q.dtype == out.dtype == k_cache.dtype == v_cache.dtype and q.dtype in _DT, "dtype mismatch")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B,
             "block_tables must be int32 [B, max_blocks]")
    _require(context_lens.dtype == torch.int32 and context_lens.shape == (B,), "context_lens must be int32 [B]")
    dev = q.device
    _require(dev.type == "cuda" and all(t.device == dev for t in (k_cache, v_cache, block_tables,
                                                                   context_lens)),
             "all tensors must be on the same CUDA device")
    # out may also be pinned host memory: the kernels only store to it, so
    # the result crosses to the host inside the launch
    _require(out.device == dev or (out.device.type == "cpu" and out.is_pinned()),
             "out must be on q's CUDA device or in pinned host memory")
    return dev


def _workspace_arg(workspace):
    if workspace is None:
        return None, 0
    buf = workspace.buffer if isinstance(workspace, DecodeWorkspace) else workspace
    return _ptr(buf), buf.numel() * buf.element_size()


def pkv_write_decode_attention(out, q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                               context_lens, scale: float, max_context_len: int = 0,
                               partition_size: int = 0, workspace=None, err_flags=None,
                               stream=None):
    """One decode step in one launch: write each sequence's new token k[b], v[b]
    ([B, KVH, D]) at slot_mapping[b] (int64 [B], negative = none), then paged
    decode attention into ``out`` [B, H, D] (returned) over contexts that
    already count the new token (slot_mapping[b] must be the slot of position
    context_lens[b] - 1).  ``out`` may be a pinned host tensor: the kernels
    only store to it, so the result reaches the host inside the launch."""
    lib = load_library()
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    _require(k.dim() == 3 and v.shape == k.shape and k.shape == (B, kvh, D), "k, v must be [B, KVH, D]")
    _require(k.stride(2) == 1 and k.stride(1) == D and v.stride(2) == 1 and v.stride(1) == D,
             "each token's [KVH, D] row must be contiguous")
    _require(k.dtype == v.dtype == q.dtype, "dtype mismatch")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
             and slot_mapping.shape == (B,), "slot_mapping must be contiguous int64 [B]")
    _require(all(t.device == dev for t in (k, v, slot_mapping)), "all tensors must be on the same CUDA device")
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    _check(lib.pkv_write_decode_attention(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), k.stride(0) if B > 0 else kvh * D,
        v.stride(0) if B > 0 else kvh * D, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), B, H, kvh, D, bs, block_tables.shape[1], nb,
        float(scale), _DT[q.dtype], int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
        _ptr(err_flags), _stream_handle(stream, dev)), "pkv_write_decode_attention")
    return out


class PreparedCall:
    """One library call whose arguments were checked and marshalled once.

    Calling it enqueues the call again on the same tensors' memory (their
    storage must stay where it was: write new inputs into the same tensors,
    as a serving loop that reuses its step buffers does) with the argument
    list built at preparation, so each call costs one ctypes call and no
    Python-side checks.  Raises PkvError on a status other than PKV_OK."""

    __slots__ = ("_fn", "_args", "_what", "_keep")

    def __init__(self, fn, args, what, keep):
        self._fn, self._args, self._what, self._keep = fn, tuple(args), what, keep

    def __call__(self):
        status = self._fn(*self._args)
        if status != 0:
            raise PkvError(status, self._what)


def prepare_write_decode_attention(out, q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                                   context_lens, scale: float, max_context_len: int = 0,
                                   partition_size: int = 0, workspace=None, err_flags=None,
                                   stream=None) -> PreparedCall:
    """pkv_write_decode_attention, checked and marshalled once: returns a
    callable that enqueues the step on the same buffers (see PreparedCall)."""
    lib = load_library()
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    _require(k.dim() == 3 and v.shape == k.shape and k.shape == (B, kvh, D), "k, v must be [B, KVH, D]")
    _require(k.stride(2) == 1 and k.stride(1) == D and v.stride(2) == 1 and v.stride(1) == D,
             "each token's [KVH, D] row must be contiguous")
    _require(k.dtype == v.dtype == q.dtype, "dtype mismatch")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
             and slot_mapping.shape == (B,), "slot_mapping must be contiguous int64 [B]")
    _require(all(t.device == dev for t in (k, v, slot_mapping)), "all tensors must be on the same CUDA device")
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    args = (_ptr(out), _ptr(q), _ptr(k), _ptr(v), k.stride(0) if B > 0 else kvh * D,
            v.stride(0) if B > 0 else kvh * D, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), _ptr(context_lens), B, H, kvh, D, bs, block_tables.shape[1], nb,
            float(scale), _DT[q.dtype], int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
            _ptr(err_flags), _stream_handle(stream, dev))
    keep = (out, q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, workspace, err_flags)
    return PreparedCall(lib.pkv_write_decode_attention, args, "pkv_write_decode_attention", keep)


def prepare_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                             max_context_len: int = 0, partition_size: int = 0, workspace=None,
                             err_flags=None, stream=None) -> PreparedCall:
    """pkv_decode_attention, checked and marshalled once (see PreparedCall)."""
    lib = load_library()
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            B, H, kvh, D, bs, block_tables.shape[1], nb, float(scale), _DT[q.dtype],
            int(max_context_len), int(partition_size), ws_ptr, ws_bytes, _ptr(err_flags),
            _stream_handle(stream, dev))
    keep = (out, q, k_cache, v_cache, block_tables, context_lens, workspace, err_flags)
    return PreparedCall(lib.pkv_decode_attention, args, "pkv_decode_attention", keep)


def pkv_prefill_attention(out, q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens,
                          scale: float, max_q_len: int = 0, err_flags=None, stream=None):
    """Paged causal prefill attention into ``out`` [total_q, H, D] (returned):
    sequence b's queries are rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of
    ``q``, the last tokens of its context_lens[b] (already written)."""
    lib = load_library()
    _require(q.dim() == 3 and out.shape == q.shape, "q and out must be [total_q, H, D]")
    total_q, H, D = q.shape
    _require(k_cache.dim() == 4 and v_cache.shape == k_cache.shape and k_cache.shape[3] == D,
             "caches must be [nb, bs, KVH, D]")
    nb, bs, kvh, _ = k_cache.shape
    for t in (out, q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens):
        _require(t.is_contiguous(), "tensors must be contiguous")
    _require(q.dtype == out.dtype == k_cache.dtype == v_cache.dtype and q.dtype in _DT, "dtype mismatch")
    B = context_lens.shape[0]
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B,
             "block_tables must be int32 [B, max_blocks]")
    _require(context_lens.dtype == torch.int32 and context_lens.dim() == 1, "context_lens must be int32 [B]")
    _require(cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.shape == (B + 1,),
             "cu_seqlens_q must be int32 [B + 1]")
    dev = q.device
    _require(dev.type == "cuda" and all(t.device == dev for t in (out, k_cache, v_cache, block_tables,
                                                                   cu_seqlens_q, context_lens)),
             "all tensors must be on the same CUDA device")
    _check(lib.pkv_prefill_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(context_lens), B,
                                     total_q, H, kvh, D, bs, block_tables.shape[1], nb, float(scale),
                                     _DT[q.dtype], int(max_q_len), _ptr(err_flags),
                                     _stream_handle(stream, dev)), "pkv_prefill_attention")
    return out


def pkv_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                         max_context_len: int = 0, partition_size: int = 0, workspace=None,
                         err_flags=None, stream=None):
    """Paged decode attention into ``out`` [B, H, D] (returned): on q's
    device, or a pinned host tensor that the kernels store the result into."""
    lib = load_library()
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    _check(lib.pkv_decode_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    _ptr(block_tables), _ptr(context_lens), B, H, kvh, D, bs,
                                    block_tables.shape[1], nb, float(scale), _DT[q.dtype],
                                    int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                                    _ptr(err_flags), _stream_handle(stream, dev)),
           "pkv_decode_attention")
    return out


KERNEL_AUTO, KERNEL_CUDA_CORE, KERNEL_TC, KERNEL_WIDE = -1, 0, 1, 2


def pkv_decode_attention_with_kernel(out, q, k_cache, v_cache, block_tables, context_lens,
                                     scale: float, kernel: int, max_context_len: int = 0,
                                     partition_size: int = 0, workspace=None, err_flags=None,
                                     stream=None):
    """pkv_decode_attention on the kernel named by ``kernel`` (-1 the plan's
    choice, 0 CUDA-core, 1 TMA + mma.sync, 2 wide-group tcgen05): for tests
    and tuning.  A kernel that cannot run the shape raises PkvError
    (status PKV_ERR_UNSUPPORTED)."""
    lib = load_library()
    dev = _decode_checks(out, q, k_cache, v_cache, block_tables, context_lens)
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    _check(lib.pkv_decode_attention_with_kernel(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        B, H, kvh, D, bs, block_tables.shape[1], nb, float(scale), _DT[q.dtype],
        int(max_context_len), int(partition_size), ws_ptr, ws_bytes, _ptr(err_flags), int(kernel),
        _stream_handle(stream, dev)), "pkv_decode_attention_with_kernel")
    return out


def _copy_args(dst, src, stream):
    nbytes = src.numel() * src.element_size()
    _require(dst.numel() * dst.element_size() == nbytes, "dst and src differ in size")
    _require(src.is_contiguous() and dst.is_contiguous(), "tensors must be contiguous")
    cuda = [t.device for t in (dst, src) if t.device.type == "cuda"]
    _require(len(cuda) > 0 and all(d == cuda[0] for d in cuda),
             "one tensor must be on a CUDA device (both on the same one)")
    return _ptr(dst), _ptr(src), nbytes, _stream_handle(stream, cuda[0])


def pkv_copy_async(dst, src, stream=None) -> None:
    """Enqueue a copy of src's bytes into dst (same byte size, contiguous;
    host or device, at least one on the GPU) on the stream: a step's staged
    inputs in, or its output out.  Pinned host tensors give an asynchronous
    copy."""
    lib = load_library()
    _check(lib.pkv_copy_async(*_copy_args(dst, src, stream)), "pkv_copy_async")


def prepare_copy_async(dst, src, stream=None) -> PreparedCall:
    """pkv_copy_async, checked and marshalled once (see PreparedCall): a
    serving loop's per-step copy in or out of the same buffers."""
    lib = load_library()
    return PreparedCall(lib.pkv_copy_async, _copy_args(dst, src, stream), "pkv_copy_async",
                        (dst, src))


def pkv_hbm_copy(dst, src, stream=None) -> None:
    """Streaming device-to-device copy of src's bytes into dst (the same
    byte size, contiguous, 16-byte aligned, not overlapping): the library's
    yardstick for HBM bandwidth."""
    lib = load_library()
    nbytes = src.numel() * src.element_size()
    _require(dst.numel() * dst.element_size() == nbytes, "dst and src differ in size")
    _require(src.is_contiguous() and dst.is_contiguous(), "tensors must be contiguous")
    _require(src.device.type == "cuda" and dst.device == src.device,
             "both tensors must be on the same CUDA device")
    _check(lib.pkv_hbm_copy(_ptr(dst), _ptr(src), nbytes, _stream_handle(stream, src.device)),
           "pkv_hbm_copy")


def pkv_hbm_gather_read(base, chunk_index, chunk_stride_bytes: int, chunk_bytes: int, sink,
                        stream=None, check_bounds: bool = True) -> None:
    """Read chunk_bytes at base + chunk_index[i] * chunk_stride_bytes for
    every i, XOR-folding the 16-byte words into sink (a 1-element int64
    device tensor): the library's yardstick for reads of randomly placed
    cache blocks.  Every chunk must lie inside ``base``'s storage
    (``check_bounds`` verifies it, at the cost of a device synchronisation)."""
    lib = load_library()
    _require(chunk_index.dtype == torch.int32 and chunk_index.dim() == 1 and chunk_index.is_contiguous(),
             "chunk_index must be contiguous int32 [n]")
    _require(sink.dtype == torch.int64 and sink.numel() == 1, "sink must be one int64")
    dev = base.device
    _require(dev.type == "cuda" and chunk_index.device == dev and sink.device == dev,
             "all tensors must be on the same CUDA device")
    n = chunk_index.numel()
    if n and check_bounds:
        span = base.numel() * base.element_size()
        hi = int(chunk_index.max()) * chunk_stride_bytes + chunk_bytes
        _require(int(chunk_index.min()) >= 0 and hi <= span, "a chunk lies outside base")
    _check(lib.pkv_hbm_gather_read(_ptr(base), _ptr(chunk_index), n, int(chunk_stride_bytes),
                                   int(chunk_bytes), _ptr(sink), _stream_handle(stream, dev)),
           "pkv_hbm_gather_read")


def pkv_hbm_gather_read_pair(base_a, base_b, chunk_index, chunk_stride_bytes: int, chunk_bytes: int,
                             sink, stream=None, check_bounds: bool = True) -> None:
    """pkv_hbm_gather_read over two buffers (a batch's K and V caches) in
    one launch: every listed chunk of base_a, then of base_b, XOR-folded
    into sink."""
    lib = load_library()
    _require(chunk_index.dtype == torch.int32 and chunk_index.dim() == 1 and chunk_index.is_contiguous(),
             "chunk_index must be contiguous int32 [n]")
    _require(sink.dtype == torch.int64 and sink.numel() == 1, "sink must be one int64")
    dev = base_a.device
    _require(dev.type == "cuda" and base_b.device == dev and chunk_index.device == dev and sink.device == dev,
             "all tensors must be on the same CUDA device")
    n = chunk_index.numel()
    if n and check_bounds:
        hi = int(chunk_index.max()) * chunk_stride_bytes + chunk_bytes
        for base in (base_a, base_b):
            _require(int(chunk_index.min()) >= 0 and hi <= base.numel() * base.element_size(),
                     "a chunk lies outside a base")
    _check(lib.pkv_hbm_gather_read_pair(_ptr(base_a), _ptr(base_b), _ptr(chunk_index), n,
                                        int(chunk_stride_bytes), int(chunk_bytes), _ptr(sink),
                                        _stream_handle(stream, dev)),
           "pkv_hbm_gather_read_pair")


FMA_THREADS = 256   # threads per block of pkv_fp32_fma_peak
FMA_CHAINS = 8      # independent multiply-add chains per thread


def pkv_fp32_fma_peak(out, iters: int, a: float = 1.0, b: float = 1.0, never: float = -1.0,
                      paired: bool = False, stream=None) -> None:
    """The CUDA-core fp32 yardstick: out.numel() blocks of FMA_THREADS
    threads, each running FMA_CHAINS multiply-add chains x <- x * a + b for
    `iters` steps (2 * FMA_CHAINS * iters flops per thread); thread 0 of
    block i stores the sum of its chains in out[i] (a contiguous float32
    CUDA tensor).  ``paired`` uses the two-lane fma.rn.f32x2."""
    lib = load_library()
    _require(out.dtype == torch.float32 and out.is_contiguous() and out.device.type == "cuda",
             "out must be a contiguous float32 CUDA tensor")
    _require(int(iters) >= 0 and 1 <= out.numel() <= (1 << 20), "iters >= 0 and 1..2^20 blocks")
    _check(lib.pkv_fp32_fma_peak(_ptr(out), out.numel(), int(iters), float(a), float(b), float(never),
                                 int(bool(paired)), _stream_handle(stream, out.device)),
           "pkv_fp32_fma_peak")


PKV_ERR_OUT_OF_BLOCKS = 5


class BlockManager:
    """Host block manager of libpkv (include/pkv_block_manager.h): block pool,
    per-sequence tables, slots for new tokens, prefix sharing of full blocks.
    Arrays go in and out as CPU torch tensors (int64 token ids and slots,
    int32 tables and lengths)."""

    def __init__(self, num_blocks: int, block_size: int, prefix_caching: bool = True):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.pkv_bm_create(int(num_blocks), int(block_size), int(bool(prefix_caching)),
                                       ctypes.byref(h)), "pkv_bm_create")
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @staticmethod
    def _i64(x):
        t = torch.as_tensor(x, dtype=torch.int64).contiguous()
        _require(t.device.type == "cpu", "host arrays only")
        return t

    def add_sequence(self, seq_id: int, token_ids):
        """Admit a sequence with its prompt; returns (slot_mapping [n] int64 with
        -1 for cached tokens, number of cached leading tokens)."""
        tok = self._i64(token_ids)
        slots = torch.empty(tok.numel(), dtype=torch.int64)
        cached = ctypes.c_int64()
        _check(self._lib.pkv_bm_add_sequence(self._h, int(seq_id), tok.data_ptr(), tok.numel(),
                                             slots.data_ptr(), ctypes.byref(cached)),
               "pkv_bm_add_sequence")
        return slots, cached.value

    def append_tokens(self, seq_ids, token_ids):
        """One decode step: append token_ids[i] to seq_ids[i] (negative id =
        padding); returns the new tokens' slots (-1 for padding)."""
        ids, tok = self._i64(seq_ids), self._i64(token_ids)
        _require(ids.numel() == tok.numel(), "seq_ids and token_ids differ in length")
        slots = torch.empty(ids.numel(), dtype=torch.int64)
        _check(self._lib.pkv_bm_append_tokens(self._h, ids.data_ptr(), tok.data_ptr(), ids.numel(),
                                              slots.data_ptr()), "pkv_bm_append_tokens")
        return slots

    def free_sequence(self, seq_id: int):
        _check(self._lib.pkv_bm_free_sequence(self._h, int(seq_id)), "pkv_bm_free_sequence")

    def build_batch(self, seq_ids, max_blocks: int, tail: int = 99999):
        """(block_tables [B, max_blocks] int32, context_lens [B] int32) of a batch."""
        ids = self._i64(seq_ids)
        tables = torch.empty((ids.numel(), max_blocks), dtype=torch.int32)
        lens = torch.empty(ids.numel(), dtype=torch.int32)
        _check(self._lib.pkv_bm_build_batch(self._h, ids.data_ptr(), ids.numel(), int(max_blocks),
                                            int(tail), tables.data_ptr(), lens.data_ptr()),
               "pkv_bm_build_batch")
        return tables, lens

    def sequence_info(self, seq_id: int):
        """(context_len, block table as a list)."""
        n, nb = ctypes.c_int64(), ctypes.c_int()
        _check(self._lib.pkv_bm_sequence_info(self._h, int(seq_id), ctypes.byref(n), ctypes.byref(nb),
                                              None, 0), "pkv_bm_sequence_info")
        table = torch.empty(nb.value, dtype=torch.int32)
        _check(self._lib.pkv_bm_sequence_info(self._h, int(seq_id), ctypes.byref(n), ctypes.byref(nb),
                                              table.data_ptr() if nb.value else None, nb.value),
               "pkv_bm_sequence_info")
        return n.value, table.tolist()

    def stats(self):
        """(free blocks, registered cached blocks, live sequences)."""
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        self._lib.pkv_bm_stats(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
        return a.value, b.value, c.value

    def refcount(self, block: int) -> int:
        return self._lib.pkv_bm_block_refcount(self._h, int(block))


# ------------------------------------------------------- layout experiment

def _xpacked_cache_checks(k_cache_x, v_cache_x):
    _require(k_cache_x.dim() == 5 and k_cache_x.shape[3] == 16 and k_cache_x.shape[4] == 8,
             "k_cache_x must be [nb, KVH, D/8, 16, 8]")
    nb, kvh, dg, bs, _ = k_cache_x.shape
    _require(v_cache_x.shape == (nb, kvh, dg * 8, bs), "v_cache_x must be [nb, KVH, D, 16]")
    _require(k_cache_x.is_contiguous() and v_cache_x.is_contiguous(), "caches must be contiguous")
    # (fp32 passes: the library answers PKV_ERR_UNSUPPORTED for it)
    _require(k_cache_x.dtype == v_cache_x.dtype and k_cache_x.dtype in _DT,
             "packed caches must have one dtype of float32, bfloat16, float16")
    _require(k_cache_x.device.type == "cuda" and v_cache_x.device == k_cache_x.device,
             "caches must be on one CUDA device")


def pkv_write_xpacked(k_cache_x, v_cache_x, k, v, slot_mapping, err_flags=None, stream=None) -> None:
    """write_kv into the packed layout: k_cache_x [nb, KVH, D/8, 16, 8],
    v_cache_x [nb, KVH, D, 16]; k, v [T, KVH, D]; slot_mapping [T] int64."""
    lib = load_library()
    _xpacked_cache_checks(k_cache_x, v_cache_x)
    nb, kvh, dg, bs, _ = k_cache_x.shape
    d = dg * 8
    _require(k.dim() == 3 and v.shape == k.shape and k.shape[1:] == (kvh, d), "k, v must be [T, KVH, D]")
    _require(k.stride(2) == 1 and k.stride(1) == d and v.stride(2) == 1 and v.stride(1) == d,
             "each token's [KVH, D] row must be contiguous")
    _require(k.dtype == v.dtype == k_cache_x.dtype and k.dtype in _DT, "dtype mismatch")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous()
             and slot_mapping.numel() == k.shape[0], "slot_mapping must be contiguous int64 [T]")
    dev = k_cache_x.device
    _require(all(t.device == dev for t in (k, v, slot_mapping)),
             "all tensors must be on the same CUDA device")
    T = k.shape[0]
    _check(lib.pkv_write_xpacked(_ptr(k_cache_x), _ptr(v_cache_x), _ptr(k), _ptr(v), _ptr(slot_mapping), T,
                                 k.stride(0) if T > 0 else kvh * d, v.stride(0) if T > 0 else kvh * d,
                                 nb, bs, kvh, d, _DT[k.dtype], _ptr(err_flags), _stream_handle(stream, dev)),
           "pkv_write_xpacked")


def pkv_decode_attention_xpacked(out, q, k_cache_x, v_cache_x, block_tables, context_lens, scale: float,
                                 max_context_len: int = 0, partition_size: int = 0, workspace=None,
                                 err_flags=None, stream=None):
    """Paged decode attention over packed caches (see pkv_write_xpacked)."""
    lib = load_library()
    _require(q.dim() == 3 and out.shape == q.shape, "q and out must be [B, H, D]")
    B, H, D = q.shape
    _xpacked_cache_checks(k_cache_x, v_cache_x)
    nb, kvh, dg, bs, _ = k_cache_x.shape
    _require(dg * 8 == D, "packed caches do not match q")
    for t in (out, q, block_tables, context_lens):
        _require(t.is_contiguous(), "tensors must be contiguous")
    _require(q.dtype == out.dtype == k_cache_x.dtype and q.dtype in _DT, "dtype mismatch")
    _require(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == B,
             "block_tables must be int32 [B, max_blocks]")
    _require(context_lens.dtype == torch.int32 and context_lens.shape == (B,), "context_lens must be int32 [B]")
    dev = q.device
    _require(dev.type == "cuda" and all(t.device == dev for t in (out, k_cache_x, v_cache_x, block_tables,
                                                                   context_lens)),
             "all tensors must be on the same CUDA device")
    ws_ptr, ws_bytes = _workspace_arg(workspace)
    _check(lib.pkv_decode_attention_xpacked(_ptr(out), _ptr(q), _ptr(k_cache_x), _ptr(v_cache_x),
                                            _ptr(block_tables), _ptr(context_lens), B, H, kvh, D, bs,
                                            block_tables.shape[1], nb, float(scale), _DT[q.dtype],
                                            int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                                            _ptr(err_flags), _stream_handle(stream, q.device)),
           "pkv_decode_attention_xpacked")
    return out
