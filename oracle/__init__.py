"""The oracle: plain fp64 CPU restatement of the paged KV-cache write, of
paged decode attention and of paged causal prefill attention.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it; the library (the package
``paged_kv_cache_67_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``pkv_oracle.c`` (plain C, compiled here with gcc);
this module only builds it and marshals torch CPU tensors into it.  Sources:
the course page "P09 · Paged KV 写入 + decode attention（参考实现）",
sections 题面速览 and 框架视角 · shape trace (write_kv and
paged_decode_attention tables), and the interview note "PagedAttention
kernel: paged KV cache 与 block table", section 直接答案 (paged equals dense
attention).  Every function here is pinned by tests/test_oracle_pins.py
against values the pages print, closed forms and a dense library routine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
# -std=c11 (ISO mode) and -ffp-contract=off: no fused multiply-add, so the
# oracle rounds the same way on x86-64 and on aarch64.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]

DT_F32, DT_BF16, DT_F16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: DT_F32, torch.bfloat16: DT_BF16, torch.float16: DT_F16}

ERRORS = {
    0: "ok",
    -1: "invalid argument",
    -2: "slot past the end of the pool",
    -3: "block table entry outside [0, num_blocks)",
    -4: "context length negative or longer than the block table",
    -5: "out of memory",
}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle error {code}: {ERRORS.get(code, 'unknown')}")
        self.code = code


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle into a shared library (skipped when up to date)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra_flags:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    i64, c_int, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.pkv_oracle_write.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, c_int]
    lib.pkv_oracle_write.restype = c_int
    lib.pkv_oracle_decode.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                      i64, ctypes.c_double, c_int, i64, i64, i64, i64]
    lib.pkv_oracle_decode.restype = c_int
    lib.pkv_oracle_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                       i64, ctypes.c_double, c_int, i64, i64]
    lib.pkv_oracle_prefill.restype = c_int
    lib.pkv_oracle_round.argtypes = [vp, vp, i64, c_int]
    lib.pkv_oracle_round.restype = c_int
    lib.pkv_oracle_widen.argtypes = [vp, vp, i64, c_int]
    lib.pkv_oracle_widen.restype = c_int
    return lib


def load(path: str | None = None):
    """Load a build of the oracle.  With ``path`` a separate copy is loaded
    (used by the tests that plant mistakes in a copy of the source)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(t: torch.Tensor) -> int:
    assert t.device.type == "cpu" and t.is_contiguous(), "oracle takes contiguous CPU tensors"
    return t.data_ptr()


def _check(rc: int):
    if rc != 0:
        raise OracleError(rc)


def write(k_cache, v_cache, k, v, slot_mapping, lib=None) -> None:
    """write_kv in place: k_cache/v_cache [num_blocks, bs, KVH, D]; k, v
    [T, KVH, D]; slot_mapping [T] int64.  Returns None like the page's op."""
    lib = lib or load()
    nblk, bs, kvh, d = k_cache.shape
    assert v_cache.shape == k_cache.shape and k.shape == v.shape
    assert k.dtype == v.dtype == k_cache.dtype == v_cache.dtype
    assert slot_mapping.dtype == torch.int64
    T = slot_mapping.numel()
    assert k.shape == (T, kvh, d)
    _check(lib.pkv_oracle_write(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v),
                                _ptr(slot_mapping), T, kvh * d, nblk, bs, kvh, d,
                                _DTYPE_CODE[k.dtype]))


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
           seqs: tuple[int, int] | None = None, heads: tuple[int, int] | None = None,
           out=None, lib=None):
    """Paged decode attention; returns out [B, H, D] in q.dtype.

    ``seqs=(b0, b1)`` / ``heads=(h0, h1)`` restrict the work to sequences
    b0..b1-1 and query heads h0..h1-1 (the other rows of ``out`` are left as
    they were)."""
    lib = lib or load()
    B, H, D = q.shape
    nblk, bs, kvh, d2 = k_cache.shape
    assert d2 == D and v_cache.shape == k_cache.shape
    assert q.dtype == k_cache.dtype == v_cache.dtype
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert block_tables.shape[0] == B and context_lens.shape == (B,)
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.zeros_like(q)
    b0, b1 = seqs if seqs is not None else (0, B)
    h0, h1 = heads if heads is not None else (0, H)
    _check(lib.pkv_oracle_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(block_tables), _ptr(context_lens), B, H, kvh, D, bs,
                                 max_blocks, nblk, float(scale), _DTYPE_CODE[q.dtype], b0, b1,
                                 h0, h1))
    return out


def prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens, scale: float,
            seqs: tuple[int, int] | None = None, out=None, lib=None):
    """Paged causal prefill attention; returns out [total_q, H, D] in q.dtype.

    Sequence b's qlen = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries are the
    last qlen of its context_lens[b] tokens; query i (row cu_seqlens_q[b] + i)
    attends to positions 0 .. context_lens[b] - qlen + i.  ``seqs=(b0, b1)``
    restricts the work to those sequences (other rows of ``out`` unchanged)."""
    lib = lib or load()
    total_q, H, D = q.shape
    nblk, bs, kvh, d2 = k_cache.shape
    assert d2 == D and v_cache.shape == k_cache.shape
    assert q.dtype == k_cache.dtype == v_cache.dtype
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert cu_seqlens_q.dtype == torch.int32
    B = context_lens.shape[0]
    assert block_tables.shape[0] == B and cu_seqlens_q.shape == (B + 1,)
    assert int(cu_seqlens_q[-1]) == total_q
    if out is None:
        out = torch.zeros_like(q)
    b0, b1 = seqs if seqs is not None else (0, B)
    _check(lib.pkv_oracle_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), _ptr(cu_seqlens_q), _ptr(context_lens), B, H,
                                  kvh, D, bs, block_tables.shape[1], nblk, float(scale),
                                  _DTYPE_CODE[q.dtype], b0, b1))
    return out


def round_to(x: torch.Tensor, dtype: torch.dtype, lib=None) -> torch.Tensor:
    """Round float64 values once, to nearest-even, into ``dtype``."""
    lib = lib or load()
    x = x.to(torch.float64).contiguous()
    out = torch.empty(x.shape, dtype=dtype)
    _check(lib.pkv_oracle_round(_ptr(x), _ptr(out), x.numel(), _DTYPE_CODE[dtype]))
    return out


def widen(x: torch.Tensor, lib=None) -> torch.Tensor:
    """Exact float64 value of every element of a float32/bf16/fp16 tensor."""
    lib = lib or load()
    x = x.contiguous()
    out = torch.empty(x.shape, dtype=torch.float64)
    _check(lib.pkv_oracle_widen(_ptr(x), _ptr(out), x.numel(), _DTYPE_CODE[x.dtype]))
    return out
