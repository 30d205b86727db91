"""The C ABI on the CPU: the library builds and loads, exports every entry
point include/pkv.h declares, and its host-only logic (argument checks,
workspace sizes, the decode plan) behaves.  No compute call needs a GPU."""
import ctypes
import subprocess

import pytest

from paged_kv_cache_67_gb300 import build as libbuild


@pytest.fixture(scope="module")
def pkv():
    libbuild.build()
    import paged_kv_cache_67_gb300 as m
    m.load_library()
    return m


def test_every_declared_symbol_is_exported(pkv):
    names = pkv.exported_symbols()
    assert set(names) >= {"pkv_write", "pkv_decode_attention", "pkv_decode_workspace_size",
                          "pkv_decode_plan", "pkv_status_string", "pkv_version",
                          "pkv_write_decode_attention", "pkv_decode_attention_static"}
    lib = pkv.load_library()
    for n in names:
        assert hasattr(lib, n), n
    dyn = subprocess.run(["nm", "-D", "--defined-only", pkv.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in dyn.splitlines() if " T " in line}
    assert set(names) <= exported
    # only the C ABI is visible
    assert all(s.startswith("pkv_") for s in exported), sorted(exported)


def test_status_strings_and_version(pkv):
    assert pkv.pkv_status_string(0) == "ok"
    assert "workspace" in pkv.pkv_status_string(4)
    assert pkv.pkv_status_string(99) == "unknown status"
    assert "sm_103a" in pkv.pkv_version()


def _ws_bytes(B, H, D, parts):
    """Workspace layout: one int counter per (sequence, head), then with more
    than one partition per sequence the partial (m, l) and weighted-V rows;
    every region 256-byte aligned."""
    al = lambda x: (x + 255) // 256 * 256
    rows = B * H
    head = al(rows * 4)
    return head if parts <= 1 else head + 2 * al(rows * parts * 4) + rows * parts * D * 4


def _ws_parts(cap, P):
    """Partitions per sequence the workspace holds: ceil(cap / P) for an
    explicit P; automatic: the partition is never below max(64, cap / 64)
    rounded up to 16, so at most 64."""
    if not P:
        P = max(64, -(-(-(-cap // 64)) // 16) * 16)
    return -(-cap // P)


def test_workspace_size(pkv):
    # one partition covers everything -> only the counters
    assert pkv.pkv_decode_workspace_size(4, 8, 2, 64, 16, 4, 0, 64) == _ws_bytes(4, 8, 64, 1)
    B, H, D, P, cap = 3, 8, 64, 64, 1000
    assert pkv.pkv_decode_workspace_size(B, H, 2, D, 16, 100, cap, P) == \
        _ws_bytes(B, H, D, _ws_parts(cap, P))
    for cap in (16, 100, 1000, 4096, 32768):
        assert pkv.pkv_decode_workspace_size(B, H, 2, D, 16, 4096, cap, 0) == \
            _ws_bytes(B, H, D, _ws_parts(cap, 0))
    # invalid sizes -> 0
    assert pkv.pkv_decode_workspace_size(4, 6, 4, 64, 16, 8, 0, 0) == 0   # H % KVH
    assert pkv.pkv_decode_workspace_size(4, 8, 2, 64, 16, 8, 0, 24) == 0  # P % 16
    # auto mode: never more than 64 partitions per sequence
    auto = pkv.pkv_decode_workspace_size(8, 32, 8, 128, 16, 2048, 0, 0)
    assert auto == _ws_bytes(8, 32, 128, 64)


def test_plan(pkv):
    import torch
    # tensor-core kernel (1): about four CTAs per resident slot, >= 1024 tokens
    P, mp, kern = pkv.pkv_decode_plan(64, 32, 8, 128, 16, 256, 4096, 0, torch.bfloat16, 152)
    assert kern == 1 and P % 16 == 0 and P >= 1024 and mp == -(-4096 // P)
    # enough (sequence, head) units to fill the GPU: no split
    P, mp, kern = pkv.pkv_decode_plan(256, 64, 8, 128, 16, 132, 2080, 0, torch.bfloat16, 152)
    assert kern == 1 and mp == 1
    # long contexts, few units: split
    P, mp, kern = pkv.pkv_decode_plan(8, 32, 8, 128, 16, 2048, 32768, 0, torch.bfloat16, 152)
    assert kern == 1 and 1024 <= P <= 4096 and mp > 1
    P, mp, kern = pkv.pkv_decode_plan(64, 32, 8, 128, 16, 256, 4096, 48, torch.bfloat16, 152)
    assert kern == 1 and (P, mp) == (48, -(-4096 // 48))
    # the workspace sized in auto mode always fits the automatic plan
    for B, H, KVH, D, bs, mb, cap in ((64, 32, 8, 128, 16, 256, 4096), (8, 32, 8, 128, 16, 2048, 32768),
                                      (128, 16, 1, 256, 32, 256, 8192), (1, 4, 4, 64, 16, 100, 0)):
        P, mp, _ = pkv.pkv_decode_plan(B, H, KVH, D, bs, mb, cap, 0, torch.bfloat16, 152)
        assert mp <= 64
        ws = pkv.pkv_decode_workspace_size(B, H, KVH, D, bs, mb, cap, 0)
        assert ws >= _ws_bytes(B, H, D, mp)
    # fp32, odd head_dim or block size not a multiple of 16 -> CUDA-core kernel
    assert pkv.pkv_decode_plan(4, 4, 2, 64, 16, 8, 0, 0, torch.float32)[2] == 0
    assert pkv.pkv_decode_plan(4, 4, 2, 96, 16, 8, 0, 0, torch.bfloat16)[2] == 0
    assert pkv.pkv_decode_plan(4, 4, 2, 128, 8, 8, 0, 0, torch.bfloat16)[2] == 0
    assert pkv.pkv_decode_plan(4, 4, 2, 128, 32, 8, 0, 0, torch.float16)[2] == 1
    # explicit partition size is honoured (CUDA-core kernel: one slot per partition)
    assert pkv.pkv_decode_plan(4, 4, 2, 96, 16, 64, 0, 48, torch.bfloat16)[:2] == (48, -(-1024 // 48))
    # invalid -> 0
    assert pkv.pkv_decode_plan(4, 6, 4, 128, 16, 8, 0, 0, torch.bfloat16)[0] == 0


def test_host_side_argument_errors(pkv):
    """Argument errors come back as a status before any CUDA call (so they
    are checkable without a GPU)."""
    lib = pkv.load_library()
    null = None
    # pkv_write: negative token count, bad sizes, stride shorter than a row
    assert lib.pkv_write(null, null, null, null, null, -1, 8, 8, 4, 16, 1, 8, 1, null, null) == 1
    assert lib.pkv_write(null, null, null, null, null, 4, 8, 8, 4, 0, 1, 8, 1, null, null) == 1
    assert lib.pkv_write(null, null, null, null, null, 4, 7, 8, 4, 16, 1, 8, 1, null, null) == 1
    assert lib.pkv_write(null, null, null, null, null, 4, 8, 8, 4, 16, 1, 8, 7, null, null) == 1
    # zero tokens: nothing to do
    assert lib.pkv_write(null, null, null, null, null, 0, 8, 8, 4, 16, 1, 8, 1, null, null) == 0
    # NULL pointers with work to do
    assert lib.pkv_write(null, null, null, null, null, 3, 8, 8, 4, 16, 1, 8, 1, null, null) == 1
    dec = lambda **kw: lib.pkv_decode_attention(
        kw.get("out"), kw.get("q"), kw.get("k"), kw.get("v"), kw.get("t"), kw.get("l"),
        kw.get("B", 2), kw.get("H", 4), kw.get("KVH", 2), kw.get("D", 64), kw.get("bs", 16),
        kw.get("mb", 4), kw.get("nb", 8), ctypes.c_float(0.125), kw.get("dt", 1), 0,
        kw.get("P", 0), None, 0, None, None)
    assert dec(H=6, KVH=4) == 1          # H % KVH
    assert dec(bs=0) == 1
    assert dec(P=24) == 1                # partition not a multiple of 16
    assert dec(dt=9) == 1
    assert dec(D=1024) == 2              # head_dim above 512
    assert dec(B=0) == 0                 # empty batch: nothing to do
    assert dec() == 1                    # NULL pointers

    # the fused step: the decode checks plus its new-token rows
    fake = 1 << 20  # a 16-byte-aligned address that is never dereferenced
    fz = lambda **kw: lib.pkv_write_decode_attention(
        kw.get("out"), kw.get("q"), kw.get("k", fake), kw.get("v", fake), kw.get("ks", 128),
        kw.get("vs", 128), kw.get("slots", fake), kw.get("kc"), kw.get("vc"), kw.get("t"),
        kw.get("l"), kw.get("B", 2), 4, 2, 64, 16, 4, 8, ctypes.c_float(0.125), kw.get("dt", 1),
        0, 0, None, 0, None, None)
    assert fz(B=0) == 0                  # empty batch
    assert fz() == 1                     # NULL q / out / caches
    assert fz(slots=None) == 1
    assert fz(k=fake + 8) == 1           # new-token row not 16-byte aligned
    assert fz(ks=100) == 1               # stride shorter than a row
    assert fz(ks=132) == 1               # stride not a multiple of 16 bytes
    assert fz(dt=9) == 1


def test_copy_async_argument_errors(pkv):
    """pkv_copy_async refuses NULL pointers and overlapping ranges on the host,
    before any CUDA call; zero bytes enqueue nothing."""
    lib = pkv.load_library()
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.addressof(buf)
    vp = ctypes.c_void_p
    assert lib.pkv_copy_async(None, vp(p), 16, None) == 1
    assert lib.pkv_copy_async(vp(p), None, 16, None) == 1
    assert lib.pkv_copy_async(vp(p + 8), vp(p), 64, None) == 1   # overlap
    assert lib.pkv_copy_async(vp(p), vp(p + 63), 64, None) == 1  # overlap
    assert lib.pkv_copy_async(None, None, 0, None) == 0
    assert lib.pkv_copy_async(vp(p), vp(p), 0, None) == 0


def test_copy_async_binding_checks_on_the_host(pkv):
    """The binding refuses, before any CUDA call, a copy with no tensor on the
    GPU, tensors of different byte sizes, and non-contiguous tensors."""
    import torch
    a = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(ValueError):
        pkv.pkv_copy_async(a, torch.zeros(64, dtype=torch.uint8))       # both on the host
    with pytest.raises(ValueError):
        pkv.pkv_copy_async(a, torch.zeros(32, dtype=torch.int16)[:16])  # 64 vs 32 bytes
    with pytest.raises(ValueError):
        pkv.prepare_copy_async(torch.zeros(8, 8)[:, 0], torch.zeros(8))  # not contiguous
