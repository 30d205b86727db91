"""pkv_decode_attention_static: decode attention for callers that may not
allocate device memory (its split-KV scratch is a fixed array inside the
library).  Called through the C ABI with ctypes; its output must match the
workspace-taking pkv_decode_attention on two calls in a row.  Kept in a file
of its own, collected last."""
import ctypes

import pytest
import torch

import paged_kv_cache_67_gb300 as pkv
from gpu_helpers import TOL, assert_close, gpu_decode
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
STATIC_BYTES = 16 * 1024 * 1024  # PKV_STATIC_SCRATCH_BYTES in include/pkv.h


def _static_fn():
    lib = pkv.load_library()
    fn = lib.pkv_decode_attention_static
    vp, c_int = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                   ctypes.c_int64, ctypes.c_float, c_int, c_int, c_int, vp, vp]
    fn.restype = c_int
    return fn


def _call_static(q, kc, vc, tables, lens, scale, partition_size, max_context_len=0):
    B, H, D = q.shape
    nb, bs, kvh, _ = kc.shape
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[q.dtype]
    status = _static_fn()(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                          tables.data_ptr(), lens.data_ptr(), B, H, kvh, D, bs, tables.shape[1],
                          nb, scale, dt, max_context_len, partition_size, err.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return status, out, int(err.item())


@pytest.mark.parametrize("dtype,D,partition_size", [(torch.bfloat16, 128, 64),
                                                    (torch.bfloat16, 128, 0),
                                                    (torch.float32, 64, 32)])
def test_static_scratch_matches_workspace_entry_point(dtype, D, partition_size):
    for call in range(2):  # two calls in a row share (and must re-clear) the scratch
        case = random_paged_case(500 + call, [1, 300, 1000, 17, 640, 2048], H=8, KVH=2, D=D,
                                 bs=16, dtype=dtype)
        args = [t.to(DEV) for t in (case["q"], case["k_cache"], case["v_cache"],
                                    case["block_tables"], case["context_lens"])]
        scale = 0.07
        status, out, err = _call_static(*args, scale, partition_size)
        assert status == 0 and err == 0, (status, err)
        want, err_ws = gpu_decode(*args, scale, partition_size=partition_size)
        assert err_ws == 0
        assert_close(out, want, dtype, f"call {call}")


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    # 64 sequences x 32 heads x 256 partitions x (128 + 2) floats >> 16 MiB
    B, H, KVH, D, bs, mb = 64, 32, 8, 128, 16, 256
    q = torch.zeros((B, H, D), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((mb, bs, KVH, D), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((B, mb), dtype=torch.int32, device=DEV)
    lens = torch.full((B,), 4096, dtype=torch.int32, device=DEV)
    need = pkv.pkv_decode_workspace_size(B, H, KVH, D, bs, mb, 4096, 16)
    assert need > STATIC_BYTES
    status, out, err = _call_static(q, kc, kc, tables, lens, 0.1, 16, 4096)
    assert status == 4  # PKV_ERR_WORKSPACE, nothing enqueued
    assert bool(torch.isnan(out).all())
