"""pkv_decode_attention_static: decode attention for callers that may not
allocate device memory -- an engine plugin whose execute step must not call
cudaMalloc, code that enqueues work while another component owns the
allocator, a deployment whose device memory is fixed at start-up.  Its
split-KV scratch is a fixed array inside the library instead of a
caller-provided workspace.

Called through the C ABI with ctypes.  Its output must match the
workspace-taking pkv_decode_attention and the oracle, on two calls in a row
(the calls share the array, so the second must clear what the first left),
on every decode kernel: CUDA-core (fp32), TMA + mma.sync (bf16 / fp16 at
four heads per KV head) and the wide-group tcgen05 kernel (16 heads per KV
head, head_dim 256, block size 32).  Kept in a file of its own, collected
last."""
import ctypes

import pytest
import torch

import paged_kv_cache_67_gb300 as pkv
from gpu_helpers import assert_close, gpu_decode, oracle_decode
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


def _call_static(q, kc, vc, tables, lens, scale, partition_size, max_context_len=0, out=None):
    B, H, D = q.shape
    nb, bs, kvh, _ = kc.shape
    if out is None:
        out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}[q.dtype]
    status = _static_fn()(out.data_ptr(), q.data_ptr(), kc.data_ptr(),
                          vc.data_ptr(), tables.data_ptr(), lens.data_ptr(), B, H, kvh, D, bs,
                          tables.shape[1], nb, scale, dt, max_context_len, partition_size,
                          err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return status, out, int(err.item())


# (dtype, H, KVH, D, block size, partition size, lengths, the kernel the plan picks)
CASES = [
    (torch.bfloat16, 8, 2, 128, 16, 64, [1, 300, 1000, 17, 640, 2048], 1),
    (torch.bfloat16, 8, 2, 128, 16, 0, [1, 300, 1000, 17, 640, 2048], 1),
    (torch.float16, 8, 2, 128, 16, 48, [1, 300, 1000, 17, 640, 2048], 1),
    (torch.float32, 8, 2, 64, 16, 32, [1, 300, 1000, 17, 640, 2048], 0),
    (torch.bfloat16, 16, 1, 256, 32, 0, [1, 32, 64, 4096, 31, 33, 700, 2500], 2),
    (torch.bfloat16, 16, 1, 256, 32, 256, [1, 32, 64, 4096, 31, 33, 700, 2500], 2),
]


@pytest.mark.parametrize("dtype,H,KVH,D,bs,partition_size,lens,kernel", CASES)
def test_static_scratch_matches_workspace_entry_point_and_oracle(dtype, H, KVH, D, bs,
                                                                 partition_size, lens, kernel):
    assert pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, -(-max(lens) // bs) + 2,
                               partition_size=partition_size, dtype=dtype)[2] == kernel
    for call in range(2):  # two calls in a row share (and must re-clear) the scratch
        case = random_paged_case(500 + call + 7 * D + H, lens, H=H, KVH=KVH, D=D, bs=bs,
                                 dtype=dtype)
        args = [t.to(DEV) for t in (case["q"], case["k_cache"], case["v_cache"],
                                    case["block_tables"], case["context_lens"])]
        scale = 0.07
        status, out, err = _call_static(*args, scale, partition_size)
        assert status == 0 and err == 0, (status, err)
        want_ws, err_ws = gpu_decode(*args, scale, partition_size=partition_size)
        assert err_ws == 0
        assert_close(out, want_ws, dtype, f"call {call} vs pkv_decode_attention")
        want = oracle_decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                             case["context_lens"], scale)
        assert_close(out, want, dtype, f"call {call} vs the oracle")


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


def test_static_scratch_rejected_arguments_enqueue_nothing():
    """A call rejected for its arguments returns its status before anything
    is enqueued (the shared array is not cleared either, which matters when
    another call is still using it): the output and the flags stay
    untouched, and a valid call afterwards runs."""
    case = random_paged_case(77, [5, 40], H=4, KVH=2, D=64, bs=16, dtype=torch.bfloat16)
    q, kc, vc, tables, lens = [t.to(DEV) for t in (case["q"], case["k_cache"], case["v_cache"],
                                                   case["block_tables"], case["context_lens"])]
    fn = _static_fn()
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    base = [out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), tables.data_ptr(),
            lens.data_ptr(), 2, 4, 2, 64, 16, tables.shape[1], kc.shape[0], 0.1, 1, 0, 0,
            err.data_ptr(), torch.cuda.current_stream().cuda_stream]

    def call(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return fn(*a)

    assert call(a1=None) == 1                  # q NULL
    assert call(a1=q.data_ptr() + 1) == 1      # q not element-aligned
    assert call(a7=3) == 1                     # H not a multiple of KVH
    assert call(a6=70000) == 1                 # B beyond the grid's range
    assert call(a14=7) == 1                    # no such dtype
    assert call(a16=24) == 1                   # partition size not a multiple of 16
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all()) and int(err.item()) == 0
    assert call() == 0
    torch.cuda.synchronize()
    assert not bool(torch.isnan(out).any())
