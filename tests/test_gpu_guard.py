"""Guard bands around every buffer a kernel writes: each output (and each
cache a write targets) is a view into the middle of a larger allocation whose
4 KB on either side hold a sentinel pattern; after the launch the sentinels
must be bit-for-bit intact and the result must still match the oracle.  This
stands in for a memory checker on the stores the kernels make (vector stores
of whole output rows, merged rows, scattered cache rows).  Decode and
prefill must also leave the caches untouched."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from gpu_helpers import assert_close, bits, oracle_decode
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
GUARD = 4096          # bytes each side (keeps the view 16-byte aligned)
SENTINEL = 0xA5


class Guarded:
    """A device tensor of `shape` inside a sentinel-banded allocation."""

    def __init__(self, shape, dtype, init=None):
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.buf = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)
        assert self.t.data_ptr() % 16 == 0

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD] == SENTINEL).all()) and bool((self.buf[GUARD + self.n:] == SENTINEL).all())


def decode_case(seed, lens, H, KVH, D, bs, dtype):
    case = random_paged_case(seed, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    return case, 1.0 / math.sqrt(D)


@pytest.mark.parametrize("H,KVH,D,bs,dtype,kernel", [
    (8, 2, 128, 16, torch.bfloat16, 1),      # TMA + mma.sync
    (16, 1, 256, 32, torch.bfloat16, 2),     # wide-group tcgen05
    (32, 2, 128, 16, torch.float16, 2),      # wide-group, D = 128
    (6, 2, 64, 8, torch.float32, 0),         # CUDA-core
])
@pytest.mark.parametrize("partition_size", [0, 48, 128])
def test_decode_writes_only_its_output(H, KVH, D, bs, dtype, kernel, partition_size):
    lens = [1, 16, 17, 127, 128, 129, 300, 700, 1000, 0]
    case, scale = decode_case(D + H + partition_size, lens, H, KVH, D, bs, dtype)
    ps = partition_size
    assert pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, case["block_tables"].shape[1], 0, ps,
                               dtype=dtype)[2] == kernel
    q = case["q"].to(DEV)
    kc = Guarded(case["k_cache"].shape, dtype, case["k_cache"])
    vc = Guarded(case["v_cache"].shape, dtype, case["v_cache"])
    out = Guarded(q.shape, dtype)
    out.t.fill_(float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tables, clens = case["block_tables"].to(DEV), case["context_lens"].to(DEV)
    ws = pkv.DecodeWorkspace(len(lens), H, KVH, D, bs, tables.shape[1], 0, ps, device=DEV)
    pkv.pkv_decode_attention(out.t, q, kc.t, vc.t, tables, clens, scale, partition_size=ps,
                             workspace=ws, err_flags=err)
    assert out.intact() and kc.intact() and vc.intact(), "a store landed outside its buffer"
    assert int(err.item()) == 0
    assert torch.equal(bits(kc.t.cpu()), bits(case["k_cache"])), "decode wrote the K cache"
    assert torch.equal(bits(vc.t.cpu()), bits(case["v_cache"])), "decode wrote the V cache"
    want = oracle_decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                         case["context_lens"], scale)
    assert_close(out.t, want, dtype, f"kernel {kernel} P={ps}")


@pytest.mark.parametrize("KVH,D,dtype", [(2, 64, torch.float32), (8, 128, torch.bfloat16),
                                         (1, 256, torch.float16)])
def test_write_stays_in_the_cache(KVH, D, dtype):
    nb, bs = 9, 16
    g = torch.Generator().manual_seed(D + KVH)
    k0 = torch.randn((nb, bs, KVH, D), generator=g).to(dtype)
    v0 = torch.randn((nb, bs, KVH, D), generator=g).to(dtype)
    T = 40
    # distinct slots (one token per slot, as the write defines it), with the
    # pool's very last row (index 1) and very first (index 2) among them
    perm = torch.randperm(nb * bs, generator=g)
    rest = perm[(perm != 0) & (perm != nb * bs - 1)]
    slots = torch.cat([rest[:1], torch.tensor([nb * bs - 1, 0]), rest[1:T - 2]]).to(torch.int64)
    slots[::7] = -1                                    # padding (indices 0, 7, 14, ...)
    k = torch.randn((T, KVH, D), generator=g).to(dtype)
    v = torch.randn((T, KVH, D), generator=g).to(dtype)
    kc, vc = Guarded(k0.shape, dtype, k0), Guarded(v0.shape, dtype, v0)
    pkv.pkv_write(kc.t, vc.t, k.to(DEV), v.to(DEV), slots.to(DEV))
    assert kc.intact() and vc.intact(), "a cache row landed outside the pool"
    ko, vo = k0.clone(), v0.clone()
    oracle.write(ko, vo, k, v, slots)
    assert torch.equal(bits(kc.t.cpu()), bits(ko)) and torch.equal(bits(vc.t.cpu()), bits(vo))


@pytest.mark.parametrize("H,KVH,D,bs", [(8, 2, 128, 16), (16, 1, 256, 32)])
def test_fused_step_writes_only_its_output_and_rows(H, KVH, D, bs):
    dtype = torch.bfloat16
    lens = [1, 17, 129, 300, 1000]
    case, scale = decode_case(7 + H, lens, H, KVH, D, bs, dtype)
    n = case["context_lens"]
    g = torch.Generator().manual_seed(H + D)
    B = len(lens)
    slots = torch.tensor([int(case["block_tables"][b, (int(n[b]) - 1) // bs]) * bs + (int(n[b]) - 1) % bs
                          for b in range(B)], dtype=torch.int64)
    k = torch.randn((B, KVH, D), generator=g).to(dtype)
    v = torch.randn((B, KVH, D), generator=g).to(dtype)
    kc = Guarded(case["k_cache"].shape, dtype, case["k_cache"])
    vc = Guarded(case["v_cache"].shape, dtype, case["v_cache"])
    out = Guarded(case["q"].shape, dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    tables, clens = case["block_tables"].to(DEV), case["context_lens"].to(DEV)
    ws = pkv.DecodeWorkspace(B, H, KVH, D, bs, tables.shape[1], 0, 0, device=DEV)
    pkv.pkv_write_decode_attention(out.t, case["q"].to(DEV), k.to(DEV), v.to(DEV), slots.to(DEV),
                                   kc.t, vc.t, tables, clens, scale, workspace=ws, err_flags=err)
    assert out.intact() and kc.intact() and vc.intact(), "a store landed outside its buffer"
    assert int(err.item()) == 0
    ko, vo = case["k_cache"].clone(), case["v_cache"].clone()
    oracle.write(ko, vo, k, v, slots)
    assert torch.equal(bits(kc.t.cpu()), bits(ko)) and torch.equal(bits(vc.t.cpu()), bits(vo))
    assert_close(out.t, oracle_decode(case["q"], ko, vo, case["block_tables"], case["context_lens"], scale),
                 dtype, f"fused H={H} D={D}")


def test_prefill_writes_only_its_output():
    dtype, H, KVH, D, bs = torch.bfloat16, 8, 2, 128, 16
    lens, qlens = [300, 17, 1000, 129], [300, 5, 200, 1]
    case = random_paged_case(31, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    g = torch.Generator().manual_seed(32)
    cu = [0]
    for ql in qlens:
        cu.append(cu[-1] + ql)
    q = torch.randn((cu[-1], H, D), generator=g).to(dtype)
    cu = torch.tensor(cu, dtype=torch.int32)
    scale = 1.0 / math.sqrt(D)
    kc = Guarded(case["k_cache"].shape, dtype, case["k_cache"])
    vc = Guarded(case["v_cache"].shape, dtype, case["v_cache"])
    out = Guarded(q.shape, dtype)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_prefill_attention(out.t, q.to(DEV), kc.t, vc.t, case["block_tables"].to(DEV), cu.to(DEV),
                              case["context_lens"].to(DEV), scale, err_flags=err)
    assert out.intact() and kc.intact() and vc.intact(), "a store landed outside its buffer"
    assert int(err.item()) == 0
    assert torch.equal(bits(kc.t.cpu()), bits(case["k_cache"])) and \
        torch.equal(bits(vc.t.cpu()), bits(case["v_cache"])), "prefill wrote a cache"
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], scale)
    assert_close(out.t, want, dtype, "prefill")
