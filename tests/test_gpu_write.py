"""pkv_write on the GPU, bit-exact against the oracle."""
import json
import os

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from paged_kv_cache_67_gb300 import workloads as wl
from gpu_helpers import bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(kc, vc, k, v, slots, stream=None):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_write(kc, vc, k, v, slots, err_flags=err, stream=stream)
    torch.cuda.synchronize()
    return int(err.item())


def test_example1_write(golden_dir):
    with open(os.path.join(golden_dir, "example1_write.json")) as f:
        ex = json.load(f)
    kc = torch.zeros(ex["cache_shape"], device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.tensor(ex["k"], device=DEV).view(-1, 1, 1)
    v = k * ex["v_is_k_times"]
    ptr = kc.data_ptr()
    assert _run(kc, vc, k, v, torch.tensor(ex["slot_mapping"], device=DEV)) == 0
    assert kc.data_ptr() == ptr  # in place
    assert kc[:, :, 0, 0].cpu().tolist() == ex["expected_k_cache"]
    assert vc[:, :, 0, 0].cpu().tolist() == ex["expected_v_cache"]
    assert not (kc == 30.0).any() and not (vc == v[2, 0, 0]).any()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("KVH,D", [(1, 1), (2, 8), (8, 128), (1, 256), (3, 5), (4, 2)])
def test_random_write_bit_exact(dtype, KVH, D):
    g = torch.Generator().manual_seed(KVH * 1000 + D)
    nblk, bs = 37, 16
    cap = nblk * bs
    kc0 = torch.randn((nblk, bs, KVH, D), generator=g).to(dtype)
    vc0 = torch.randn((nblk, bs, KVH, D), generator=g).to(dtype)
    T = 300
    perm = torch.randperm(cap, generator=g)[:T]
    slots = perm.clone()
    pads = torch.rand(T, generator=g) < 0.2
    slots[pads] = -1
    slots[torch.rand(T, generator=g) < 0.05] = -987654321  # any negative is padding
    k = torch.randn((T, KVH, D), generator=g).to(dtype)
    v = torch.randn((T, KVH, D), generator=g).to(dtype)
    k[slots < 0] = wl.SENTINEL
    v[slots < 0] = wl.SENTINEL
    kc_o, vc_o = kc0.clone(), vc0.clone()
    oracle.write(kc_o, vc_o, k, v, slots)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    assert _run(kc, vc, k.to(DEV), v.to(DEV), slots.to(DEV)) == 0
    assert torch.equal(bits(kc.cpu()), bits(kc_o)) and torch.equal(bits(vc.cpu()), bits(vc_o))
    assert int((kc == wl.SENTINEL).sum()) == 0 and int((vc == wl.SENTINEL).sum()) == 0  # I1


def test_strided_tokens_and_stream():
    """k / v rows taken out of a wider per-token buffer (token stride >
    KVH*D, as a fused QKV projection gives), on a side stream."""
    g = torch.Generator().manual_seed(3)
    nblk, bs, KVH, D, T = 20, 16, 4, 64, 100
    qkv = torch.randn((T, 3 * KVH * D + 8), generator=g).to(torch.bfloat16)
    k = qkv[:, KVH * D: 2 * KVH * D].view(T, KVH, D)
    v = qkv[:, 2 * KVH * D + 8:].view(T, KVH, D)
    assert k.stride(0) == 3 * KVH * D + 8
    slots = torch.randperm(nblk * bs, generator=g)[:T]
    kc0 = torch.zeros((nblk, bs, KVH, D), dtype=torch.bfloat16)
    vc0 = torch.zeros_like(kc0)
    kc_o, vc_o = kc0.clone(), vc0.clone()
    oracle.write(kc_o, vc_o, k.contiguous(), v.contiguous(), slots)
    qkv_d = qkv.to(DEV)
    kd = qkv_d[:, KVH * D: 2 * KVH * D].view(T, KVH, D)
    vd = qkv_d[:, 2 * KVH * D + 8:].view(T, KVH, D)
    kc, vc = kc0.to(DEV), vc0.to(DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _run(kc, vc, kd, vd, slots.to(DEV), stream=s) == 0
    assert torch.equal(kc.cpu(), kc_o) and torch.equal(vc.cpu(), vc_o)


def test_slot_past_pool_is_flagged_and_skipped():
    kc = torch.zeros((4, 4, 1, 8), device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.arange(3 * 8, dtype=torch.float32, device=DEV).view(3, 1, 8) + 1
    slots = torch.tensor([2, 16, 5], device=DEV)  # 16 == num_blocks * bs
    assert _run(kc, vc, k, k.clone(), slots) == pkv.FLAG_SLOT_OUT_OF_RANGE
    flat = kc.view(-1, 1, 8)
    assert torch.equal(flat[2], k[0]) and torch.equal(flat[5], k[2])
    assert int((kc != 0).sum()) == 16


def test_zero_tokens_is_a_no_op():
    kc = torch.ones((2, 16, 1, 8), device=DEV)
    empty = torch.empty((0, 1, 8), device=DEV)
    assert _run(kc, kc.clone(), empty, empty, torch.empty(0, dtype=torch.int64, device=DEV)) == 0
    assert bool((kc == 1).all())


def test_bulk_fill_llama8b_full_size():
    """Every context token of the Llama-3-8B-shaped workload (~147k tokens,
    2 KB rows) written in a random order: the whole pool bit-exact."""
    cfg = wl.CONFIGS["llama8b_bf16"]
    inp = wl.make_decode_inputs(cfg, seed=1234, device="cuda")
    wb = wl.make_bulk_fill(inp, seed=5, device="cuda")
    kc_o, vc_o = inp.k_cache.cpu(), inp.v_cache.cpu()
    oracle.write(kc_o, vc_o, wb.k.cpu(), wb.v.cpu(), wb.slot_mapping.cpu())
    assert _run(inp.k_cache, inp.v_cache, wb.k, wb.v, wb.slot_mapping) == 0
    assert torch.equal(bits(inp.k_cache.cpu()), bits(kc_o))
    assert torch.equal(bits(inp.v_cache.cpu()), bits(vc_o))
