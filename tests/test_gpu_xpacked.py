"""The layout experiment on the GPU: vLLM's packed cache layout (K
[nb, KVH, D/8, 16, 8], V [nb, KVH, D, 16]) holds the same values as the
token-major caches, so the packed write must produce exactly the packed
image of the oracle's token-major write, and the packed decode must match the
oracle's decode of the token-major cache.  The packed image is the
permutation the layout defines, written out here with views."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from paged_kv_cache_67_gb300 import workloads as wl
from gpu_helpers import assert_close, bits, gpu_decode, oracle_decode
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def packed(kc, vc):
    """Token-major [nb, 16, KVH, D] caches -> packed images."""
    nb, bs, kvh, d = kc.shape
    kx = kc.view(nb, bs, kvh, d // 8, 8).permute(0, 2, 3, 1, 4).contiguous()
    vx = vc.permute(0, 2, 3, 1).contiguous()
    return kx, vx


def decode_x(q, kx, vx, tables, lens, scale, partition_size=0, max_context_len=0):
    d = lambda t: t.to(DEV)
    B, H, D = q.shape
    nb, kvh = kx.shape[0], kx.shape[1]
    out = torch.full((B, H, D), float("nan"), dtype=q.dtype, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = pkv.DecodeWorkspace(B, H, kvh, D, 16, tables.shape[1], max_context_len, partition_size,
                             device=DEV)
    pkv.pkv_decode_attention_xpacked(out, d(q), d(kx), d(vx), d(tables), d(lens), scale,
                                     max_context_len=max_context_len, partition_size=partition_size,
                                     workspace=ws, err_flags=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("KVH,D", [(2, 64), (8, 128), (1, 256)])
def test_packed_write_bit_exact(dtype, KVH, D):
    nb, T = 40, 300
    g = torch.Generator().manual_seed(D + KVH)
    kc = torch.randn((nb, 16, KVH, D), generator=g).to(dtype)
    vc = torch.randn((nb, 16, KVH, D), generator=g).to(dtype)
    k = torch.randn((T, KVH, D), generator=g).to(dtype)
    v = torch.randn((T, KVH, D), generator=g).to(dtype)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                                   # padding tokens
    kx, vx = packed(kc, vc)
    kx, vx = kx.to(DEV), vx.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_write_xpacked(kx, vx, k.to(DEV), v.to(DEV), slots.to(DEV), err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc_o, vc_o = kc.clone(), vc.clone()
    oracle.write(kc_o, vc_o, k, v, slots)
    kx_o, vx_o = packed(kc_o, vc_o)
    assert torch.equal(bits(kx.cpu()), bits(kx_o)) and torch.equal(bits(vx.cpu()), bits(vx_o))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("H,KVH", [(8, 2), (16, 1), (32, 1)])
def test_packed_decode_matches_oracle(dtype, D, H, KVH):
    lens = [1, 15, 16, 17, 64, 100, 250]
    case = random_paged_case(D + H + KVH, lens, H=H, KVH=KVH, D=D, bs=16, dtype=dtype)
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"],
            1.0 / math.sqrt(D))
    want = oracle_decode(*args)
    kx, vx = packed(case["k_cache"], case["v_cache"])
    for ps in (0, 32):
        out, err = decode_x(case["q"], kx, vx, case["block_tables"], case["context_lens"],
                            1.0 / math.sqrt(D), partition_size=ps)
        assert err == 0
        assert_close(out, want, dtype, f"packed D={D} H={H} KVH={KVH} P={ps}")


@pytest.mark.parametrize("name", ["llama8b_bf16", "long_bf16"])
def test_packed_workloads_small(name):
    cfg = wl.small_variant(wl.CONFIGS[name], B=4, len_hi=1500)
    inp = wl.make_decode_inputs(cfg, seed=31, poison_unused=True)
    args = (inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    want = oracle_decode(*args)
    kx, vx = packed(inp.k_cache, inp.v_cache)
    out, err = decode_x(inp.q, kx, vx, inp.block_tables, inp.context_lens, inp.scale)
    assert err == 0
    assert_close(out, want, cfg.dtype, name)
    # and against the token-major kernel on the same data
    ref, err = gpu_decode(*args)
    assert err == 0
    assert_close(out, ref.cpu().double(), cfg.dtype, f"{name} vs token-major")


def test_packed_unsupported_shapes():
    q = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device=DEV)
    kx = torch.zeros((4, 2, 8, 16, 8), dtype=torch.bfloat16, device=DEV)
    vx = torch.zeros((4, 2, 64, 16), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((2, 2), dtype=torch.int32, device=DEV)
    lens = torch.ones(2, dtype=torch.int32, device=DEV)
    ws = pkv.DecodeWorkspace(2, 4, 2, 64, 16, 2, device=DEV)
    out = torch.empty_like(q)
    pkv.pkv_decode_attention_xpacked(out, q, kx, vx, tables, lens, 0.1, workspace=ws)
    with pytest.raises(pkv.PkvError) as e:
        f = q.float()
        pkv.pkv_decode_attention_xpacked(torch.empty_like(f), f, kx.float(), vx.float(), tables, lens,
                                         0.1, workspace=ws)
    assert e.value.status == 2
