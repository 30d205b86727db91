"""Shared helpers for the GPU parity tests: run the library through its C ABI
binding and the oracle on CPU copies of the same tensors, and compare."""
from __future__ import annotations

import torch

import oracle
import paged_kv_cache_67_gb300 as pkv

# Parity bar: |gpu - oracle| <= tol + tol * |oracle| (bf16/fp16 1e-2, fp32 1e-5).
TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2, torch.float16: 1e-2}


def assert_close(got, want, dtype, what=""):
    got = got.detach().cpu().double()
    want = want.detach().cpu().double()
    tol = TOL[dtype]
    assert got.shape == want.shape, (got.shape, want.shape)
    nan_got, nan_want = torch.isnan(got), torch.isnan(want)
    assert torch.equal(nan_got, nan_want), f"{what}: NaN pattern differs ({int(nan_got.sum())} vs {int(nan_want.sum())})"
    err = (got - want).abs().nan_to_num(0.0)
    bad = err > tol + tol * want.abs().nan_to_num(0.0)
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements off, max err {err.max().item():.3e} "
                           f"at {tuple(int(i) for i in (err == err.max()).nonzero()[0])}")


def bits(t):
    t = t.contiguous()
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def gpu_decode(q, k_cache, v_cache, tables, lens, scale, partition_size=0, max_context_len=0,
               err=None, out=None, workspace=None, stream=None):
    """Run pkv_decode_attention on device copies; returns (out, err flags)."""
    dev = torch.device("cuda")
    B, H, D = q.shape
    nb, bs, kvh, _ = k_cache.shape
    d = lambda t: t if t.device.type == "cuda" else t.to(dev)
    q, k_cache, v_cache, tables, lens = map(d, (q, k_cache, v_cache, tables, lens))
    if out is None:
        out = torch.full_like(q, float("nan"))
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = pkv.DecodeWorkspace(B, H, kvh, D, bs, tables.shape[1], max_context_len,
                                        partition_size, device=dev)
    pkv.pkv_decode_attention(out, q, k_cache, v_cache, tables, lens, scale,
                             max_context_len=max_context_len, partition_size=partition_size,
                             workspace=workspace, err_flags=err, stream=stream)
    torch.cuda.synchronize()
    return out, int(err.item())


def oracle_decode(q, k_cache, v_cache, tables, lens, scale, seqs=None):
    c = lambda t: t.detach().cpu().contiguous()
    return oracle.decode(c(q), c(k_cache), c(v_cache), c(tables), c(lens), scale, seqs=seqs)


def oracle_decode_parallel(q, k_cache, v_cache, tables, lens, scale, seqs=None, threads=None):
    """The oracle's decode of the given sequences (all by default), one task
    per (sequence, KV head's query heads) on a thread pool (the oracle is C
    called through ctypes, which releases the GIL).  Rows of other sequences
    are zero."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    c = lambda t: t.detach().cpu().contiguous()
    q, k_cache, v_cache, tables, lens = map(c, (q, k_cache, v_cache, tables, lens))
    B, H, _ = q.shape
    kvh = k_cache.shape[2]
    G = H // kvh
    out = torch.zeros_like(q)
    seqs = range(B) if seqs is None else seqs
    tasks = [(b, g) for b in seqs for g in range(kvh)]
    lib = oracle.load()

    def one(task):
        b, g = task
        oracle.decode(q, k_cache, v_cache, tables, lens, scale, seqs=(b, b + 1),
                      heads=(g * G, (g + 1) * G), out=out, lib=lib)

    with ThreadPoolExecutor(max_workers=threads or max(1, min(os.cpu_count() or 1, 32))) as ex:
        list(ex.map(one, tasks))
    return out
