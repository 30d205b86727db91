"""Every decode workload at its full size, in the launch configuration
bench.py times (its inputs, its max_context_len, the automatic plan, the
fused write + decode step, the per-step loop replayed from one CUDA graph),
checked against the oracle on EVERY sequence and every head.

The bench's own helpers build the inputs and the context bound, so the test
and the timed run cannot drift apart.  Unused cache rows are NaN: a read of
any row outside a context shows in the output.  The course page "P09 · Paged
KV 写入 + decode attention（参考实现）" asks for exactly this check in its
section 自检 (random lengths, shuffled blocks, garbage table tails, compared
with dense attention); the oracle is that dense attention over the gathered
rows."""
import pytest
import torch

import bench
import oracle
import paged_kv_cache_67_gb300 as pkv
from paged_kv_cache_67_gb300 import workloads as wl
from gpu_helpers import assert_close, bits, gpu_decode, oracle_decode_parallel

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

# the kernel the plan must pick for each workload (1: TMA + mma.sync,
# 2: wide-group tcgen05, 0: CUDA-core)
EXPECTED_KERNEL = {"llama8b_bf16": 1, "long_bf16": 1, "mqa_bf16": 2, "tiny_fp32": 0}


@pytest.mark.parametrize("name", ["llama8b_bf16", "long_bf16", "mqa_bf16", "tiny_fp32"])
def test_single_step_workload_full_size(name):
    """One fused step (each sequence's new token at position n - 1 written,
    then attention over contexts that count it): the caches bit-exact
    against the oracle's write, every output row within tolerance of the
    oracle's decode, and (tensor-core workloads) bit-identical to the
    library's two-launch sequence."""
    cfg = wl.CONFIGS[name]
    elem = torch.empty((), dtype=cfg.dtype).element_size()
    inp = wl.make_decode_inputs(cfg, seed=1234, device=DEV, poison_unused=True)
    st = bench.make_step_inputs(cfg, inp, 0, DEV, elem)[0]
    max_ctx = bench.max_context(cfg)
    P, parts, kern = pkv.pkv_decode_plan(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width,
                                         max_ctx, dtype=cfg.dtype)
    assert kern == EXPECTED_KERNEL[name]
    if name == "long_bf16":
        assert parts > 1  # the partitioned path and its merge, at full size
    kc0, vc0 = inp.k_cache.cpu(), inp.v_cache.cpu()

    # the library: two launches (write, then decode) on copies, then the
    # fused step as the bench launches it
    kc2, vc2 = inp.k_cache.clone(), inp.v_cache.clone()
    pkv.pkv_write(kc2, vc2, st["k"], st["v"], st["slots"])
    out2, err2 = gpu_decode(st["q"], kc2, vc2, st["tables"], st["lens"], inp.scale,
                            max_context_len=max_ctx)
    assert err2 == 0
    del kc2, vc2
    ws = pkv.DecodeWorkspace(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width, max_ctx, 0,
                             device=DEV)
    out = torch.full_like(st["q"], float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_write_decode_attention(out, st["q"], st["k"], st["v"], st["slots"], inp.k_cache,
                                   inp.v_cache, st["tables"], st["lens"], inp.scale,
                                   max_context_len=max_ctx, workspace=ws, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # the oracle: write, then decode, on CPU copies
    kc_o, vc_o = kc0.clone(), vc0.clone()
    oracle.write(kc_o, vc_o, st["k"].cpu(), st["v"].cpu(), st["slots"].cpu())
    assert torch.equal(bits(inp.k_cache.cpu()), bits(kc_o)), "k cache differs from the oracle's write"
    assert torch.equal(bits(inp.v_cache.cpu()), bits(vc_o)), "v cache differs from the oracle's write"
    want = oracle_decode_parallel(st["q"], kc_o, vc_o, st["tables"], st["lens"], inp.scale)
    lens = st["lens"].cpu()
    for b in range(cfg.B):
        assert_close(out[b], want[b], cfg.dtype, f"{name} sequence {b} (n={int(lens[b])})")
    if kern != 2:
        # one launch or two: the same partitions, the same bits
        assert torch.equal(bits(out), bits(out2)), f"{name}: fused step != write + decode"
    else:
        assert_close(out2, want, cfg.dtype, f"{name}: write + decode")


def test_per_step_loop_full_size_in_cuda_graph():
    """The per-step workload (200 live sequences padded to 256, H = 64,
    contexts U[1, 2048], 32 steps of one appended token each) as the bench
    runs it: the 32 fused steps captured in one CUDA graph and replayed.
    After the replay the caches are bit-exact against the oracle's 32
    writes; the outputs of steps 0, 1, 16 and 31 match the oracle on every
    sequence, and every padded sequence's rows are exactly zero."""
    cfg = wl.CONFIGS["step_bf16"]
    elem = torch.empty((), dtype=cfg.dtype).element_size()
    inp = wl.make_decode_inputs(cfg, seed=1234, device=DEV, poison_unused=True)
    steps = bench.make_step_inputs(cfg, inp, 0, DEV, elem)
    assert len(steps) == cfg.steps == 32
    max_ctx = bench.max_context(cfg)
    assert pkv.pkv_decode_plan(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width, max_ctx,
                               dtype=cfg.dtype)[2] == 1
    kc0, vc0 = inp.k_cache.cpu(), inp.v_cache.cpu()
    ws = pkv.DecodeWorkspace(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width, max_ctx, 0,
                             device=DEV)
    outs = torch.full((cfg.steps, cfg.B, cfg.H, cfg.D), float("nan"), dtype=cfg.dtype, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step(s, kc, vc):
        t = steps[s]
        pkv.pkv_write_decode_attention(outs[s], t["q"], t["k"], t["v"], t["slots"], kc, vc,
                                       t["tables"], t["lens"], inp.scale, max_context_len=max_ctx,
                                       workspace=ws, err_flags=err)

    # one untimed launch outside the capture (kernel attributes), on a
    # throwaway copy of the caches
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    kc_w, vc_w = inp.k_cache.clone(), inp.v_cache.clone()
    with torch.cuda.stream(side):
        step(0, kc_w, vc_w)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    del kc_w, vc_w
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for s in range(cfg.steps):
            step(s, inp.k_cache, inp.v_cache)
    outs.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    kc_o, vc_o = kc0.clone(), vc0.clone()
    live = cfg.B - cfg.pad_seqs
    checked = (0, 1, 16, 31)
    for s in range(cfg.steps):
        t = steps[s]
        oracle.write(kc_o, vc_o, t["k"].cpu(), t["v"].cpu(), t["slots"].cpu())
        if s not in checked:
            continue
        want = oracle_decode_parallel(t["q"], kc_o, vc_o, t["tables"], t["lens"], inp.scale)
        got = outs[s].cpu()
        lens = t["lens"].cpu()
        for b in range(cfg.B):
            assert_close(got[b], want[b], cfg.dtype, f"step {s} sequence {b} (n={int(lens[b])})")
        assert bool((got[live:] == 0).all()), f"step {s}: a padded sequence's rows are not zero"
    assert torch.equal(bits(inp.k_cache.cpu()), bits(kc_o)), "k cache differs after 32 steps"
    assert torch.equal(bits(inp.v_cache.cpu()), bits(vc_o)), "v cache differs after 32 steps"
