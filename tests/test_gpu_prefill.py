"""pkv_prefill_attention (tcgen05 kernel) on the GPU against the oracle's
causal prefill: varlen queries that are the last tokens of each context,
whole-context prefills and chunks on top of a cached prefix, one query
(decode), lengths on and off the 128-token tile and 16-token chunk edges,
several query tiles per sequence, GQA groups, NaN in every unused cache
row and garbage table tails."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from gpu_helpers import assert_close
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def make_case(seed, lens, qlens, H, KVH, D, bs, dtype):
    case = random_paged_case(seed, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 17)
    cu = [0]
    for ql in qlens:
        cu.append(cu[-1] + ql)
    q = torch.randn((cu[-1], H, D), generator=g).to(dtype)
    return case, q, torch.tensor(cu, dtype=torch.int32)


def gpu_prefill(q, case, cu, scale, max_q_len=0, err=None):
    d = lambda t: t.to(DEV)
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device=DEV)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_prefill_attention(out, d(q), d(case["k_cache"]), d(case["v_cache"]),
                              d(case["block_tables"]), d(cu), d(case["context_lens"]), scale,
                              max_q_len=max_q_len, err_flags=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def check(seed, lens, qlens, H, KVH, D, bs, dtype, what):
    case, q, cu = make_case(seed, lens, qlens, H, KVH, D, bs, dtype)
    scale = 1.0 / math.sqrt(D)
    out, err = gpu_prefill(q, case, cu, scale)
    assert err == 0, f"{what}: flags {err:#x}"
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], scale)
    assert_close(out, want, dtype, what)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,KVH", [(2, 2), (8, 2), (8, 1)])
def test_shapes(dtype, D, H, KVH):
    lens = [1, 16, 17, 127, 128, 129, 200, 300]
    qlens = [1, 16, 5, 127, 1, 129, 70, 300]
    check(D + H * 3 + KVH, lens, qlens, H, KVH, D, 16, dtype, f"{dtype} D={D} H={H} KVH={KVH}")


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_block_sizes(bs):
    lens = [33, 250, 400]
    qlens = [33, 100, 7]
    check(bs, lens, qlens, 4, 2, 128, bs, torch.bfloat16, f"bs={bs}")


def test_many_query_tiles_and_long_cached_prefix():
    """Up to five 128-query tiles per sequence; chunks on top of 1-3k cached tokens."""
    lens = [600, 1500, 3000, 257]
    qlens = [600, 256, 129, 257]
    check(11, lens, qlens, 4, 1, 128, 16, torch.bfloat16, "long")


def test_qlen_one_matches_decode():
    """One query per sequence is decode: the prefill kernel and the decode
    kernel both match the oracle's decode on the same inputs."""
    lens = [5, 130, 1000, 64]
    case, q, cu = make_case(12, lens, [1] * 4, 8, 2, 128, 16, torch.bfloat16)
    out, err = gpu_prefill(q, case, cu, 0.1)
    assert err == 0
    want = oracle.decode(q, case["k_cache"], case["v_cache"], case["block_tables"],
                         case["context_lens"], 0.1)
    assert_close(out, want, torch.bfloat16, "qlen 1")


def test_empty_sequences_and_batch():
    lens = [0, 40, 0]
    qlens = [0, 40, 0]
    case, q, cu = make_case(13, [1, 40, 1], qlens, 4, 2, 64, 16, torch.bfloat16)
    case["context_lens"] = torch.tensor(lens, dtype=torch.int32)
    out, err = gpu_prefill(q, case, cu, 0.2)
    assert err == 0
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], 0.2)
    assert_close(out, want, torch.bfloat16, "empty sequences")
    # no queries at all: nothing to do
    empty = torch.zeros((0, 4, 64), dtype=torch.bfloat16, device=DEV)
    pkv.pkv_prefill_attention(empty, empty, case["k_cache"].to(DEV), case["v_cache"].to(DEV),
                              case["block_tables"].to(DEV), torch.zeros(4, dtype=torch.int32, device=DEV),
                              case["context_lens"].to(DEV), 0.2)


def test_error_flags_and_unsupported():
    case, q, cu = make_case(14, [10, 300], [10, 300], 2, 1, 64, 16, torch.bfloat16)
    # more queries than context: flagged, that sequence skipped, the other exact
    bad = dict(case)
    bad["context_lens"] = torch.tensor([5, 300], dtype=torch.int32)
    out, err = gpu_prefill(q, bad, cu, 0.3)
    assert err == pkv.FLAG_QUERY_LEN
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], 0.3, seqs=(1, 2))
    assert_close(out[10:], want[10:], torch.bfloat16, "good sequence")
    # a host hint smaller than a sequence's query count
    out, err = gpu_prefill(q, case, cu, 0.3, max_q_len=128)
    assert err == pkv.FLAG_QUERY_OVER_HINT
    # fp32 / other head sizes: not served by this kernel
    with pytest.raises(pkv.PkvError) as e:
        f = q.float().to(DEV)
        pkv.pkv_prefill_attention(torch.empty_like(f), f, case["k_cache"].float().to(DEV),
                                  case["v_cache"].float().to(DEV), case["block_tables"].to(DEV),
                                  cu.to(DEV), case["context_lens"].to(DEV), 0.3)
    assert e.value.status == 2


def test_persistent_many_items_per_cta():
    """Several hundred (head, sequence, 256-query) items, several per CTA of
    the persistent grid, varied lengths (whole prompts and chunks on cached
    prefixes) so that one CTA's items differ in shape."""
    g = torch.Generator().manual_seed(77)
    lens = torch.randint(1, 700, (24,), generator=g).tolist()
    qlens = [n if b % 3 else max(1, n // 3) for b, n in enumerate(lens)]
    check(77, lens, qlens, 16, 4, 64, 16, torch.bfloat16, "many items")


def test_claim_order_by_work_many_sequences():
    """40 sequences (the claim search runs over two 32-lane chunks), chunks
    on long cached prefixes mixed with whole prompts, so that items of one
    tile-count class come from many sequences."""
    g = torch.Generator().manual_seed(79)
    lens = torch.randint(64, 900, (40,), generator=g).tolist()
    qlens = [n if b % 2 else int(torch.randint(1, min(n, 300) + 1, (1,), generator=g)) for b, n in enumerate(lens)]
    check(79, lens, qlens, 8, 2, 64, 16, torch.bfloat16, "claim order by work")


def test_claim_order_fallback_for_large_batches():
    """More (sequence, tile) slots than the work-ordered claims cover (here
    300 sequences x 16 tiles of the host's bound): the plain order, exact."""
    g = torch.Generator().manual_seed(80)
    lens = torch.randint(1, 60, (300,), generator=g).tolist()
    qlens = [max(1, n // 2) for n in lens]
    case, q, cu = make_case(80, lens, qlens, 4, 2, 64, 16, torch.bfloat16)
    scale = 0.125
    out, err = gpu_prefill(q, case, cu, scale, max_q_len=4096)
    assert err == 0
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], scale)
    assert_close(out, want, torch.bfloat16, "fallback order")


def test_persistent_relaunch_and_graph_replay():
    """The work counters are taken back by each launch's last CTA: back-to-back
    launches and replays of one captured launch all give the oracle's result."""
    case, q, cu = make_case(78, [300, 17, 529, 256], [300, 1, 200, 256], 8, 2, 128, 16,
                            torch.bfloat16)
    scale = 0.09
    want = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                          case["context_lens"], scale)
    for _ in range(3):
        out, err = gpu_prefill(q, case, cu, scale)
        assert err == 0
        assert_close(out, want, torch.bfloat16, "relaunch")
    d = {k: case[k].to(DEV) for k in ("k_cache", "v_cache", "block_tables", "context_lens")}
    qd, cud = q.to(DEV), cu.to(DEV)
    out = torch.zeros_like(qd)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        pkv.pkv_prefill_attention(out, qd, d["k_cache"], d["v_cache"], d["block_tables"], cud,
                                  d["context_lens"], scale, err_flags=err, stream=side)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out, want, torch.bfloat16, "graph replay")


def test_full_size_llama8b_prefill_sampled():
    """An 8B-shaped varlen prefill batch at the bench's size: a sample of
    sequences against the oracle."""
    from paged_kv_cache_67_gb300 import workloads as wl
    cfg = wl.PREFILL_CONFIGS["prefill_bf16"]
    inp = wl.make_prefill_inputs(cfg, seed=1234, device=DEV)
    out = torch.empty_like(inp.q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_prefill_attention(out, inp.q, inp.k_cache, inp.v_cache, inp.block_tables.to(DEV),
                              inp.cu_seqlens_q.to(DEV), inp.context_lens.to(DEV), inp.scale,
                              max_q_len=inp.max_q_len, err_flags=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    q_c, kc, vc = inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu()
    # a chunked sequence whole, against the oracle's prefill
    b = 1
    want = oracle.prefill(q_c, kc, vc, inp.block_tables, inp.cu_seqlens_q, inp.context_lens,
                          inp.scale, seqs=(b, b + 1))
    r0, r1 = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
    assert_close(out[r0:r1], want[r0:r1], cfg.dtype, f"sequence {b}")
    # sampled rows of whole-prompt sequences: by definition the query at
    # position p is the oracle's decode over the first p + 1 tokens
    for b in (0, 2, cfg.B - 2):
        r0, r1 = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
        n = int(inp.context_lens[b])
        for i in (0, 1, 127, 128, (r1 - r0) // 2, r1 - r0 - 1):
            p = n - (r1 - r0) + i
            want = oracle.decode(q_c[r0 + i:r0 + i + 1], kc, vc, inp.block_tables[b:b + 1],
                                 torch.tensor([p + 1], dtype=torch.int32), inp.scale)
            assert_close(out[r0 + i:r0 + i + 1], want, cfg.dtype, f"sequence {b} row {i}")
