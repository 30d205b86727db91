"""The wide-group decode kernel (16 query heads per KV head, D = 128 or 256:
MQA and wide GQA) on the GPU against the oracle: lengths on and off the
128-token tile, the 16-token chunk and the partition edges, several
partitions per sequence (log-sum-exp merge), empty contexts, NaN in every
unused cache row, garbage table tails, back-to-back launches and graph
replays (the work counters reset themselves), and the full-size MQA batch
on sampled sequences."""
import math

import pytest
import torch

import paged_kv_cache_67_gb300 as pkv
from paged_kv_cache_67_gb300 import workloads as wl
from gpu_helpers import assert_close, gpu_decode, oracle_decode
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

LENS = [1, 15, 16, 17, 127, 128, 129, 255, 256, 300, 511, 512, 513, 700]


def case_args(seed, lens, H, KVH, D, bs, dtype):
    case = random_paged_case(seed, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    return case, (case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                  case["context_lens"], 1.0 / math.sqrt(D))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("H,KVH,bs", [(16, 1, 32), (32, 2, 16)])
def test_shapes_and_partitions(dtype, D, H, KVH, bs):
    case, args = case_args(D + H + bs, LENS, H, KVH, D, bs, dtype)
    assert pkv.pkv_decode_plan(len(LENS), H, KVH, D, bs, case["block_tables"].shape[1],
                               dtype=dtype)[2] == 2
    want = oracle_decode(*args)
    for ps in (0, 128, 256, 48, 16):
        out, err = gpu_decode(*args, partition_size=ps)
        assert err == 0, f"flags {err:#x}"
        assert_close(out, want, dtype, f"D={D} H={H} KVH={KVH} bs={bs} P={ps}")


def test_empty_contexts_and_short_tables():
    lens = [0, 5, 0, 130]
    case = random_paged_case(21, [1, 5, 1, 130], H=16, KVH=1, D=256, bs=32, dtype=torch.bfloat16)
    case["context_lens"] = torch.tensor(lens, dtype=torch.int32)
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"],
            0.0625)
    out, err = gpu_decode(*args)
    assert err == 0
    assert bool((out[0] == 0).all()) and bool((out[2] == 0).all())
    assert_close(out, oracle_decode(*args), torch.bfloat16, "empty contexts")


def test_bound_hint_and_bad_blocks_flagged():
    case, args = case_args(22, [40, 600], 16, 1, 128, 16, torch.bfloat16)
    # a host bound below a real length: flagged, the shorter sequence exact
    out, err = gpu_decode(*args, max_context_len=256, partition_size=128)
    assert err & pkv.FLAG_CONTEXT_OVER_HINT
    assert_close(out[:1], oracle_decode(*args)[:1], torch.bfloat16, "sequence within the bound")
    # a table entry outside the pool inside the context: flagged, no fault
    bad = case["block_tables"].clone()
    bad[1, 3] = case["k_cache"].shape[0] + 5
    out, err = gpu_decode(args[0], args[1], args[2], bad, args[4], args[5])
    assert err & pkv.FLAG_BLOCK_OUT_OF_RANGE


def test_many_items_per_cta():
    """About 900 work items (several per CTA of the persistent grid),
    contexts log-uniform like the MQA workload."""
    g = torch.Generator().manual_seed(23)
    lens = torch.exp(torch.rand(300, generator=g) * math.log(2048)).to(torch.int64).tolist()
    lens[:4] = [1, 2048, 512, 1024]
    case, args = case_args(23, lens, 16, 1, 128, 16, torch.bfloat16)
    out, err = gpu_decode(*args, partition_size=128)
    assert err == 0
    assert_close(out, oracle_decode(*args), torch.bfloat16, "many items")


def test_many_units_and_unsorted_claims():
    """300 sequences (more units than the claim search keeps in registers),
    and a partition size small enough that the claims fall back to unit
    order (more than 64 partitions per sequence)."""
    g = torch.Generator().manual_seed(25)
    lens = torch.randint(1, 1200, (300,), generator=g).tolist()
    lens[:3] = [1, 1199, 1024]
    case, args = case_args(25, lens, 16, 1, 128, 16, torch.bfloat16)
    want = oracle_decode(*args)
    out, err = gpu_decode(*args)
    assert err == 0
    assert_close(out, want, torch.bfloat16, "300 units")
    assert pkv.pkv_decode_plan(300, 16, 1, 128, 16, case["block_tables"].shape[1], 2048, 16)[1] > 64
    out, err = gpu_decode(*args, partition_size=16, max_context_len=2048)
    assert err == 0
    assert_close(out, want, torch.bfloat16, "unit-order claims")


def test_relaunch_and_graph_replay():
    case, args = case_args(24, [300, 17, 1000, 128], 16, 1, 256, 32, torch.bfloat16)
    want = oracle_decode(*args)
    d = [t.to(DEV) for t in args[:5]]
    ws = pkv.DecodeWorkspace(4, 16, 1, 256, 32, d[3].shape[1], 0, 256, device=DEV)
    for _ in range(3):
        out, err = gpu_decode(*d, args[5], partition_size=256, workspace=ws)
        assert err == 0
        assert_close(out, want, torch.bfloat16, "relaunch")
    out = torch.zeros_like(d[0])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        pkv.pkv_decode_attention(out, *d, args[5], partition_size=256, workspace=ws, err_flags=err,
                                 stream=side)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(out, want, torch.bfloat16, "graph replay")
