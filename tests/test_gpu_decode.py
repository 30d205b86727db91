"""pkv_decode_attention on the GPU against the oracle (oracle-sized cases:
several tiles, ragged tails, both kernels, every config's shapes)."""
import json
import math
import os

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from paged_kv_cache_67_gb300 import workloads as wl
from gpu_helpers import assert_close, bits, gpu_decode, oracle_decode
from oracle_pins import random_paged_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def test_example2_on_gpu(golden_dir):
    with open(os.path.join(golden_dir, "example2_decode.json")) as f:
        ex = json.load(f)
    bs, nblk, KVH, D = ex["block_size"], ex["num_blocks"], ex["num_kv_heads"], ex["head_dim"]
    kc = torch.zeros((nblk, bs, KVH, D), device=DEV)
    vc = torch.zeros_like(kc)
    k = torch.tensor(ex["seq0_k"] + ex["seq1_k"], dtype=torch.float32, device=DEV).view(-1, KVH, D)
    v = torch.tensor(ex["seq0_v"] + ex["seq1_v"], dtype=torch.float32, device=DEV).view(-1, KVH, D)
    pkv.pkv_write(kc, vc, k, v, torch.tensor(ex["seq0_slots"] + ex["seq1_slots"], device=DEV))
    q = torch.tensor([ex["seq0_q"], [[0.3, -1.2], [5.0, 2.0]]], dtype=torch.float32)
    tables = torch.tensor(ex["block_tables"], dtype=torch.int32)
    lens = torch.tensor(ex["context_lens"], dtype=torch.int32)
    out, err = gpu_decode(q, kc, vc, tables, lens, ex["scale"])
    assert err == 0
    want = torch.tensor(ex["expected_out"], dtype=torch.float64)
    assert (out.cpu().double() - want).abs().max() <= 0.5e-4
    assert_close(out, oracle_decode(q, kc, vc, tables, lens, ex["scale"]), torch.float32)


SMALL = {
    "tiny_fp32": wl.CONFIGS["tiny_fp32"],
    "llama8b_small": wl.small_variant(wl.CONFIGS["llama8b_bf16"], B=6, len_hi=700),
    "long_small": wl.small_variant(wl.CONFIGS["long_bf16"], B=2, len_hi=3000),
    "mqa_small": wl.small_variant(wl.CONFIGS["mqa_bf16"], B=10, len_hi=700),
    "step_small": wl.small_variant(wl.CONFIGS["step_bf16"], B=12, len_hi=400),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("partition_size", [0, 16, 48, 256])
def test_configs_small(name, partition_size):
    """Each workload's shapes with NaN in every unused cache row (a read of
    one would show) and garbage table tails; split sizes from one 16-token
    chunk per partition to none."""
    cfg = SMALL[name]
    inp = wl.make_decode_inputs(cfg, seed=sum(map(ord, name)), poison_unused=True)
    args = (inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    out, err = gpu_decode(*args, partition_size=partition_size)
    assert err == 0
    assert_close(out, oracle_decode(*args), cfg.dtype, name)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128, 192, 256])
@pytest.mark.parametrize("H,KVH", [(4, 4), (8, 2), (16, 2), (32, 1), (48, 3)])
def test_tensor_core_shapes(dtype, D, H, KVH):
    """GQA groups of 1..32 heads (over 16: several CTAs per KV head; exactly 16
    at D = 128 / 256: the wide-group kernel)."""
    lens = [1, 15, 16, 17, 33, 64, 100, 250]
    bs = 16 if D != 192 else 32
    case = random_paged_case(D + H * 7 + KVH, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    P, _, kern = pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, case["block_tables"].shape[1],
                                     dtype=dtype)
    # groups of exactly 16 heads at D = 128 / 256 run on the wide-group
    # kernel, the others on the TMA + mma.sync kernel
    assert kern == (2 if H // KVH == 16 and D in (128, 256) else 1)
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"],
            1.0 / math.sqrt(D))
    for ps in (0, 32):
        out, err = gpu_decode(*args, partition_size=ps)
        assert err == 0
        assert_close(out, oracle_decode(*args), dtype, f"D={D} H={H} KVH={KVH} P={ps}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D,bs", [(1, 3), (2, 2), (40, 16), (96, 8), (128, 8), (320, 5), (512, 16)])
def test_cuda_core_shapes(dtype, D, bs):
    lens = [1, bs, bs + 1, 3 * bs, 77, 130]
    case = random_paged_case(D * 3 + bs, lens, H=6, KVH=2, D=D, bs=bs, dtype=dtype)
    assert pkv.pkv_decode_plan(len(lens), 6, 2, D, bs, case["block_tables"].shape[1], dtype=dtype)[2] == 0
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], 0.3)
    for ps in (0, 16, 64):
        out, err = gpu_decode(*args, partition_size=ps)
        assert err == 0
        assert_close(out, oracle_decode(*args), dtype, f"D={D} bs={bs} P={ps}")


def test_both_kernels_agree_on_bf16():
    """The same bf16 inputs through the tensor-core kernel (16-byte aligned)
    and the CUDA-core kernel (q and out offset by one element)."""
    case = random_paged_case(5, [3, 40, 200, 513], H=8, KVH=2, D=128, bs=16, dtype=torch.bfloat16)
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], 0.09)
    want = oracle_decode(*args)
    out_tc, err = gpu_decode(*args)
    assert err == 0
    qbuf = torch.zeros(case["q"].numel() + 1, dtype=torch.bfloat16, device=DEV)
    obuf = torch.full_like(qbuf, float("nan"))
    q_mis = qbuf[1:].view(case["q"].shape)
    q_mis.copy_(case["q"])
    out_mis = obuf[1:].view(case["q"].shape)
    out_simt, err = gpu_decode(q_mis, *args[1:], out=out_mis)
    assert err == 0
    assert_close(out_tc, want, torch.bfloat16, "tensor-core")
    assert_close(out_simt, want, torch.bfloat16, "cuda-core")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_edge_lengths(dtype):
    """Empty contexts (zero rows), one token, exact multiples of the block
    size, and a context filling the whole table."""
    bs, mb = 16, 6
    lens = [0, 1, 16, 32, 17, 0, mb * bs, 95]
    case = random_paged_case(8, lens, H=4, KVH=2, D=64, bs=bs, dtype=dtype)
    tables = torch.full((len(lens), mb), 99999, dtype=torch.int32)
    tables[:, : case["block_tables"].shape[1]] = case["block_tables"][:, :mb]
    args = (case["q"], case["k_cache"], case["v_cache"], tables, case["context_lens"], 0.2)
    for ps in (0, 16):
        out, err = gpu_decode(*args, partition_size=ps)
        assert err == 0
        assert_close(out, oracle_decode(*args), dtype)
        assert bool((out[0] == 0).all()) and bool((out[5] == 0).all())
    # a batch of only empty contexts
    z = torch.zeros(3, dtype=torch.int32)
    out, err = gpu_decode(case["q"][:3], case["k_cache"], case["v_cache"], tables[:3], z, 0.2)
    assert err == 0 and bool((out == 0).all())


def test_shared_prefix_blocks():
    case = random_paged_case(12, [100, 70, 129, 33], H=8, KVH=2, D=128, bs=16, dtype=torch.bfloat16,
                             share_prefix=3)
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], 0.1)
    out, err = gpu_decode(*args, partition_size=32)
    assert err == 0
    assert_close(out, oracle_decode(*args), torch.bfloat16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_error_flags(dtype):
    """Data-dependent contract violations are reported, not trapped."""
    case = random_paged_case(2, [20, 40, 5], H=4, KVH=2, D=64, bs=16, dtype=dtype, poison=False)
    q, kc, vc, tb, lens = (case[k] for k in ("q", "k_cache", "v_cache", "block_tables", "context_lens"))
    nblk = kc.shape[0]
    # an entry of the used prefix past the pool, and a negative one
    for bad in (nblk, 99999, -1):
        t2 = tb.clone()
        t2[1, 1] = bad
        _, err = gpu_decode(q, kc, vc, t2, lens, 0.2)
        assert err == pkv.FLAG_BLOCK_OUT_OF_RANGE
    # longer than the table
    l2 = lens.clone()
    l2[0] = tb.shape[1] * 16 + 1
    _, err = gpu_decode(q, kc, vc, tb, l2, 0.2)
    assert err & pkv.FLAG_CONTEXT_TOO_LONG
    # negative length: flagged and treated as empty
    l3 = lens.clone()
    l3[2] = -4
    out, err = gpu_decode(q, kc, vc, tb, l3, 0.2)
    assert err == pkv.FLAG_CONTEXT_NEGATIVE and bool((out[2] == 0).all())
    # longer than the host hint that sized the grid
    _, err = gpu_decode(q, kc, vc, tb, lens, 0.2, max_context_len=16, partition_size=16)
    assert err == pkv.FLAG_CONTEXT_OVER_HINT
    # the inputs that follow the contract raise nothing, and the workspace
    # is left clean for the next call
    _, err = gpu_decode(q, kc, vc, tb, lens, 0.2, max_context_len=40, partition_size=16)
    assert err == 0


def test_guard_bands_and_read_only_caches():
    """Nothing outside out is written; the caches are only read."""
    case = random_paged_case(6, [50, 1, 129], H=8, KVH=2, D=128, bs=16, dtype=torch.bfloat16, poison=False)
    q, kc, vc, tb, lens = (case[k] for k in ("q", "k_cache", "v_cache", "block_tables", "context_lens"))
    n = q.numel()
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[guard: guard + n].view(q.shape)
    kc_d, vc_d = kc.to(DEV), vc.to(DEV)
    out, err = gpu_decode(q, kc_d, vc_d, tb, lens, 0.1, partition_size=32, out=out)
    assert err == 0
    assert bool((buf[:guard] == 7).all()) and bool((buf[guard + n:] == 7).all())
    assert torch.equal(kc_d.cpu(), kc) and torch.equal(vc_d.cpu(), vc)
    assert_close(out, oracle_decode(q, kc, vc, tb, lens, 0.1), torch.bfloat16)


def test_workspace_reused_across_calls():
    """Counters return to zero, so one workspace serves call after call."""
    ws = pkv.DecodeWorkspace(4, 8, 2, 128, 16, 40, 0, 32, device=DEV)
    for seed in range(3):
        case = random_paged_case(40 + seed, [100, 600, 3, 257], H=8, KVH=2, D=128, bs=16,
                                 dtype=torch.bfloat16)
        tb = torch.full((4, 40), 99999, dtype=torch.int32)
        tb[:, : case["block_tables"].shape[1]] = case["block_tables"]
        args = (case["q"], case["k_cache"], case["v_cache"], tb, case["context_lens"], 0.1)
        out, err = gpu_decode(*args, partition_size=32, workspace=ws)
        assert err == 0
        assert_close(out, oracle_decode(*args), torch.bfloat16, f"call {seed}")
    assert int(ws.buffer[: 4 * 8 * 4].view(torch.int32).abs().sum()) == 0


def test_missing_or_short_workspace_is_an_error():
    case = random_paged_case(1, [300], H=4, KVH=2, D=128, bs=16, dtype=torch.bfloat16)
    args = [t.to(DEV) for t in (case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                case["context_lens"])]
    out = torch.empty_like(args[0])
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention(out, *args, 0.1, partition_size=64)
    assert e.value.status == 4
    short = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention(out, *args, 0.1, partition_size=64, workspace=short)
    assert e.value.status == 4


@pytest.mark.parametrize("lens", [
    [1] * 300,                                   # many one-chunk sequences
    [5000],                                      # one sequence split into many partitions
    [3],                                         # a single tiny sequence
    [0, 0, 0],                                   # no work at all: only zero rows
    [1, 2, 3, 16, 17, 4096, 33, 1000, 0, 15] * 3,
])
@pytest.mark.parametrize("partition_size", [0, 16, 160])
def test_work_distribution(lens, partition_size):
    """Ragged, tiny, single and empty workloads; automatic and explicit
    partition sizes (16 tokens: every chunk its own partition, most
    sequences merged from many partials); two calls on one workspace."""
    B = len(lens)
    case = random_paged_case(len(lens) + sum(lens) % 97, lens, H=8, KVH=2, D=128, bs=16,
                             dtype=torch.bfloat16, extra_blocks=1)
    assert pkv.pkv_decode_plan(B, 8, 2, 128, 16, case["block_tables"].shape[1])[2] == 1
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], 0.1)
    ws = pkv.DecodeWorkspace(B, 8, 2, 128, 16, case["block_tables"].shape[1], 0, partition_size,
                             device=DEV)
    want = oracle_decode(*args)
    for call in range(2):  # the merge counters reset themselves between calls
        out, err = gpu_decode(*args, partition_size=partition_size, workspace=ws)
        assert err == 0
        assert_close(out, want, torch.bfloat16, f"call {call}")
    assert int(ws.buffer[: B * 8 * 4].view(torch.int32).abs().sum()) == 0


def test_large_batch():
    """2100 short sequences in one call."""
    lens = [1 + (i * 37) % 200 for i in range(2100)]
    case = random_paged_case(9, lens, H=4, KVH=1, D=64, bs=16, dtype=torch.bfloat16, extra_blocks=1)
    assert pkv.pkv_decode_plan(len(lens), 4, 1, 64, 16, case["block_tables"].shape[1])[2] == 1
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], 0.125)
    want = oracle_decode(*args)
    for ps in (0, 48):
        out, err = gpu_decode(*args, partition_size=ps)
        assert err == 0
        assert_close(out, want, torch.bfloat16, f"P={ps}")


def test_step_loop_in_cuda_graph():
    """The per-step loop (padded batch, slot -1 pads with length 0, one new
    token per live sequence, then attend) captured once in a CUDA graph and
    replayed with each step's inputs copied into the static buffers."""
    cfg = wl.small_variant(wl.CONFIGS["step_bf16"], B=16, len_hi=300, steps=6)
    inp = wl.make_decode_inputs(cfg, seed=77)
    st = wl.make_steps(inp, seed=78)
    B, H, D = cfg.B, cfg.H, cfg.D
    kc, vc = inp.k_cache.to(DEV), inp.v_cache.to(DEV)
    s_k = torch.empty((B, cfg.KVH, D), dtype=cfg.dtype, device=DEV)
    s_v = torch.empty_like(s_k)
    s_slots = torch.empty(B, dtype=torch.int64, device=DEV)
    s_q = torch.empty((B, H, D), dtype=cfg.dtype, device=DEV)
    s_tb = torch.empty((B, cfg.table_width), dtype=torch.int32, device=DEV)
    s_lens = torch.empty(B, dtype=torch.int32, device=DEV)
    s_out = torch.empty_like(s_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cap = cfg.table_width * cfg.bs
    ws = pkv.DecodeWorkspace(B, H, cfg.KVH, D, cfg.bs, cfg.table_width, cap, 0, device=DEV)

    def load(s):
        s_k.copy_(st.k[s]); s_v.copy_(st.v[s]); s_slots.copy_(st.slots[s]); s_q.copy_(st.q[s])
        s_tb.copy_(st.tables[s]); s_lens.copy_(st.lens[s])

    def step():
        pkv.pkv_write(kc, vc, s_k, s_v, s_slots, err_flags=err)
        pkv.pkv_decode_attention(s_out, s_q, kc, vc, s_tb, s_lens, inp.scale, max_context_len=cap,
                                 workspace=ws, err_flags=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        load(0)
        step()  # warm-up outside the capture (sets kernel attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    # restore the cache (the warm-up wrote step 0's tokens; writes are idempotent anyway)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kc_o, vc_o = inp.k_cache.clone(), inp.v_cache.clone()
    for s in range(cfg.steps):
        load(s)
        g.replay()
        torch.cuda.synchronize()
        oracle.write(kc_o, vc_o, st.k[s], st.v[s], st.slots[s])
        want = oracle.decode(st.q[s], kc_o, vc_o, st.tables[s], st.lens[s], inp.scale)
        assert int(err.item()) == 0
        assert_close(s_out, want, cfg.dtype, f"step {s}")
        assert bool((s_out[B - cfg.pad_seqs:] == 0).all())  # padded sequences
    assert torch.equal(kc.cpu(), kc_o) and torch.equal(vc.cpu(), vc_o)
    assert int((kc == wl.SENTINEL).sum()) == 0  # I1 across the loop


def test_forced_kernels_agree_and_refuse_what_they_cannot_run():
    """pkv_decode_attention_with_kernel: the CUDA-core and the TMA +
    mma.sync kernels on the same bf16 batch both match the oracle (and the
    plan's choice, -1, is pkv_decode_attention itself); a kernel that cannot
    run the shape (the wide-group kernel at 4 heads per KV head, the
    tensor-core kernels on fp32) answers PKV_ERR_UNSUPPORTED."""
    lens = [1, 17, 300, 1000]
    case = random_paged_case(71, lens, H=8, KVH=2, D=128, bs=16, dtype=torch.bfloat16)
    d = [t.to(DEV) for t in (case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                             case["context_lens"])]
    want = oracle_decode(*[case[k] for k in ("q", "k_cache", "v_cache", "block_tables",
                                             "context_lens")], 0.1)
    ws = pkv.DecodeWorkspace(4, 8, 2, 128, 16, d[3].shape[1], device=DEV)
    outs = {}
    for kern in (pkv.KERNEL_AUTO, pkv.KERNEL_CUDA_CORE, pkv.KERNEL_TC):
        out = torch.full_like(d[0], float("nan"))
        pkv.pkv_decode_attention_with_kernel(out, *d, 0.1, kern, workspace=ws)
        torch.cuda.synchronize()
        assert_close(out, want, torch.bfloat16, f"kernel {kern}")
        outs[kern] = out
    plain, _ = gpu_decode(*d, 0.1)
    assert torch.equal(bits(outs[pkv.KERNEL_AUTO]), bits(plain))
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_with_kernel(torch.empty_like(d[0]), *d, 0.1, pkv.KERNEL_WIDE,
                                             workspace=ws)
    assert e.value.status == 2
    f = [t.float() if t.is_floating_point() else t for t in d]
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_with_kernel(torch.empty_like(f[0]), *f, 0.1, pkv.KERNEL_TC,
                                             workspace=ws)
    assert e.value.status == 2
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_with_kernel(torch.empty_like(d[0]), *d, 0.1, 7, workspace=ws)
    assert e.value.status == 1


@pytest.mark.parametrize("kernel,H,KVH,D,dtype", [
    (pkv.KERNEL_CUDA_CORE, 4, 2, 64, torch.float32),
    (pkv.KERNEL_TC, 8, 2, 128, torch.bfloat16),
    (pkv.KERNEL_WIDE, 16, 1, 128, torch.bfloat16),
])
def test_output_into_pinned_host_memory(kernel, H, KVH, D, dtype):
    """out may be pinned host memory: every decode kernel only stores to it,
    so the result lands on the host inside the launch.  Bit-identical to the
    same call into device memory, over one-partition, merged (partition 128)
    and empty contexts, on each kernel."""
    lens = [300, 0, 129, 5, 1000, 64]
    case = random_paged_case(71 + kernel, lens, H=H, KVH=KVH, D=D, bs=16, dtype=dtype)
    d = lambda t: t.to(DEV)
    args = (d(case["q"]), d(case["k_cache"]), d(case["v_cache"]), d(case["block_tables"]),
            d(case["context_lens"]), 0.11)
    for P in (0, 128):
        ws = pkv.DecodeWorkspace(len(lens), H, KVH, D, 16, case["block_tables"].shape[1], 0, P,
                                 device=DEV)
        want = torch.full((len(lens), H, D), float("nan"), dtype=dtype, device=DEV)
        pkv.pkv_decode_attention_with_kernel(want, *args, kernel=kernel, partition_size=P,
                                             workspace=ws)
        got = torch.full((len(lens), H, D), float("nan"), dtype=dtype).pin_memory()
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        pkv.pkv_decode_attention_with_kernel(got, *args, kernel=kernel, partition_size=P,
                                             workspace=ws, err_flags=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(bits(got), bits(want.cpu())), f"partition {P}"
        assert bool((got[1] == 0).all())
    with pytest.raises(ValueError):  # pageable host memory is refused
        pkv.pkv_decode_attention(torch.empty((len(lens), H, D), dtype=dtype), *args)
