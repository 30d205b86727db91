"""pkv_write_decode_attention (one decode step in one launch: write each
sequence's new token, then attend over contexts that count it) on the GPU.

The fused step is defined as write_kv followed by decode attention, so the
oracle is the oracle's write followed by the oracle's decode on CPU copies.
Caches must come out bit-identical to the oracle's writes; outputs within
the parity tolerance of the oracle, and bit-identical to the library's own
two-launch sequence (pkv_write, then pkv_decode_attention with the same
partition size)."""
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


def fused(q, k, v, slots, kc, vc, tables, lens, scale, partition_size=0, max_context_len=0,
          workspace=None, err=None):
    """Run the fused step on device tensors (kc / vc are written in place)."""
    B, H, D = q.shape
    nb, bs, kvh, _ = kc.shape
    out = torch.full_like(q, float("nan"))
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if workspace is None:
        workspace = pkv.DecodeWorkspace(B, H, kvh, D, bs, tables.shape[1], max_context_len,
                                        partition_size, device=DEV)
    pkv.pkv_write_decode_attention(out, q, k, v, slots, kc, vc, tables, lens, scale,
                                   max_context_len=max_context_len,
                                   partition_size=partition_size, workspace=workspace,
                                   err_flags=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def check_step(q, k, v, slots, kc, vc, tables, lens, scale, dtype, what, partition_size=0):
    """Fused step vs oracle write+decode and vs the library's two launches."""
    kc0, vc0 = kc.cpu(), vc.cpu()
    # oracle: write, then decode, on CPU copies
    kc_o, vc_o = kc0.clone(), vc0.clone()
    oracle.write(kc_o, vc_o, k.cpu(), v.cpu(), slots.cpu())
    want = oracle_decode(q, kc_o, vc_o, tables, lens, scale)
    # two launches
    kc2, vc2 = kc0.to(DEV), vc0.to(DEV)
    d = lambda t: t.to(DEV)
    pkv.pkv_write(kc2, vc2, d(k), d(v), d(slots))
    out2, err2 = gpu_decode(q, kc2, vc2, tables, lens, scale, partition_size=partition_size)
    assert err2 == 0
    # fused
    kcf, vcf = kc0.to(DEV), vc0.to(DEV)
    out, err = fused(d(q), d(k), d(v), d(slots), kcf, vcf, d(tables), d(lens), scale,
                     partition_size=partition_size)
    assert err == 0, f"{what}: flags {err:#x}"
    assert torch.equal(bits(kcf.cpu()), bits(kc_o)) and torch.equal(bits(vcf.cpu()), bits(vc_o)), \
        f"{what}: cache differs from the oracle's write"
    assert_close(out, want, dtype, what)
    assert torch.equal(bits(out.cpu()), bits(out2.cpu())), f"{what}: fused != write + decode"
    return out


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
    """Every workload's shapes: the new token is the last of each context
    (padded sequences: length 0, slot -1); unused cache rows are NaN."""
    cfg = SMALL[name]
    inp = wl.make_decode_inputs(cfg, seed=sum(map(ord, name)) + 5, poison_unused=True)
    lens = inp.context_lens
    positions = [int(n) - 1 if int(n) > 0 else None for n in lens]
    wb = wl.make_write_batch(inp, positions, seed=11)
    check_step(inp.q, wb.k, wb.v, wb.slot_mapping, inp.k_cache, inp.v_cache, inp.block_tables,
               lens, inp.scale, cfg.dtype, f"{name} P={partition_size}", partition_size)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [64, 128, 192, 256])
@pytest.mark.parametrize("H,KVH", [(8, 2), (16, 2), (48, 2)])
def test_tensor_core_shapes(dtype, D, H, KVH):
    """New token at every position of a 16-token chunk, on chunk and
    partition edges, GQA groups up to 24 heads (two CTAs per KV head read the
    new row)."""
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 64, 100]
    bs = 16 if D != 192 else 32
    case = random_paged_case(D * 3 + H + KVH, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    assert pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, case["block_tables"].shape[1],
                               dtype=dtype)[2] == 1
    g = torch.Generator().manual_seed(D + H)
    k = torch.randn((len(lens), KVH, D), generator=g).to(dtype)
    v = torch.randn((len(lens), KVH, D), generator=g).to(dtype)
    slots = torch.tensor([wl.slot_of(case["owned"][b], n - 1, bs) for b, n in enumerate(lens)])
    for ps in (0, 16, 32):
        check_step(case["q"], k, v, slots, case["k_cache"], case["v_cache"], case["block_tables"],
                   case["context_lens"], 1.0 / math.sqrt(D), dtype, f"D={D} H={H} KVH={KVH} P={ps}",
                   partition_size=ps)


@pytest.mark.parametrize("dtype,D,bs", [(torch.float32, 64, 16), (torch.float32, 128, 8),
                                        (torch.bfloat16, 96, 16), (torch.bfloat16, 128, 8),
                                        (torch.float16, 40, 5)])
def test_cuda_core_shapes(dtype, D, bs):
    lens = [1, 5, 8, 9, 40, 77]
    case = random_paged_case(D + bs, lens, H=6, KVH=2, D=D, bs=bs, dtype=dtype)
    assert pkv.pkv_decode_plan(len(lens), 6, 2, D, bs, case["block_tables"].shape[1],
                               dtype=dtype)[2] == 0
    g = torch.Generator().manual_seed(D * bs)
    k = torch.randn((len(lens), 2, D), generator=g).to(dtype)
    v = torch.randn((len(lens), 2, D), generator=g).to(dtype)
    slots = torch.tensor([wl.slot_of(case["owned"][b], n - 1, bs) for b, n in enumerate(lens)])
    for ps in (0, 16):
        check_step(case["q"], k, v, slots, case["k_cache"], case["v_cache"], case["block_tables"],
                   case["context_lens"], 0.2, dtype, f"{dtype} D={D} bs={bs} P={ps}",
                   partition_size=ps)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_sequences_without_a_new_token(dtype):
    """slot -1 with a non-empty context: nothing is written for that sequence
    and its output is plain decode attention over the cached rows."""
    lens = [20, 33, 1, 64]
    case = random_paged_case(5, lens, H=8, KVH=2, D=64, bs=16, dtype=dtype)
    g = torch.Generator().manual_seed(55)
    k = torch.randn((4, 2, 64), generator=g).to(dtype)
    v = torch.randn((4, 2, 64), generator=g).to(dtype)
    slots = torch.tensor([wl.slot_of(case["owned"][0], 19, 16), -1, -1,
                          wl.slot_of(case["owned"][3], 63, 16)])
    check_step(case["q"], k, v, slots, case["k_cache"], case["v_cache"], case["block_tables"],
               case["context_lens"], 0.125, dtype, "mixed")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_append_mismatch_is_flagged(dtype):
    """A kept slot that is not position n-1's: the token is still written
    where slot_mapping says, the flag is raised, other sequences are exact."""
    lens = [20, 33]
    case = random_paged_case(6, lens, H=4, KVH=2, D=64, bs=16, dtype=dtype, poison=False)
    q, kc, vc = case["q"].to(DEV), case["k_cache"].to(DEV), case["v_cache"].to(DEV)
    tables, lens_t = case["block_tables"].to(DEV), case["context_lens"].to(DEV)
    g = torch.Generator().manual_seed(66)
    k = torch.randn((2, 2, 64), generator=g).to(dtype).to(DEV)
    v = torch.randn((2, 2, 64), generator=g).to(dtype).to(DEV)
    good = wl.slot_of(case["owned"][1], 32, 16)
    wrong = wl.slot_of(case["owned"][0], 3, 16)  # inside sequence 0, not its last position
    slots = torch.tensor([wrong, good], device=DEV)
    out, err = fused(q, k, v, slots, kc, vc, tables, lens_t, 0.125)
    assert err == pkv.FLAG_APPEND_MISMATCH
    blk, off = divmod(wrong, 16)
    assert torch.equal(bits(kc[blk, off].cpu()), bits(k[0].cpu()))
    assert torch.equal(bits(vc[blk, off].cpu()), bits(v[0].cpu()))
    kc_o, vc_o = case["k_cache"].clone(), case["v_cache"].clone()
    oracle.write(kc_o, vc_o, k.cpu(), v.cpu(), slots.cpu())
    want = oracle_decode(case["q"], kc_o, vc_o, case["block_tables"], case["context_lens"], 0.125)
    assert_close(out[1:], want[1:], dtype, "the sequence with a matching slot")


def test_empty_context_with_a_slot_and_slot_past_pool():
    """Length 0 with a kept slot: written, flagged, output zero.  A slot past
    the pool: flagged, nothing written."""
    lens = [0, 17]
    case = random_paged_case(7, [1, 17], H=4, KVH=2, D=64, bs=16, dtype=torch.bfloat16, poison=False)
    q, kc, vc = case["q"].to(DEV), case["k_cache"].to(DEV), case["v_cache"].to(DEV)
    tables = case["block_tables"].to(DEV)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    g = torch.Generator().manual_seed(77)
    k = torch.randn((2, 2, 64), generator=g).to(torch.bfloat16).to(DEV)
    v = torch.randn((2, 2, 64), generator=g).to(torch.bfloat16).to(DEV)
    s0 = wl.slot_of(case["owned"][0], 0, 16)
    s1 = wl.slot_of(case["owned"][1], 16, 16)
    out, err = fused(q, k, v, torch.tensor([s0, s1], device=DEV), kc, vc, tables, lens_t, 0.125)
    assert err == pkv.FLAG_APPEND_MISMATCH
    assert bool((out[0] == 0).all())
    assert torch.equal(bits(kc[s0 // 16, s0 % 16].cpu()), bits(k[0].cpu()))
    nb = kc.shape[0]
    before = kc.clone()
    out, err = fused(q, k, v, torch.tensor([-1, nb * 16 + 3], device=DEV), kc, vc, tables,
                     lens_t, 0.125)
    assert err == pkv.FLAG_APPEND_MISMATCH | pkv.FLAG_SLOT_OUT_OF_RANGE
    assert torch.equal(bits(kc.cpu()), bits(before.cpu()))


def test_argument_errors():
    case = random_paged_case(8, [5, 9], H=4, KVH=2, D=64, bs=16, dtype=torch.bfloat16)
    q, kc, vc = case["q"].to(DEV), case["k_cache"].to(DEV), case["v_cache"].to(DEV)
    tables, lens = case["block_tables"].to(DEV), case["context_lens"].to(DEV)
    k = torch.zeros((2, 2, 64), dtype=torch.bfloat16, device=DEV)
    slots = torch.zeros(2, dtype=torch.int64, device=DEV)
    out = torch.empty_like(q)
    with pytest.raises(ValueError):  # k of the wrong shape
        pkv.pkv_write_decode_attention(out, q, k[:1], k[:1], slots, kc, vc, tables, lens, 0.1)
    lib = pkv.load_library()
    ws = pkv.DecodeWorkspace(2, 4, 2, 64, 16, tables.shape[1], device=DEV)
    base = dict(k=k.data_ptr(), ks=128, vs=128, slots=slots.data_ptr())

    def call(**kw):
        a = dict(base, **kw)
        return lib.pkv_write_decode_attention(
            out.data_ptr(), q.data_ptr(), a["k"], k.data_ptr(), a["ks"], a["vs"], a["slots"],
            kc.data_ptr(), vc.data_ptr(), tables.data_ptr(), lens.data_ptr(), 2, 4, 2, 64, 16,
            tables.shape[1], kc.shape[0], 0.1, 1, 0, 0, ws.buffer.data_ptr(),
            ws.buffer.numel(), None, None)

    assert call() == 0
    torch.cuda.synchronize()
    assert call(slots=None) == 1
    assert call(k=k.data_ptr() + 2) == 1   # row not 16-byte aligned
    assert call(ks=100) == 1               # stride shorter than a row
    assert call(ks=132) == 1               # stride not a multiple of 16 bytes


@pytest.mark.parametrize("name", ["step", "mqa"])
def test_step_loop_fused_in_cuda_graph(name):
    """The per-step loop with the fused launch: every step's launch captured
    in one CUDA graph (each step its own slice of device-resident step
    inputs), replayed once; caches and every step's output against the
    oracle's write-then-decode sequence.  "mqa" runs the wide-group kernel,
    which writes each new row to the cache and over row n - 1 of its landed
    tiles in the same launch: each step must see its own token and the next
    step its cache row (contexts up to 2500 tokens, so some are split and
    merged)."""
    cfg = (wl.small_variant(wl.CONFIGS["step_bf16"], B=16, len_hi=300, steps=6) if name == "step" else
           wl.small_variant(wl.CONFIGS["mqa_bf16"], B=12, len_hi=2500, steps=5))
    inp = wl.make_decode_inputs(cfg, seed=97)
    st = wl.make_steps(inp, seed=98)
    B, H, D = cfg.B, cfg.H, cfg.D
    kc, vc = inp.k_cache.to(DEV), inp.v_cache.to(DEV)
    d_k, d_v, d_slots, d_q = st.k.to(DEV), st.v.to(DEV), st.slots.to(DEV), st.q.to(DEV)
    d_tb, d_lens = st.tables.to(DEV), st.lens.to(DEV)
    outs = torch.empty((cfg.steps, B, H, D), dtype=cfg.dtype, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cap = cfg.table_width * cfg.bs
    ws = pkv.DecodeWorkspace(B, H, cfg.KVH, D, cfg.bs, cfg.table_width, cap, 0, device=DEV)
    kern = pkv.pkv_decode_plan(B, H, cfg.KVH, D, cfg.bs, cfg.table_width, cap, dtype=cfg.dtype)[2]
    assert kern == (2 if name == "mqa" else 1)

    def step(s):
        pkv.pkv_write_decode_attention(outs[s], d_q[s], d_k[s], d_v[s], d_slots[s], kc, vc,
                                       d_tb[s], d_lens[s], inp.scale, max_context_len=cap,
                                       workspace=ws, err_flags=err)

    # warm-up outside the capture (kernel attributes), on a throwaway cache
    kc_w, vc_w = kc.clone(), vc.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pkv.pkv_write_decode_attention(outs[0], d_q[0], d_k[0], d_v[0], d_slots[0], kc_w, vc_w,
                                       d_tb[0], d_lens[0], inp.scale, max_context_len=cap,
                                       workspace=ws, err_flags=err)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    del kc_w, vc_w
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(cfg.steps):
            step(s)
    g.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc_o, vc_o = inp.k_cache.clone(), inp.v_cache.clone()
    for s in range(cfg.steps):
        oracle.write(kc_o, vc_o, st.k[s], st.v[s], st.slots[s])
        want = oracle.decode(st.q[s], kc_o, vc_o, st.tables[s], st.lens[s], inp.scale)
        assert_close(outs[s], want, cfg.dtype, f"step {s}")
        assert bool((outs[s][B - cfg.pad_seqs:] == 0).all())
    assert torch.equal(kc.cpu(), kc_o) and torch.equal(vc.cpu(), vc_o)


@pytest.mark.parametrize("H,KVH,D,bs", [(16, 1, 128, 16), (32, 2, 256, 32), (16, 1, 128, 32)])
@pytest.mark.parametrize("partition_size", [0, 128, 256])
def test_wide_group_fused_step_edges(H, KVH, D, bs, partition_size):
    """The wide-group kernel's one-launch fused step (16 query heads per
    head chunk; 1 or 2 KV heads; block sizes 16 and 32): the new
    token at every edge of a 128-token tile and of a partition, against the
    oracle's write-then-decode and bit-identical to the two launches."""
    lens = [1, 2, 127, 128, 129, 255, 256, 257, 1000, 1024, 1025]
    case = random_paged_case(D + H + bs + partition_size, lens, H=H, KVH=KVH, D=D, bs=bs,
                             dtype=torch.bfloat16)
    assert pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, case["block_tables"].shape[1],
                               partition_size=partition_size)[2] == 2
    g = torch.Generator().manual_seed(D * H + bs)
    k = torch.randn((len(lens), KVH, D), generator=g).to(torch.bfloat16)
    v = torch.randn((len(lens), KVH, D), generator=g).to(torch.bfloat16)
    slots = torch.tensor([wl.slot_of(case["owned"][b], n - 1, bs) for b, n in enumerate(lens)])
    check_step(case["q"], k, v, slots, case["k_cache"], case["v_cache"], case["block_tables"],
               case["context_lens"], 1.0 / math.sqrt(D), torch.bfloat16,
               f"wide H={H} KVH={KVH} D={D} bs={bs} P={partition_size}", partition_size)


@pytest.mark.parametrize("H,KVH,D,bs", [(16, 1, 256, 32), (8, 2, 128, 16)])
def test_fused_step_odd_slots_and_cut_contexts(H, KVH, D, bs):
    """On the wide-group kernel (16 heads per KV head) and the TMA +
    mma.sync kernel: an empty context with a kept slot (written, flagged),
    a slot of -1 (nothing written), a slot that is not position n - 1
    (written where it says, flagged), and contexts longer than the host's
    bound (cut, flagged; their new rows still written).  The caches must
    equal the oracle's write bit for bit; the sequences with a regular
    append must match the oracle's decode."""
    lens = [0, 40, 300, 77, 900, 600]
    case = random_paged_case(H + D + 3, [max(n, 1) for n in lens], H=H, KVH=KVH, D=D, bs=bs,
                             dtype=torch.bfloat16, poison=False)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    g = torch.Generator().manual_seed(H + D)
    k = torch.randn((len(lens), KVH, D), generator=g).to(torch.bfloat16)
    v = torch.randn((len(lens), KVH, D), generator=g).to(torch.bfloat16)
    own = case["owned"]
    slots = torch.tensor([wl.slot_of(own[0], 0, bs),          # empty context, kept slot
                          -1,                                  # no new token
                          wl.slot_of(own[2], 299, bs),        # regular
                          wl.slot_of(own[3], 10, bs),         # not position n - 1
                          wl.slot_of(own[4], 899, bs),        # cut by the bound below
                          wl.slot_of(own[5], 599, bs)])       # regular
    hint = 640   # sequence 4 (900 tokens) is longer: cut
    kern = pkv.pkv_decode_plan(len(lens), H, KVH, D, bs, case["block_tables"].shape[1], hint)[2]
    assert kern == (2 if H // KVH == 16 else 1)
    kc, vc = case["k_cache"].to(DEV), case["v_cache"].to(DEV)
    d = lambda t: t.to(DEV)
    out, err = fused(d(case["q"]), d(k), d(v), d(slots), kc, vc, d(case["block_tables"]),
                     d(lens_t), 0.11, max_context_len=hint)
    assert err == pkv.FLAG_APPEND_MISMATCH | pkv.FLAG_CONTEXT_OVER_HINT, hex(err)
    kc_o, vc_o = case["k_cache"].clone(), case["v_cache"].clone()
    oracle.write(kc_o, vc_o, k, v, slots)
    assert torch.equal(bits(kc.cpu()), bits(kc_o)) and torch.equal(bits(vc.cpu()), bits(vc_o))
    want = oracle_decode(case["q"], kc_o, vc_o, case["block_tables"], lens_t, 0.11)
    for b in (1, 2, 5):
        assert_close(out[b], want[b], torch.bfloat16, f"sequence {b}")
    assert bool((out[0] == 0).all())


def test_prepared_call_matches_the_plain_call():
    """prepare_write_decode_attention: checked once, then each call enqueues
    the step on the same buffers; refilling the input tensors between calls
    gives each step's own result, equal to the plain call's bit for bit."""
    lens = [40, 1, 333, 128]
    case = random_paged_case(91, lens, H=8, KVH=2, D=128, bs=16, dtype=torch.bfloat16, poison=False)
    d = lambda t: t.to(DEV)
    q, tables, lens_t = d(case["q"]), d(case["block_tables"]), d(case["context_lens"])
    kc, vc = d(case["k_cache"]), d(case["v_cache"])
    kc2, vc2 = kc.clone(), vc.clone()
    g = torch.Generator().manual_seed(92)
    k = torch.empty((4, 2, 128), dtype=torch.bfloat16, device=DEV)
    v = torch.empty_like(k)
    slots = torch.tensor([wl.slot_of(case["owned"][b], n - 1, 16) for b, n in enumerate(lens)],
                         device=DEV)
    out = torch.empty_like(q)
    ws = pkv.DecodeWorkspace(4, 8, 2, 128, 16, tables.shape[1], device=DEV)
    ws2 = pkv.DecodeWorkspace(4, 8, 2, 128, 16, tables.shape[1], device=DEV)
    call = pkv.prepare_write_decode_attention(out, q, k, v, slots, kc, vc, tables, lens_t, 0.09,
                                              workspace=ws)
    for step in range(3):
        k.copy_(torch.randn((4, 2, 128), generator=g).to(torch.bfloat16))
        v.copy_(torch.randn((4, 2, 128), generator=g).to(torch.bfloat16))
        q.copy_(torch.randn((4, 8, 128), generator=g).to(torch.bfloat16))
        call()
        want = pkv.pkv_write_decode_attention(torch.empty_like(q), q, k, v, slots, kc2, vc2, tables,
                                              lens_t, 0.09, workspace=ws2)
        torch.cuda.synchronize()
        assert torch.equal(bits(out), bits(want)), f"step {step}"
        assert torch.equal(bits(kc), bits(kc2)) and torch.equal(bits(vc), bits(vc2))
    with pytest.raises(ValueError):  # checked at preparation
        pkv.prepare_write_decode_attention(out, q, k[:1], v, slots, kc, vc, tables, lens_t, 0.09,
                                           workspace=ws)


def test_staged_step_through_prepared_copies():
    """A serving loop's step from host memory: the inputs staged in one pinned
    host buffer go over in one pkv_copy_async into a device buffer whose
    views the prepared fused call reads, and the output comes back by a
    second copy into pinned host memory.  Each step's host result equals the
    device-only call's bit for bit, and the caches are written the same."""
    lens = [17, 200, 64, 1, 129]
    B, H, KVH, D, bs = 5, 8, 2, 128, 16
    case = random_paged_case(93, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=torch.bfloat16, poison=False)
    d = lambda t: t.to(DEV)
    kc, vc = d(case["k_cache"]), d(case["v_cache"])
    kc2, vc2 = kc.clone(), vc.clone()
    slots = torch.tensor([wl.slot_of(case["owned"][b], n - 1, bs) for b, n in enumerate(lens)])
    parts = {"q": case["q"], "k": torch.empty((B, KVH, D), dtype=torch.bfloat16),
             "v": torch.empty((B, KVH, D), dtype=torch.bfloat16), "slots": slots,
             "tables": case["block_tables"], "lens": case["context_lens"]}
    offs, off = {}, 0
    for name, t in parts.items():
        offs[name] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256

    def views(buf):
        return {n: buf[offs[n]:offs[n] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for n, t in parts.items()}

    h_in = torch.zeros(off, dtype=torch.uint8).pin_memory()
    d_in = torch.zeros(off, dtype=torch.uint8, device=DEV)
    hv, dv = views(h_in), views(d_in)
    out = torch.empty((B, H, D), dtype=torch.bfloat16, device=DEV)
    h_out = torch.empty((B, H, D), dtype=torch.bfloat16).pin_memory()
    ws = pkv.DecodeWorkspace(B, H, KVH, D, bs, case["block_tables"].shape[1], device=DEV)
    ws2 = pkv.DecodeWorkspace(B, H, KVH, D, bs, case["block_tables"].shape[1], device=DEV)
    stream = torch.cuda.Stream()
    copy_in = pkv.prepare_copy_async(d_in, h_in, stream=stream)
    step = pkv.prepare_write_decode_attention(out, dv["q"], dv["k"], dv["v"], dv["slots"], kc, vc,
                                              dv["tables"], dv["lens"], 0.09, workspace=ws,
                                              stream=stream)
    copy_out = pkv.prepare_copy_async(h_out, out, stream=stream)
    g = torch.Generator().manual_seed(94)
    for s in range(3):
        for n, t in parts.items():
            hv[n].copy_(t)
        hv["q"].copy_(torch.randn((B, H, D), generator=g).to(torch.bfloat16))
        hv["k"].copy_(torch.randn((B, KVH, D), generator=g).to(torch.bfloat16))
        hv["v"].copy_(torch.randn((B, KVH, D), generator=g).to(torch.bfloat16))
        copy_in()
        step()
        copy_out()
        stream.synchronize()
        want = pkv.pkv_write_decode_attention(torch.empty_like(out), d(hv["q"]), d(hv["k"]),
                                              d(hv["v"]), d(slots), kc2, vc2,
                                              d(case["block_tables"]), d(case["context_lens"]),
                                              0.09, workspace=ws2)
        torch.cuda.synchronize()
        assert torch.equal(bits(h_out), bits(want.cpu())), f"step {s}"
        assert torch.equal(bits(kc), bits(kc2)) and torch.equal(bits(vc), bits(vc2))
    # the same step with out in pinned host memory: no copy after the launch
    h_out2 = torch.empty_like(h_out).pin_memory()
    step2 = pkv.prepare_write_decode_attention(h_out2, dv["q"], dv["k"], dv["v"], dv["slots"], kc,
                                               vc, dv["tables"], dv["lens"], 0.09, workspace=ws,
                                               stream=stream)
    step2()
    stream.synchronize()
    assert torch.equal(bits(h_out2), bits(h_out))
    # device to device and pageable host memory go through the same call
    back = torch.empty(off, dtype=torch.uint8)
    d2 = torch.empty_like(d_in)
    pkv.pkv_copy_async(d2, d_in)
    pkv.pkv_copy_async(back, d2)
    torch.cuda.synchronize()
    assert torch.equal(back, h_in)
