"""Pins for the oracle: checks against what the pages and the mathematics fix.

Every ``pin_*`` function takes a loaded oracle library (the real one, or a
copy with a planted mistake) and raises AssertionError (or OracleError) when
the oracle disagrees with:
  - the values the course page "P09 · Paged KV 写入 + decode attention
    （参考实现）" prints for its worked examples 1-3 and its key answers
    (fixtures under tests/golden/, each with its citation);
  - the invariants I1-I5 of that page (section 不变量);
  - dense softmax attention computed by a library routine
    (torch.nn.functional.scaled_dot_product_attention, float64, CPU) on
    contiguous K/V built before they are scattered into the pool -- the
    page's own self-check (section 自检) and the interview note's claim that
    paged and dense attention agree (section 直接答案);
  - closed forms (one token, zero query, constant V, zero / huge scale);
  - IEEE round-to-nearest-even, against torch's float32->bf16/fp16
    conversion where no double rounding is possible, and hand-worked ties.
None of these re-types the oracle's formula.
"""
from __future__ import annotations

import json
import math
import os

import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# ----------------------------------------------------------------- helpers

def scatter_dense(dense_k, dense_v, owned, pool_k, pool_v, bs):
    """Place a sequence's contiguous rows into its physical blocks (test side,
    plain loop: logical token t -> block owned[t // bs], row t % bs)."""
    for t in range(dense_k.shape[0]):
        pool_k[owned[t // bs], t % bs] = dense_k[t]
        pool_v[owned[t // bs], t % bs] = dense_v[t]


def dense_attention(q, k, v, scale):
    """q [H, D], k/v [n, KVH, D] -> [H, D] float64 via SDPA with GQA."""
    q64 = q.double().view(1, q.shape[0], 1, q.shape[1])
    k64 = k.double().permute(1, 0, 2).unsqueeze(0)
    v64 = v.double().permute(1, 0, 2).unsqueeze(0)
    o = F.scaled_dot_product_attention(q64, k64, v64, scale=scale,
                                       enable_gqa=k64.shape[1] != q64.shape[1])
    return o.view(q.shape[0], q.shape[1])


def random_paged_case(seed, lens, H, KVH, D, bs, dtype, extra_blocks=3, tail=99999,
                      poison=True, share_prefix=0):
    """Dense per-sequence K/V first, then a shuffled scatter into a pool.

    Unused rows are NaN when ``poison`` (any read of them shows).  With
    ``share_prefix`` > 0 every sequence reuses the first ``share_prefix``
    physical blocks of sequence 0 (prefix caching), and its rows there are
    sequence 0's rows."""
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    nbs = [-(-n // bs) for n in lens]
    total = sum(nbs) + extra_blocks
    perm = torch.randperm(total, generator=g).tolist()
    fill = float("nan") if poison else 0.0
    pool_k = torch.full((total, bs, KVH, D), fill, dtype=torch.float64)
    pool_v = torch.full((total, bs, KVH, D), fill, dtype=torch.float64)
    width = max(nbs) + 2
    tables = torch.full((B, width), tail, dtype=torch.int32)
    dense, owned_all, cursor = [], [], 0
    for b, n in enumerate(lens):
        dk = torch.randn((n, KVH, D), generator=g, dtype=torch.float64)
        dv = torch.randn((n, KVH, D), generator=g, dtype=torch.float64)
        owned = perm[cursor:cursor + nbs[b]]
        cursor += nbs[b]
        if share_prefix and b > 0:
            k0, v0, own0 = dense[0][0], dense[0][1], owned_all[0]
            sp = min(share_prefix, nbs[b], len(own0))
            rows = min(sp * bs, k0.shape[0], n)
            dk[:rows], dv[:rows] = k0[:rows], v0[:rows]
            owned = own0[:sp] + owned[sp:]
        dense.append((dk, dv))
        owned_all.append(owned)
        tables[b, :nbs[b]] = torch.tensor(owned, dtype=torch.int32)
    for b in range(B):
        scatter_dense(dense[b][0], dense[b][1], owned_all[b], pool_k, pool_v, bs)
    q = torch.randn((B, H, D), generator=g, dtype=torch.float64)
    # round every value to the working dtype once; dense copies see the same values
    to = lambda t: t.to(dtype)
    case = dict(q=to(q), k_cache=to(pool_k), v_cache=to(pool_v), block_tables=tables,
                context_lens=torch.tensor(lens, dtype=torch.int32),
                dense=[(to(a), to(b)) for a, b in dense], owned=owned_all)
    return case


def _bits(t):
    return t.contiguous().view(torch.int32 if t.element_size() == 4 else torch.int16)


def _assert_close(got, want, atol, rtol, what):
    got, want = got.double(), want.double()
    err = (got - want).abs()
    bad = err > atol + rtol * want.abs()
    assert not torch.isnan(got).any(), f"{what}: NaN in result"
    assert not bad.any(), f"{what}: max err {err.max().item():.3e}"


# ------------------------------------------------------------------- pins

def pin_example1_write(lib):
    ex = _golden("example1_write.json")
    shape = ex["cache_shape"]
    kc = torch.zeros(shape, dtype=torch.float32)
    vc = torch.zeros(shape, dtype=torch.float32)
    k = torch.tensor(ex["k"], dtype=torch.float32).view(-1, 1, 1)
    v = k * ex["v_is_k_times"]
    slots = torch.tensor(ex["slot_mapping"], dtype=torch.int64)
    oracle.write(kc, vc, k, v, slots, lib=lib)
    assert torch.equal(kc[:, :, 0, 0], torch.tensor(ex["expected_k_cache"])), kc[:, :, 0, 0]
    assert torch.equal(vc[:, :, 0, 0], torch.tensor(ex["expected_v_cache"])), vc[:, :, 0, 0]
    assert not (kc == ex["absent_values"]["k"]).any()
    assert not (vc == v[2, 0, 0]).any()


def pin_key_answer_slot7(lib):
    a = _golden("key_answers.json")["slot7"]
    bs = a["block_size"]
    kc = torch.zeros((3, bs, 1, 2), dtype=torch.float32)
    vc = torch.zeros_like(kc)
    k = torch.tensor([[[5.0, 6.0]]])
    oracle.write(kc, vc, k, k.clone(), torch.tensor([a["slot"]]), lib=lib)
    nz = (kc != 0).any(dim=-1).any(dim=-1).nonzero().tolist()
    assert nz == [[a["block"], a["offset"]]], nz
    # the flattened view indexes the same row by the slot itself
    assert torch.equal(kc.view(-1, 1, 2)[a["slot"]], k[0])


def pin_I1_sentinel(lib):
    """Padding tokens (every element 9.0, slot -1) appear nowhere; every other
    token lands bit-exactly at cache[slot // bs, slot % bs]."""
    g = torch.Generator().manual_seed(11)
    for dtype in (torch.float32, torch.bfloat16, torch.float16):
        nblk, bs, KVH, D = 6, 4, 2, 8
        kc = torch.randn((nblk, bs, KVH, D), generator=g).to(dtype)
        vc = torch.randn((nblk, bs, KVH, D), generator=g).to(dtype)
        before_k, before_v = kc.clone(), vc.clone()
        slots = torch.tensor([3, -1, 23, 0, -1, 9, -7], dtype=torch.int64)
        k = torch.randn((7, KVH, D), generator=g).to(dtype)
        v = torch.randn((7, KVH, D), generator=g).to(dtype)
        k[slots < 0] = 9.0
        v[slots < 0] = 9.0
        oracle.write(kc, vc, k, v, slots, lib=lib)
        assert int((kc == 9).sum()) == 0 and int((vc == 9).sum()) == 0
        for i, s in enumerate(slots.tolist()):
            if s >= 0:
                assert torch.equal(_bits(kc[s // bs, s % bs]), _bits(k[i]))
                assert torch.equal(_bits(vc[s // bs, s % bs]), _bits(v[i]))
        written = {s for s in slots.tolist() if s >= 0}
        for s in range(nblk * bs):
            if s not in written:
                assert torch.equal(kc[s // bs, s % bs], before_k[s // bs, s % bs])
                assert torch.equal(vc[s // bs, s % bs], before_v[s // bs, s % bs])


def _example2_cache(ex, lib, dtype=torch.float32):
    bs, nblk, KVH, D = ex["block_size"], ex["num_blocks"], ex["num_kv_heads"], ex["head_dim"]
    kc = torch.zeros((nblk, bs, KVH, D), dtype=dtype)
    vc = torch.zeros_like(kc)
    k = torch.tensor(ex["seq0_k"] + ex["seq1_k"], dtype=dtype).view(-1, KVH, D)
    v = torch.tensor(ex["seq0_v"] + ex["seq1_v"], dtype=dtype).view(-1, KVH, D)
    slots = torch.tensor(ex["seq0_slots"] + ex["seq1_slots"], dtype=torch.int64)
    oracle.write(kc, vc, k, v, slots, lib=lib)
    return kc, vc


def pin_example2_decode(lib):
    ex = _golden("example2_decode.json")
    kc, vc = _example2_cache(ex, lib)
    # the gather of sequence 0 before truncation, as the page draws it
    tbl0 = ex["block_tables"][0]
    gathered = kc[torch.tensor(tbl0)].reshape(-1, ex["head_dim"])
    assert gathered.tolist() == ex["expected_gather_before_truncation_seq0"]
    g = torch.Generator().manual_seed(5)
    for trial in range(3):
        q1 = torch.randn((ex["num_heads"], ex["head_dim"]), generator=g) * (trial + 1)
        q = torch.stack([torch.tensor(ex["seq0_q"], dtype=torch.float32), q1])
        out = oracle.decode(q, kc, vc, torch.tensor(ex["block_tables"], dtype=torch.int32),
                            torch.tensor(ex["context_lens"], dtype=torch.int32), ex["scale"], lib=lib)
        want = torch.tensor(ex["expected_out"], dtype=torch.float64)
        tol = 0.5 * 10 ** -ex["expected_out_decimals"]
        assert (out.double() - want).abs().max() <= tol, out


def pin_example2_softmax(lib):
    """The page's intermediate softmax rows: same keys and queries, with the
    value rows replaced by one-hot vectors, so that out = the weights."""
    ex = _golden("example2_decode.json")
    bs = ex["block_size"]
    D = 4
    keys = torch.zeros((3, 1, D))
    keys[:, 0, :2] = torch.tensor(ex["seq0_k"], dtype=torch.float32)
    vals = torch.zeros((3, 1, D))
    for t in range(3):
        vals[t, 0, t] = 1.0
    kc = torch.zeros((ex["num_blocks"], bs, 1, D))
    vc = torch.zeros_like(kc)
    oracle.write(kc, vc, keys, vals, torch.tensor(ex["seq0_slots"]), lib=lib)
    q = torch.zeros((1, 2, D))
    q[0, :, :2] = torch.tensor(ex["seq0_q"], dtype=torch.float32)
    out = oracle.decode(q, kc, vc, torch.tensor([ex["block_tables"][0]], dtype=torch.int32),
                        torch.tensor([3], dtype=torch.int32), ex["scale"], lib=lib)
    want = torch.tensor(ex["expected_softmax_seq0"], dtype=torch.float64)
    assert (out[0, :, :3].double() - want).abs().max() <= 0.5e-4, out
    assert torch.equal(out[0, :, 3], torch.zeros(2))


def pin_key_answer_n5_truncation(lib):
    """context_len 5 with bs 4: two table entries, 8 positions, 3 dropped.
    The 3 dropped rows hold NaN; the third table entry is garbage."""
    a = _golden("key_answers.json")["n5"]
    bs, n = a["block_size"], a["context_len"]
    case = random_paged_case(3, [n], H=2, KVH=1, D=8, bs=bs, dtype=torch.float32)
    tbl = case["block_tables"]
    assert (tbl[0] != 99999).sum().item() == a["entries"]
    assert a["entries"] * bs == a["positions"] and a["positions"] - n == a["truncated"]
    out = oracle.decode(case["q"], case["k_cache"], case["v_cache"], tbl,
                        case["context_lens"], 0.35, lib=lib)
    want = dense_attention(case["q"][0], *case["dense"][0], 0.35)
    _assert_close(out[0], want, 1e-6, 1e-6, "n=5 bs=4")


def pin_gqa_mapping(lib):
    """Examples 3 and I5: query head h reads KV head h // (H / KVH).  Each KV
    head's V rows are a distinct constant, so out[h] names the head read."""
    ans = _golden("key_answers.json")
    for key in ("gqa8", "gqa4"):
        H, KVH = ans[key]["H"], ans[key]["KVH"]
        D, bs, n = 4, 2, 5
        nblk = 3
        g = torch.Generator().manual_seed(H)
        kc = torch.randn((nblk, bs, KVH, D), generator=g)
        vc = torch.empty((nblk, bs, KVH, D))
        for j in range(KVH):
            vc[:, :, j, :] = float(10 + j)
        q = torch.randn((1, H, D), generator=g)
        out = oracle.decode(q, kc, vc, torch.tensor([[2, 0, 1]], dtype=torch.int32),
                            torch.tensor([n], dtype=torch.int32), 0.5, lib=lib)
        heads = [int(round(out[0, h, 0].item())) - 10 for h in range(H)]
        assert heads == ans[key]["kv_head_of"], heads


def pin_I2_tail_never_read(lib):
    """Tail entries 99999 (and negative garbage) give the same result as a
    tail of valid indices; only ceil(n/bs) entries are read."""
    case = random_paged_case(21, [7, 1, 16, 9], H=4, KVH=2, D=8, bs=4, dtype=torch.float32)
    args = (case["q"], case["k_cache"], case["v_cache"])
    out1 = oracle.decode(*args, case["block_tables"], case["context_lens"], 0.3, lib=lib)
    tb2 = case["block_tables"].clone()
    tb2[tb2 == 99999] = 0
    out2 = oracle.decode(*args, tb2, case["context_lens"], 0.3, lib=lib)
    tb3 = case["block_tables"].clone()
    tb3[tb3 == 99999] = -123456
    out3 = oracle.decode(*args, tb3, case["context_lens"], 0.3, lib=lib)
    assert torch.equal(out1, out2) and torch.equal(out1, out3)


def pin_I4_dense_equality(lib):
    """Random lengths including 1, multiples of bs and non-multiples,
    shuffled blocks, garbage tails, NaN in every unused row: equals dense
    SDPA on the contiguous rows (fp32: 1e-6; bf16/fp16: within one rounding
    of the fp64 dense result)."""
    bs = 4
    lens = [1, 4, 8, 5, 13, 2, 31]
    for dtype, atol in ((torch.float32, 2e-6), (torch.bfloat16, None), (torch.float16, None)):
        for H, KVH in ((4, 4), (4, 2), (6, 1), (8, 2)):
            case = random_paged_case(100 + H * 10 + KVH, lens, H=H, KVH=KVH, D=16, bs=bs,
                                     dtype=dtype)
            scale = 0.25
            out = oracle.decode(case["q"], case["k_cache"], case["v_cache"],
                                case["block_tables"], case["context_lens"], scale, lib=lib)
            for b in range(len(lens)):
                want = dense_attention(case["q"][b], *case["dense"][b], scale)
                if dtype == torch.float32:
                    _assert_close(out[b], want, atol, atol, f"dense b={b}")
                else:
                    # within one unit in the last place of the output type
                    ulp = torch.finfo(dtype).eps
                    _assert_close(out[b], want, 1e-30, ulp, f"dense {dtype} b={b}")


def pin_shared_prefix(lib):
    """Prefix caching: sequences share the first physical blocks of
    sequence 0 (legal for reads); each still equals dense attention."""
    case = random_paged_case(77, [12, 9, 16, 3], H=4, KVH=2, D=8, bs=4, dtype=torch.float32,
                             share_prefix=2)
    assert case["owned"][1][:2] == case["owned"][0][:2]
    out = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                        case["context_lens"], 0.5, lib=lib)
    for b in range(4):
        want = dense_attention(case["q"][b], *case["dense"][b], 0.5)
        _assert_close(out[b], want, 2e-6, 2e-6, f"shared prefix b={b}")


def pin_closed_forms(lib):
    g = torch.Generator().manual_seed(9)
    bs, KVH, D, H = 4, 2, 8, 4
    case = random_paged_case(9, [1, 6, 11], H=H, KVH=KVH, D=D, bs=bs, dtype=torch.bfloat16)
    args = (case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"])
    # one token: out = that token's V row exactly, whatever q and scale
    out = oracle.decode(case["q"], *args, 3.7, lib=lib)
    vrow = case["dense"][0][1][0]                   # [KVH, D]
    for h in range(H):
        assert torch.equal(out[0, h], vrow[h // (H // KVH)])
    # zero query (or zero scale): uniform weights, out = mean of the V rows
    for q, scale in ((torch.zeros_like(case["q"]), 1.0), (case["q"], 0.0)):
        out = oracle.decode(q, *args, scale, lib=lib)
        for b, n in enumerate([1, 6, 11]):
            vmean = case["dense"][b][1].double().mean(dim=0)     # [KVH, D]
            for h in range(H):
                want = oracle.round_to(vmean[h // (H // KVH)], torch.bfloat16, lib=lib)
                assert torch.equal(out[b, h], want), (b, h)
    # a huge scale turns softmax into argmax: out = V row of the best key
    case32 = random_paged_case(10, [9], H=2, KVH=1, D=8, bs=bs, dtype=torch.float32)
    out = oracle.decode(case32["q"], case32["k_cache"], case32["v_cache"],
                        case32["block_tables"], case32["context_lens"], 1e4, lib=lib)
    dk, dv = case32["dense"][0]
    for h in range(2):
        best = int(torch.argmax(dk[:, 0, :].double() @ case32["q"][0, h].double()))
        _assert_close(out[0, h], dv[best, 0], 1e-6, 1e-6, "argmax")
    # constant V rows: out = the constant
    vc = torch.full_like(case32["v_cache"], -2.5)
    out = oracle.decode(case32["q"], case32["k_cache"], vc, case32["block_tables"],
                        case32["context_lens"], 0.7, lib=lib)
    assert torch.equal(out, torch.full_like(out, -2.5))


def pin_empty_context(lib):
    """context_len 0: a zero output row; nothing is read (a garbage table)."""
    case = random_paged_case(4, [3], H=2, KVH=1, D=4, bs=2, dtype=torch.float32)
    tables = torch.cat([case["block_tables"], torch.full((1, case["block_tables"].shape[1]), 99999,
                                                           dtype=torch.int32)])
    q = torch.cat([case["q"], torch.ones((1, 2, 4))])
    out = oracle.decode(q, case["k_cache"], case["v_cache"], tables,
                        torch.tensor([3, 0], dtype=torch.int32), 1.0, lib=lib)
    assert torch.equal(out[1], torch.zeros((2, 4)))


def pin_error_codes(lib):
    kc = torch.zeros((2, 2, 1, 2))
    k = torch.ones((1, 1, 2))
    try:
        oracle.write(kc, kc.clone(), k, k, torch.tensor([4]), lib=lib)
    except oracle.OracleError as e:
        assert e.code == -2
    else:
        raise AssertionError("slot past the pool accepted")
    q = torch.ones((1, 1, 2))
    for tables, lens, code in (([[5, 0]], [3], -3), ([[-1, 0]], [1], -3), ([[0, 1]], [5], -4),
                               ([[0, 1]], [-1], -4)):
        try:
            oracle.decode(q, kc, kc, torch.tensor(tables, dtype=torch.int32),
                          torch.tensor(lens, dtype=torch.int32), 1.0, lib=lib)
        except oracle.OracleError as e:
            assert e.code == code, (tables, lens, e.code)
        else:
            raise AssertionError(f"bad input accepted: {tables} {lens}")


def pin_rounding(lib):
    """Round-to-nearest-even from float64, single rounding."""
    # hand-worked bf16 ties and the double-rounding trap
    cases = [(1 + 2**-8, 1.0), (1 + 3 * 2**-8, 1 + 2**-6), (1 + 2**-8 + 2**-40, 1 + 2**-7),
             (-(1 + 2**-8 + 2**-40), -(1 + 2**-7)), (2.0**-130, 2.0**-130),
             (2.0**-134, 0.0), (3 * 2.0**-134, 2.0**-132), (255 * 2.0**120, 255 * 2.0**120),
             (255.5 * 2.0**120, math.inf), (255.49 * 2.0**120, 255 * 2.0**120)]
    x = torch.tensor([c[0] for c in cases], dtype=torch.float64)
    got = oracle.widen(oracle.round_to(x, torch.bfloat16, lib=lib), lib=lib)
    want = torch.tensor([c[1] for c in cases], dtype=torch.float64)
    assert torch.equal(got, want), (got, want)
    # fp16: ties, overflow at 65520 (a tie between 65504 and 2^16 -> inf), subnormals
    cases = [(1 + 2**-11, 1.0), (1 + 3 * 2**-11, 1 + 2**-9), (65504.0, 65504.0),
             (65519.99, 65504.0), (65520.0, math.inf), (2.0**-24, 2.0**-24),
             (2.0**-25, 0.0), (3 * 2.0**-25, 2.0**-23), (1 + 2**-11 + 2**-45, 1 + 2**-10)]
    x = torch.tensor([c[0] for c in cases], dtype=torch.float64)
    got = oracle.widen(oracle.round_to(x, torch.float16, lib=lib), lib=lib)
    want = torch.tensor([c[1] for c in cases], dtype=torch.float64)
    assert torch.equal(got, want), (got, want)
    # against torch's float32 -> bf16 / fp16 conversion (float32 inputs: no
    # double rounding possible), including exact ties and subnormals
    g = torch.Generator().manual_seed(1)
    f = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-40, 40, (20000,), generator=g).float())
    ties = (torch.randint(-2**15, 2**15, (2000,), generator=g).to(torch.int32) << 16) | 0x8000
    f = torch.cat([f, ties.view(torch.float32), torch.tensor([1e-40, -3e-39, 6e-8, 3e-5])])
    f = f[torch.isfinite(f)]
    for dt in (torch.bfloat16, torch.float16):
        mine = oracle.round_to(f.double(), dt, lib=lib)
        ref = f.to(dt)
        assert torch.equal(mine.view(torch.int16), ref.view(torch.int16)), dt
    # float64 -> float32 against torch's conversion
    d = torch.randn(20000, generator=g, dtype=torch.float64) * 1e3
    assert torch.equal(oracle.round_to(d, torch.float32, lib=lib), d.float())


def pin_widen(lib):
    g = torch.Generator().manual_seed(2)
    bits = torch.randint(-2**15, 2**15, (50000,), generator=g, dtype=torch.int32).to(torch.int16)
    for dt in (torch.bfloat16, torch.float16):
        x = bits.view(dt)
        mine = oracle.widen(x, lib=lib)
        ref = x.double()
        same = (mine == ref) | (torch.isnan(mine) & torch.isnan(ref))
        assert same.all(), dt


# ------------------------------------------------------------------ prefill

def _prefill_case(seed, lens, qlens, H, KVH, D, bs, dtype):
    """A paged case plus varlen queries: sequence b's queries are its last
    qlens[b] positions."""
    case = random_paged_case(seed, lens, H=H, KVH=KVH, D=D, bs=bs, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 1)
    cu = [0]
    for ql in qlens:
        cu.append(cu[-1] + ql)
    q = torch.randn((cu[-1], H, D), generator=g, dtype=torch.float64).to(dtype)
    return case, q, torch.tensor(cu, dtype=torch.int32)


def dense_causal(q, k, v, scale, n, is_causal=False):
    """q [qlen, H, D] at positions n-qlen .. n-1; k/v [n, KVH, D]; SDPA in fp64
    with an explicit mask (query at p sees keys 0..p), or SDPA's own causal
    flag when the queries cover the whole context."""
    qlen, H = q.shape[0], q.shape[1]
    q64 = q.double().permute(1, 0, 2).unsqueeze(0)
    k64 = k.double().permute(1, 0, 2).unsqueeze(0)
    v64 = v.double().permute(1, 0, 2).unsqueeze(0)
    gqa = k64.shape[1] != H
    if is_causal:
        assert qlen == n
        o = F.scaled_dot_product_attention(q64, k64, v64, scale=scale, is_causal=True, enable_gqa=gqa)
    else:
        pos = torch.arange(n - qlen, n).unsqueeze(1)
        mask = torch.arange(n).unsqueeze(0) <= pos          # [qlen, n]
        o = F.scaled_dot_product_attention(q64, k64, v64, attn_mask=mask, scale=scale, enable_gqa=gqa)
    return o.squeeze(0).permute(1, 0, 2)                     # [qlen, H, D]


def pin_prefill_dense_causal(lib):
    """Varlen causal prefill over shuffled paged blocks (NaN in unused rows,
    garbage tails) equals masked dense SDPA on the contiguous rows; query
    counts from 1 (decode) to the whole context, lengths on and off block
    edges."""
    lens = [1, 4, 9, 16, 13, 30]
    qlens = [1, 4, 3, 16, 1, 11]
    for dtype in (torch.float32, torch.bfloat16):
        for H, KVH in ((4, 4), (4, 2), (6, 1)):
            case, q, cu = _prefill_case(200 + H + KVH, lens, qlens, H, KVH, 16, 4, dtype)
            out = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                                 case["context_lens"], 0.3, lib=lib)
            for b, (n, ql) in enumerate(zip(lens, qlens)):
                want = dense_causal(q[cu[b]:cu[b + 1]], *case["dense"][b], 0.3, n)
                got = out[cu[b]:cu[b + 1]]
                if dtype == torch.float32:
                    _assert_close(got, want, 2e-6, 2e-6, f"prefill b={b}")
                else:
                    _assert_close(got, want, 1e-30, torch.finfo(dtype).eps, f"prefill {dtype} b={b}")


def pin_prefill_full_is_causal(lib):
    """Queries covering the whole context: SDPA's own causal flag."""
    lens = [7, 12, 5]
    case, q, cu = _prefill_case(301, lens, lens, 4, 2, 8, 4, torch.float32)
    out = oracle.prefill(q, case["k_cache"], case["v_cache"], case["block_tables"], cu,
                         case["context_lens"], 0.5, lib=lib)
    for b, n in enumerate(lens):
        want = dense_causal(q[cu[b]:cu[b + 1]], *case["dense"][b], 0.5, n, is_causal=True)
        _assert_close(out[cu[b]:cu[b + 1]], want, 2e-6, 2e-6, f"full prefill b={b}")


def pin_prefill_closed_forms(lib):
    """Whole-context prefill: the first query sees only token 0 (its V row
    exactly); with zero scale query i gets the mean of V rows 0..i; one
    query per sequence is decode (the decode pins' function)."""
    lens = [6, 11]
    H, KVH = 4, 2
    case, q, cu = _prefill_case(302, lens, lens, H, KVH, 8, 4, torch.bfloat16)
    args = (case["k_cache"], case["v_cache"], case["block_tables"], cu, case["context_lens"])
    out = oracle.prefill(q, *args, 2.3, lib=lib)
    for b in range(2):
        v0 = case["dense"][b][1][0]
        for h in range(H):
            assert torch.equal(out[cu[b], h], v0[h // (H // KVH)]), (b, h)
    out = oracle.prefill(q, *args, 0.0, lib=lib)
    for b, n in enumerate(lens):
        dv = case["dense"][b][1].double()
        for i in range(n):
            mean = dv[:i + 1].mean(dim=0)
            for h in range(H):
                want = oracle.round_to(mean[h // (H // KVH)], torch.bfloat16, lib=lib)
                assert torch.equal(out[cu[b] + i, h], want), (b, i, h)
    # one query per sequence == decode
    case1, q1, cu1 = _prefill_case(303, [5, 9, 1], [1, 1, 1], H, KVH, 8, 4, torch.float32)
    got = oracle.prefill(q1, case1["k_cache"], case1["v_cache"], case1["block_tables"], cu1,
                         case1["context_lens"], 0.4, lib=lib)
    want = oracle.decode(q1, case1["k_cache"], case1["v_cache"], case1["block_tables"],
                         case1["context_lens"], 0.4, lib=lib)
    assert torch.equal(got, want)


def pin_prefill_errors(lib):
    case, q, cu = _prefill_case(304, [3, 4], [2, 2], 2, 1, 4, 2, torch.float32)
    args = (case["k_cache"], case["v_cache"], case["block_tables"])
    bad_lens = torch.tensor([1, 4], dtype=torch.int32)        # more queries than context
    for cu_, lens_ in ((cu, bad_lens), (torch.tensor([1, 3, 4], dtype=torch.int32), case["context_lens"])):
        try:
            oracle.prefill(q if int(cu_[-1]) == q.shape[0] else q[:int(cu_[-1])], *args, cu_, lens_,
                           1.0, lib=lib)
        except oracle.OracleError:
            continue
        raise AssertionError("accepted an invalid prefill batch")


ALL_PINS = [
    pin_example1_write, pin_key_answer_slot7, pin_I1_sentinel, pin_example2_decode,
    pin_example2_softmax, pin_key_answer_n5_truncation, pin_gqa_mapping,
    pin_I2_tail_never_read, pin_I4_dense_equality, pin_shared_prefix, pin_closed_forms,
    pin_empty_context, pin_error_codes, pin_rounding, pin_widen, pin_prefill_dense_causal,
    pin_prefill_full_is_causal, pin_prefill_closed_forms, pin_prefill_errors,
]
