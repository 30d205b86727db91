"""Seeded synthetic inputs for the paged KV-cache write and decode attention.

This module only draws inputs: context lengths, a shuffled physical-block
assignment, block tables with garbage tails, pool contents, queries, new
tokens and their slots.  It computes nothing the operations compute, and it
is shared by the tests (which feed the same tensors to the oracle and to the
CUDA library) and by ``bench.py``.

The workloads follow the shapes and distributions of the course page
"P09 · Paged KV 写入 + decode attention（参考实现）": shuffled physical
blocks (section 题面速览, "物理块不连续（测试会打乱分配）"), block-table
tails filled with garbage such as 99999 (invariant I2), padding tokens with
slot -1 whose rows hold a sentinel (invariant I1), and lengths that include
1, exact multiples of the block size and non-multiples (invariant I4).
Slot assignment (which physical slot a new token gets) is the scheduler's
job upstream of these operations; it is synthesised here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

SENTINEL = 9.0  # value of every element of a padding token (invariant I1)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int                      # sequences in the batch (padded batch for `pad_seqs`)
    H: int                      # query heads
    KVH: int                    # KV heads
    D: int                      # head dim
    bs: int                     # block size (tokens per physical block)
    dtype: torch.dtype
    len_dist: str               # "uniform" | "loguniform"
    len_lo: int
    len_hi: int
    forced_lens: tuple = ()     # lengths that must appear (1, multiples of bs, ...)
    pool_factor: float = 1.25   # physical pool = pool_factor x blocks needed
    num_blocks: int = 0         # fixed pool size (0: from pool_factor)
    max_blocks: int = 0         # table width (0: enough for len_hi)
    tail: str = "garbage"       # "99999" | "garbage": unused table entries
    pad_seqs: int = 0           # trailing padded sequences: length 0, slot -1
    steps: int = 1              # decode steps (per-step workload)
    write_pads: int = 0         # extra padding tokens (slot -1) in the write batch

    @property
    def G(self) -> int:
        return self.H // self.KVH

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def table_width(self) -> int:
        if self.max_blocks:
            return self.max_blocks
        return -(-(self.len_hi + self.steps) // self.bs)


# The five workloads: small fp32 case, Llama-3-8B-shaped decode, long-context
# split-KV, MQA / wide head, and the per-step write+attend loop with a padded
# (CUDA-graph sized) batch.
CONFIGS = {
    "tiny_fp32": DecodeConfig("tiny_fp32", B=4, H=4, KVH=2, D=64, bs=16, dtype=torch.float32,
                              len_dist="uniform", len_lo=1, len_hi=100, forced_lens=(1, 16, 17),
                              num_blocks=64, tail="99999", write_pads=3),
    "llama8b_bf16": DecodeConfig("llama8b_bf16", B=64, H=32, KVH=8, D=128, bs=16,
                                 dtype=torch.bfloat16, len_dist="uniform", len_lo=512,
                                 len_hi=4096, forced_lens=(512, 4096), max_blocks=256),
    "long_bf16": DecodeConfig("long_bf16", B=8, H=32, KVH=8, D=128, bs=16, dtype=torch.bfloat16,
                              len_dist="uniform", len_lo=16384, len_hi=32768, max_blocks=2048),
    "mqa_bf16": DecodeConfig("mqa_bf16", B=128, H=16, KVH=1, D=256, bs=32, dtype=torch.bfloat16,
                             len_dist="loguniform", len_lo=1, len_hi=8192,
                             forced_lens=(1, 32, 64, 4096, 8192), max_blocks=256),
    "step_bf16": DecodeConfig("step_bf16", B=256, H=64, KVH=8, D=128, bs=16, dtype=torch.bfloat16,
                              len_dist="uniform", len_lo=1, len_hi=2048, pad_seqs=56, steps=32,
                              max_blocks=132),
}


def small_variant(cfg: DecodeConfig, B: int | None = None, len_hi: int | None = None,
                  **kw) -> DecodeConfig:
    """The same shapes with fewer / shorter sequences (for oracle-sized tests)."""
    changes = dict(kw)
    if B is not None:
        changes["B"] = B
        changes["pad_seqs"] = min(cfg.pad_seqs, max(0, B // 4)) if cfg.pad_seqs else 0
    if len_hi is not None:
        changes["len_hi"] = len_hi
        changes["len_lo"] = min(cfg.len_lo, len_hi)
        changes["forced_lens"] = tuple(x for x in cfg.forced_lens if x <= len_hi)
        if cfg.max_blocks:
            changes["max_blocks"] = -(-(len_hi + cfg.steps) // cfg.bs) + 2
    return replace(cfg, **changes)


@dataclass
class DecodeInputs:
    cfg: DecodeConfig
    q: torch.Tensor             # [B, H, D] (queries of the first step)
    k_cache: torch.Tensor       # [num_blocks, bs, KVH, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor  # [B, max_blocks] int32, garbage past ceil(n/bs)
    context_lens: torch.Tensor  # [B] int32 (lengths seen by the first decode step)
    scale: float
    num_blocks: int
    owned: list = field(default_factory=list)  # per sequence: its physical blocks, in order


def _lengths(cfg: DecodeConfig, g: torch.Generator) -> torch.Tensor:
    live = cfg.B - cfg.pad_seqs
    if cfg.len_dist == "uniform":
        n = torch.randint(cfg.len_lo, cfg.len_hi + 1, (live,), generator=g, dtype=torch.int64)
    elif cfg.len_dist == "loguniform":
        u = torch.rand(live, generator=g, dtype=torch.float64)
        lo, hi = math.log(cfg.len_lo), math.log(cfg.len_hi + 1)
        n = torch.exp(lo + u * (hi - lo)).floor().to(torch.int64).clamp(cfg.len_lo, cfg.len_hi)
    else:
        raise ValueError(cfg.len_dist)
    forced = [x for x in cfg.forced_lens][:live]
    if forced:
        n[: len(forced)] = torch.tensor(forced, dtype=torch.int64)
        n = n[torch.randperm(live, generator=g)]
    return torch.cat([n, torch.zeros(cfg.pad_seqs, dtype=torch.int64)])


def draw_lengths(cfg: DecodeConfig, seed: int) -> torch.Tensor:
    """The context lengths make_decode_inputs(cfg, seed) draws (its first
    draw), without the rest of the batch: to size a run before making it."""
    return _lengths(cfg, torch.Generator().manual_seed(seed)).to(torch.int32)


def _garbage_tail(cfg: DecodeConfig, shape, num_blocks: int, g: torch.Generator) -> torch.Tensor:
    if cfg.tail == "99999":
        return torch.full(shape, 99999, dtype=torch.int32)
    # indices that are never valid: past the pool, or negative
    hi = torch.randint(num_blocks, 2**31 - 1, shape, generator=g, dtype=torch.int64)
    neg = -torch.randint(1, 2**31 - 1, shape, generator=g, dtype=torch.int64)
    pick = torch.rand(shape, generator=g) < 0.75
    return torch.where(pick, hi, neg).to(torch.int32)


def _randn(shape, dtype, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32, device=device).to(dtype)


def make_decode_inputs(cfg: DecodeConfig, seed: int, device="cpu",
                       poison_unused: bool = False) -> DecodeInputs:
    """Draw one decode batch.

    Lengths, block assignment and tables are drawn on the CPU from ``seed``;
    the pool and queries are drawn with a generator on ``device`` (so the
    same seed gives different floats on CPU and GPU: compare the CUDA path
    and the oracle on the SAME tensors, copied).  ``poison_unused`` fills
    every cache row no sequence uses (unassigned blocks and the tail of each
    last block) with NaN, so that any read of them shows in the output."""
    g = torch.Generator().manual_seed(seed)
    lens = _lengths(cfg, g)   # the first draw (draw_lengths gives the same)
    # room to grow for per-step runs: step s appends the token at position n + s
    total_len = lens + (cfg.steps if cfg.steps > 1 else 0)
    total_len[cfg.B - cfg.pad_seqs:] = 0
    need = [-(-int(x) // cfg.bs) for x in total_len]
    total_blocks = sum(need)
    num_blocks = cfg.num_blocks or max(1, math.ceil(cfg.pool_factor * total_blocks))
    if num_blocks < total_blocks:
        raise ValueError(f"pool of {num_blocks} blocks < {total_blocks} needed")
    perm = torch.randperm(num_blocks, generator=g)
    width = cfg.table_width
    if max(need, default=0) > width:
        raise ValueError("table narrower than the longest sequence")
    tables = _garbage_tail(cfg, (cfg.B, width), num_blocks, g)
    owned, cursor = [], 0
    for b, nb in enumerate(need):
        blocks = perm[cursor:cursor + nb]
        cursor += nb
        owned.append(blocks.tolist())
        first_nb = -(-int(lens[b]) // cfg.bs)        # entries valid at the first step
        tables[b, :first_nb] = blocks[:first_nb].to(torch.int32)

    dg = torch.Generator(device=device).manual_seed(seed + 7919)
    shape = (num_blocks, cfg.bs, cfg.KVH, cfg.D)
    k_cache = _randn(shape, cfg.dtype, dg, device)
    v_cache = _randn(shape, cfg.dtype, dg, device)
    q = _randn((cfg.B, cfg.H, cfg.D), cfg.dtype, dg, device)
    if poison_unused:
        used = torch.zeros(num_blocks * cfg.bs, dtype=torch.bool)
        for b, blocks in enumerate(owned):
            for t in range(int(lens[b])):
                used[blocks[t // cfg.bs] * cfg.bs + t % cfg.bs] = True
        mask = (~used).view(num_blocks, cfg.bs).to(device)
        k_cache[mask] = float("nan")
        v_cache[mask] = float("nan")
    return DecodeInputs(cfg, q, k_cache, v_cache, tables, lens.to(torch.int32), cfg.scale,
                        num_blocks, owned)


@dataclass
class WriteBatch:
    k: torch.Tensor             # [T, KVH, D]
    v: torch.Tensor
    slot_mapping: torch.Tensor  # [T] int64, -1 for padding tokens


def slot_of(owned_blocks, t: int, bs: int) -> int:
    """The flat slot the scheduler assigned to logical token t of a sequence."""
    return owned_blocks[t // bs] * bs + t % bs


def make_write_batch(inp: DecodeInputs, positions, seed: int, device="cpu",
                     extra_pads: int = 0) -> WriteBatch:
    """New tokens to write: for sequence b, logical token positions[b] (None or
    a negative position: a padding token).  ``extra_pads`` padding tokens are
    appended.  Padding tokens get slot -1 and every element = SENTINEL."""
    cfg = inp.cfg
    slots = []
    for b, pos in enumerate(positions):
        if pos is None or pos < 0:
            slots.append(-1)
        else:
            slots.append(slot_of(inp.owned[b], int(pos), cfg.bs))
    slots += [-1] * extra_pads
    T = len(slots)
    dg = torch.Generator(device=device).manual_seed(seed + 104729)
    k = _randn((T, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    v = _randn((T, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    slot_t = torch.tensor(slots, dtype=torch.int64)
    pad = (slot_t < 0).to(device)
    k[pad] = SENTINEL
    v[pad] = SENTINEL
    return WriteBatch(k, v, slot_t.to(device))


def make_bulk_fill(inp: DecodeInputs, seed: int, device="cpu") -> WriteBatch:
    """Every context token of every sequence, as one write batch (the prefill
    of the whole pool), in a random token order."""
    cfg = inp.cfg
    slots = []
    for b in range(cfg.B):
        for t in range(int(inp.context_lens[b])):
            slots.append(slot_of(inp.owned[b], t, cfg.bs))
    g = torch.Generator().manual_seed(seed)
    slot_t = torch.tensor(slots, dtype=torch.int64)
    slot_t = slot_t[torch.randperm(slot_t.numel(), generator=g)]
    dg = torch.Generator(device=device).manual_seed(seed + 15485863)
    T = slot_t.numel()
    k = _randn((T, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    v = _randn((T, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    return WriteBatch(k, v, slot_t.to(device))


@dataclass
class StepInputs:
    """Per-step write+attend loop: before step s every live sequence appends
    one token (slot from its own next block when it crosses a block edge),
    padded sequences get slot -1 and length 0."""
    slots: torch.Tensor         # [steps, B] int64
    lens: torch.Tensor          # [steps, B] int32, lengths seen by the step's decode
    tables: torch.Tensor        # [steps, B, max_blocks] int32
    k: torch.Tensor             # [steps, B, KVH, D] new tokens
    v: torch.Tensor
    q: torch.Tensor             # [steps, B, H, D]


def make_steps(inp: DecodeInputs, seed: int, device="cpu") -> StepInputs:
    cfg = inp.cfg
    S, B = cfg.steps, cfg.B
    live = B - cfg.pad_seqs
    g = torch.Generator().manual_seed(seed)
    base_tail = _garbage_tail(cfg, (B, cfg.table_width), inp.num_blocks, g)
    slots = torch.full((S, B), -1, dtype=torch.int64)
    lens = torch.zeros((S, B), dtype=torch.int32)
    tables = base_tail.unsqueeze(0).repeat(S, 1, 1)
    for s in range(S):
        for b in range(live):
            n0 = int(inp.context_lens[b])
            pos = n0 + s                              # the token appended before step s
            slots[s, b] = slot_of(inp.owned[b], pos, cfg.bs)
            lens[s, b] = pos + 1
            nb = -(-(pos + 1) // cfg.bs)
            tables[s, b, :nb] = torch.tensor(inp.owned[b][:nb], dtype=torch.int32)
    dg = torch.Generator(device=device).manual_seed(seed + 32452843)
    k = _randn((S, B, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    v = _randn((S, B, cfg.KVH, cfg.D), cfg.dtype, dg, device)
    q = _randn((S, B, cfg.H, cfg.D), cfg.dtype, dg, device)
    pad = (slots < 0).to(device)
    k[pad] = SENTINEL
    v[pad] = SENTINEL
    return StepInputs(slots.to(device), lens.to(device), tables.to(device), k, v, q)


def decode_bytes(context_lens, B: int, H: int, KVH: int, D: int, bs: int, elem: int) -> int:
    """Algorithmic bytes of one decode call: K and V rows actually used, q and
    out, the used table prefix and the lengths."""
    lens = [int(x) for x in context_lens]
    kv = sum(2 * n * KVH * D * elem for n in lens)
    qo = 2 * B * H * D * elem
    tbl = sum(-(-n // bs) * 4 for n in lens) + 4 * B
    return kv + qo + tbl


def write_bytes(slot_mapping, KVH: int, D: int, elem: int) -> int:
    """Algorithmic bytes of one write call: read k and v rows of the kept
    tokens, write them into both caches, read every slot."""
    s = torch.as_tensor(slot_mapping).cpu()
    kept = int((s >= 0).sum())
    return kept * 4 * KVH * D * elem + 8 * s.numel()


# ------------------------------------------------------------------ prefill

@dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int                      # sequences
    H: int
    KVH: int
    D: int
    bs: int
    dtype: torch.dtype
    len_lo: int                 # context lengths uniform in [len_lo, len_hi]
    len_hi: int
    chunk_lo: int               # sequences 1, 3, 5, ...: a chunk of this many new
    chunk_hi: int               # queries on top of a cached prefix; the others whole
    pool_factor: float = 1.25

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def table_width(self) -> int:
        return -(-self.len_hi // self.bs)


# A Llama-3-8B-shaped varlen prefill batch: half the sequences prefill their
# whole prompt, half prefill a chunk on top of a cached prefix.
PREFILL_CONFIGS = {
    "prefill_bf16": PrefillConfig("prefill_bf16", B=16, H=32, KVH=8, D=128, bs=16,
                                  dtype=torch.bfloat16, len_lo=512, len_hi=4096, chunk_lo=128,
                                  chunk_hi=512),
}


@dataclass
class PrefillInputs:
    cfg: PrefillConfig
    q: torch.Tensor             # [total_q, H, D]
    k_cache: torch.Tensor       # [num_blocks, bs, KVH, D], every context token written
    v_cache: torch.Tensor
    block_tables: torch.Tensor  # [B, max_blocks] int32, garbage past ceil(n/bs)
    context_lens: torch.Tensor  # [B] int32
    cu_seqlens_q: torch.Tensor  # [B + 1] int32
    scale: float
    max_q_len: int
    num_blocks: int


def make_prefill_inputs(cfg: PrefillConfig, seed: int, device="cpu") -> PrefillInputs:
    """Lengths, shuffled block assignment and tables on the CPU from ``seed``;
    pool and queries with a generator on ``device`` (compare the CUDA path
    and the oracle on the SAME tensors, copied)."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(cfg.len_lo, cfg.len_hi + 1, (cfg.B,), generator=g, dtype=torch.int64)
    qlens = lens.clone()
    chunk = torch.randint(cfg.chunk_lo, cfg.chunk_hi + 1, (cfg.B,), generator=g, dtype=torch.int64)
    qlens[1::2] = torch.minimum(chunk[1::2], lens[1::2])
    need = [-(-int(n) // cfg.bs) for n in lens]
    num_blocks = max(1, math.ceil(cfg.pool_factor * sum(need)))
    perm = torch.randperm(num_blocks, generator=g)
    shim = DecodeConfig(cfg.name, cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.dtype, "uniform",
                        cfg.len_lo, cfg.len_hi)
    tables = _garbage_tail(shim, (cfg.B, cfg.table_width), num_blocks, g)
    cursor = 0
    for b, nb in enumerate(need):
        tables[b, :nb] = perm[cursor:cursor + nb].to(torch.int32)
        cursor += nb
    cu = torch.zeros(cfg.B + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(qlens, 0).to(torch.int32)
    dg = torch.Generator(device=device).manual_seed(seed + 7919)
    shape = (num_blocks, cfg.bs, cfg.KVH, cfg.D)
    k_cache = _randn(shape, cfg.dtype, dg, device)
    v_cache = _randn(shape, cfg.dtype, dg, device)
    q = _randn((int(cu[-1]), cfg.H, cfg.D), cfg.dtype, dg, device)
    return PrefillInputs(cfg, q, k_cache, v_cache, tables, lens.to(torch.int32), cu, cfg.scale,
                         int(qlens.max()), num_blocks)


def prefill_flops(context_lens, cu_seqlens_q, H: int, D: int) -> int:
    """Multiply-add flops of one causal prefill call: query i of a sequence
    with n tokens and qlen queries sees n - qlen + i + 1 keys; each key costs
    2 * D flops for q.k and 2 * D for p.v, per query head."""
    total = 0
    for b in range(len(context_lens)):
        n = int(context_lens[b])
        ql = int(cu_seqlens_q[b + 1]) - int(cu_seqlens_q[b])
        keys = ql * (n - ql) + ql * (ql + 1) // 2
        total += 4 * D * H * keys
    return total
