"""The block manager feeding the CUDA path: prompts admitted with prefix
sharing (cached tokens get slot -1 and are not written again), then fused
write + decode steps with the manager's slots, tables and lengths, a
sequence freed and a new one reviving its cached prefix mid-way.

Every token's K/V is a deterministic function of the sequence's tokens up
to it (as a model's would be), so sharing a block is only correct when the
prefixes really agree.  Checks: the device cache read through each table
equals every sequence's own rows bit-exactly, and each step's output
matches the oracle's write-then-decode on the same cache."""
import math

import pytest
import torch

import oracle
import paged_kv_cache_67_gb300 as pkv
from gpu_helpers import assert_close, bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
KVH, D, H, BS = 2, 128, 8, 16
DT = torch.bfloat16


def kv_row(prefix):
    """K and V rows [KVH, D] of the last token of `prefix` (a tuple of ids)."""
    g = torch.Generator().manual_seed(hash(prefix) & 0x7FFFFFFF)
    return (torch.randn((KVH, D), generator=g).to(DT), torch.randn((KVH, D), generator=g).to(DT))


def rows_for(tokens, start=0):
    k, v = zip(*(kv_row(tuple(tokens[:t + 1])) for t in range(start, len(tokens))))
    return torch.stack(k), torch.stack(v)


def test_block_manager_drives_fused_steps():
    num_blocks, max_blocks = 64, 12
    bm = pkv.BlockManager(num_blocks, BS)
    kc = torch.full((num_blocks, BS, KVH, D), float("nan"), dtype=DT, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    kc_o, vc_o = kc.cpu(), vc.cpu()                  # the oracle's copy of the cache
    stem = [7] * 20 + list(range(30))
    prompts = {0: stem[:40], 1: stem[:37] + [5, 6], 2: stem[:33], 3: [9] * 50}
    tokens = {}
    for sid, p in prompts.items():
        slots, cached = bm.add_sequence(sid, p)
        k, v = rows_for(p)
        pkv.pkv_write(kc, vc, k.to(DEV), v.to(DEV), slots.to(DEV))
        oracle.write(kc_o, vc_o, k, v, slots)
        tokens[sid] = list(p)
        if sid in (1, 2):
            assert cached == 32                       # two shared full blocks of the stem
    gen = torch.Generator().manual_seed(3)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = pkv.DecodeWorkspace(5, H, KVH, D, BS, max_blocks, max_blocks * BS, 0, device=DEV)
    for step in range(12):
        if step == 5:                                 # free one, admit one sharing its prefix
            bm.free_sequence(0)
            del tokens[0]
            p = stem[:36] + [1]
            slots, cached = bm.add_sequence(4, p)
            assert cached == 32
            k, v = rows_for(p)
            pkv.pkv_write(kc, vc, k.to(DEV), v.to(DEV), slots.to(DEV))
            oracle.write(kc_o, vc_o, k, v, slots)
            tokens[4] = list(p)
        batch = sorted(tokens) + [-1]                 # one padding entry
        new_tok = [int(torch.randint(0, 50, (1,), generator=gen)) for _ in batch]
        slots = bm.append_tokens(batch, new_tok)
        for sid, t in zip(batch, new_tok):
            if sid >= 0:
                tokens[sid].append(t)
        k = torch.zeros((len(batch), KVH, D), dtype=DT)
        v = torch.zeros_like(k)
        for i, sid in enumerate(batch):
            if sid >= 0:
                k[i], v[i] = kv_row(tuple(tokens[sid]))
        tables, lens = bm.build_batch(batch, max_blocks)
        q = torch.randn((len(batch), H, D), generator=gen).to(DT)
        out = torch.empty((len(batch), H, D), dtype=DT, device=DEV)
        pkv.pkv_write_decode_attention(out, q.to(DEV), k.to(DEV), v.to(DEV), slots.to(DEV), kc, vc,
                                       tables.to(DEV), lens.to(DEV), 1 / math.sqrt(D),
                                       max_context_len=max_blocks * BS, workspace=ws, err_flags=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        oracle.write(kc_o, vc_o, k, v, slots)
        want = oracle.decode(q, kc_o, vc_o, tables, lens, 1 / math.sqrt(D))
        assert_close(out, want, DT, f"step {step}")
        assert bool((out[-1] == 0).all())
    # the device cache, read through each table, holds every sequence's own rows
    kc_c, vc_c = kc.cpu(), vc.cpu()
    assert torch.equal(bits(kc_c), bits(kc_o)) and torch.equal(bits(vc_c), bits(vc_o))
    for sid, toks in tokens.items():
        n, table = bm.sequence_info(sid)
        k, v = rows_for(toks)
        idx = torch.tensor([table[t // BS] * BS + t % BS for t in range(n)])
        assert torch.equal(bits(kc_c.view(-1, KVH, D)[idx]), bits(k))
        assert torch.equal(bits(vc_c.view(-1, KVH, D)[idx]), bits(v))
