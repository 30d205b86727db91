"""The host block manager (include/pkv_block_manager.h) on the CPU.

Its results are checked against what a paged cache must guarantee, not
against a second implementation: a simulated cache of token ids is
written at every slot the manager hands out (exactly what write_kv would
do with the K/V of those tokens), and after every operation each live
sequence, read back through its block table, must hold exactly its own
tokens -- which fails for a wrong slot, a block handed to two sequences
with different contents, a wrong prefix match, an evicted block still in
use, or a cached token whose slot was withheld but whose block was not
really shared.  Reference counts and the free count are checked against
the tables."""
import random
import threading

import pytest
import torch

from paged_kv_cache_67_gb300 import build as libbuild


@pytest.fixture(scope="module")
def pkv():
    libbuild.build()
    import paged_kv_cache_67_gb300 as m
    m.load_library()
    return m


class Model:
    """The caller's view: live sequences' tokens and a cache of token ids."""

    def __init__(self, bm, num_blocks, bs):
        self.bm, self.bs = bm, bs
        self.cache = [None] * (num_blocks * bs)
        self.tokens = {}

    def add(self, sid, toks):
        slots, cached = self.bm.add_sequence(sid, toks)
        assert cached % self.bs == 0 and 0 <= cached <= len(toks)
        for t, s in enumerate(slots.tolist()):
            assert (s == -1) == (t < cached)
            if s >= 0:
                self.cache[s] = toks[t]
        self.tokens[sid] = list(toks)
        return cached

    def append(self, sids, toks):
        slots = self.bm.append_tokens(sids, toks).tolist()
        for sid, tok, s in zip(sids, toks, slots):
            if sid < 0:
                assert s == -1
                continue
            assert s >= 0
            self.cache[s] = tok
            self.tokens[sid].append(tok)
        return slots

    def free(self, sid):
        self.bm.free_sequence(sid)
        del self.tokens[sid]

    def check(self):
        bs = self.bm.block_size
        owners = {}
        for sid, toks in self.tokens.items():
            n, table = self.bm.sequence_info(sid)
            assert n == len(toks)
            assert len(table) == -(-n // bs)
            assert len(set(table)) == len(table)
            got = [self.cache[table[t // bs] * bs + t % bs] for t in range(n)]
            assert got == toks, f"sequence {sid} reads back other tokens"
            for j, blk in enumerate(table):
                owners.setdefault(blk, []).append((sid, j))
        for blk, who in owners.items():
            assert self.bm.refcount(blk) == len(who)
            if len(who) > 1:  # shared: same logical index, full block, same prefix
                j0 = who[0][1]
                for sid, j in who:
                    assert j == j0 and len(self.tokens[sid]) >= (j + 1) * bs
                ref = self.tokens[who[0][0]][:(j0 + 1) * bs]
                assert all(self.tokens[sid][:(j0 + 1) * bs] == ref for sid, _ in who)
        free, _, live = self.bm.stats()
        assert live == len(self.tokens)
        assert free == self.bm.num_blocks - len(owners)
        for blk in range(self.bm.num_blocks):
            if blk not in owners:
                assert self.bm.refcount(blk) == 0


def test_slots_and_tables(pkv):
    bm = pkv.BlockManager(16, 4)
    m = Model(bm, 16, 4)
    assert m.add(0, list(range(10))) == 0
    n, table = bm.sequence_info(0)
    assert n == 10 and len(table) == 3
    m.check()
    slots = m.append([0], [10])
    assert slots == [table[2] * 4 + 2]
    m.append([0], [11])
    m.append([0], [12])  # crosses a block edge: a fourth block
    assert len(bm.sequence_info(0)[1]) == 4
    m.check()
    tables, lens = bm.build_batch([0, -1], 6, tail=-7)
    assert lens.tolist() == [13, 0]
    assert tables[0, :4].tolist() == bm.sequence_info(0)[1] and tables[0, 4:].tolist() == [-7, -7]
    assert tables[1].tolist() == [-7] * 6


def test_prefix_sharing_full_blocks_only(pkv):
    bm = pkv.BlockManager(32, 4)
    m = Model(bm, 32, 4)
    a = [1, 2, 3, 4, 5, 6, 7, 8, 9, 10]
    assert m.add(0, a) == 0
    assert m.add(1, a[:8] + [99, 98, 97]) == 8       # two full blocks shared
    assert m.add(2, a) == 8                          # the partial third block is never shared
    assert m.add(3, [1, 2, 3, 4, 0, 6, 7, 8]) == 4   # differs inside block 1
    assert m.add(4, [0] + a[1:]) == 0                # differs in the first token
    t0, t1 = bm.sequence_info(0)[1], bm.sequence_info(1)[1]
    assert t0[:2] == t1[:2] and t0[2] != t1[2]
    assert bm.refcount(t0[0]) == 4 and bm.refcount(t0[1]) == 3
    m.check()
    # a block filled by appends is shared too
    m.append([1, 0], [96, 11])
    m.append([0], [12])                              # sequence 0's third block is full now
    assert m.add(5, a + [11, 12, 13]) == 12
    m.check()


def test_prefix_caching_off(pkv):
    bm = pkv.BlockManager(32, 4, prefix_caching=False)
    m = Model(bm, 32, 4)
    a = list(range(12))
    assert m.add(0, a) == 0 and m.add(1, a) == 0
    assert set(bm.sequence_info(0)[1]).isdisjoint(bm.sequence_info(1)[1])
    assert bm.stats()[1] == 0
    m.check()


def test_free_revive_and_lru_eviction(pkv):
    bm = pkv.BlockManager(6, 4)
    m = Model(bm, 6, 4)
    A, B = [1] * 8, [2] * 8
    m.add(0, A)
    m.add(1, B)
    tA, tB = bm.sequence_info(0)[1], bm.sequence_info(1)[1]
    m.free(0)
    m.free(1)                                        # A freed before B: A is older
    assert bm.stats()[:2] == (6, 4)
    m.check()
    assert m.add(2, A) == 8                          # revived, same blocks
    assert bm.sequence_info(2)[1] == tA
    m.free(2)                                        # now B is the older cached prefix
    m.add(3, [3] * 8)                                # two fresh blocks: the 2 plain ones
    m.add(4, [4] * 8)                                # two more: evict the oldest cached (B)
    assert m.add(5, B) == 0                          # B was evicted ...
    m.free(5)
    m.free(3)
    m.free(4)
    m.check()


def test_out_of_blocks_changes_nothing(pkv):
    bm = pkv.BlockManager(5, 4)
    m = Model(bm, 5, 4)
    m.add(0, list(range(8)))
    m.add(1, list(range(100, 108)))
    before = (bm.stats(), bm.sequence_info(0), bm.sequence_info(1))
    with pytest.raises(pkv.PkvError) as e:
        bm.add_sequence(2, list(range(200, 209)))    # needs 3 blocks, 1 free
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    with pytest.raises(pkv.PkvError) as e:
        bm.append_tokens([0, 1], [8, 108])            # both cross an edge: 2 needed
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert (bm.stats(), bm.sequence_info(0), bm.sequence_info(1)) == before
    m.append([0], [8])
    m.check()


def test_argument_errors(pkv):
    bm = pkv.BlockManager(8, 4)
    bm.add_sequence(0, [1, 2])
    for call in (lambda: bm.add_sequence(0, [1]),            # duplicate id
                 lambda: bm.add_sequence(-1, [1]),           # negative id
                 lambda: bm.add_sequence(1, []),             # empty prompt
                 lambda: bm.append_tokens([5], [1]),         # unknown id
                 lambda: bm.append_tokens([0, 0], [1, 2]),   # repeated id
                 lambda: bm.free_sequence(5),
                 lambda: bm.build_batch([0], 0),             # table wider than the row
                 lambda: bm.sequence_info(9)):
        with pytest.raises(pkv.PkvError) as e:
            call()
        assert e.value.status == 1
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(0, 4)
    with pytest.raises(pkv.PkvError):
        pkv.BlockManager(4, 0)
    assert bm.refcount(-1) == -1 and bm.refcount(8) == -1


@pytest.mark.parametrize("seed,prefix", [(1, True), (2, True), (3, False), (4, True)])
def test_random_workload_reads_back(seed, prefix, pkv):
    """Random admissions (prompts built from a few shared stems), decode
    steps with padding entries, frees and pool exhaustion."""
    rng = random.Random(seed)
    bs = rng.choice([1, 2, 4, 16])
    nb = rng.choice([8, 40, 120])
    bm = pkv.BlockManager(nb, bs, prefix_caching=prefix)
    m = Model(bm, nb, bs)
    stems = [[rng.randrange(50) for _ in range(rng.randrange(1, 5 * bs + 3))] for _ in range(4)]
    next_id, shared_seen = 0, 0
    for _ in range(300):
        op = rng.random()
        live = list(m.tokens)
        if op < 0.35 or not live:
            stem = rng.choice(stems)
            toks = stem[:rng.randrange(1, len(stem) + 1)] + \
                [rng.randrange(50) for _ in range(rng.randrange(0, 2 * bs + 1))]
            free_before = bm.stats()[0]
            try:
                cached = m.add(next_id, toks)
                shared_seen += cached > 0
            except pkv.PkvError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
                assert bm.stats()[0] == free_before
            next_id += 1
        elif op < 0.8:
            batch = rng.sample(live, rng.randrange(1, len(live) + 1))
            batch += [-1] * rng.randrange(0, 3)
            rng.shuffle(batch)
            try:
                m.append(batch, [rng.randrange(50) for _ in batch])
            except pkv.PkvError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
        else:
            m.free(rng.choice(live))
        m.check()
    if prefix:
        assert shared_seen > 0
    else:
        assert shared_seen == 0


def test_threads(pkv):
    """Several host threads admitting, appending and freeing their own
    sequences on one handle."""
    bm = pkv.BlockManager(4096, 16)
    errors = []

    def worker(k):
        try:
            rng = random.Random(k)
            for i in range(40):
                sid = k * 1000 + i
                toks = [rng.randrange(4) for _ in range(rng.randrange(1, 64))]
                bm.add_sequence(sid, toks)
                for _ in range(rng.randrange(0, 20)):
                    bm.append_tokens([sid], [rng.randrange(4)])
                n, table = bm.sequence_info(sid)
                assert len(table) == -(-n // 16)
                if rng.random() < 0.7:
                    bm.free_sequence(sid)
        except Exception as e:  # noqa: BLE001
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    free, _, live = bm.stats()
    used = set()
    for k in range(8):
        for i in range(40):
            try:
                used.update(bm.sequence_info(k * 1000 + i)[1])
            except pkv.PkvError:
                pass
    assert free == 4096 - len(used)
