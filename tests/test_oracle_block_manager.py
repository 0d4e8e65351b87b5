"""Pins of the block-manager reference model against things other than itself.

The main pin is a model of what the physical pool must hold: every slot a
sequence writes receives the identity of the KV that would be computed there
-- its position and the whole token prefix up to it (a KV vector depends on
both).  After every operation, reading any live sequence's positions through
its block table must give back exactly its own prefix identities: this fails
for a missed copy-on-write, a block shared or reused with the wrong content,
a false prefix-cache hit, or a slot computed from the wrong table entry.  The
other pins are the bookkeeping invariants (reference counts equal the number
of tables holding a block; every block is in use, cached-and-idle or free;
cache keys point at their blocks), hand-worked scenarios from the pages (a
second request sharing a 200-token system prompt; 8 sequences sharing a
13-block prefix), a copy-on-write and an eviction-order scenario, the FNV-1a
test vectors, and planted mistakes.
"""
from __future__ import annotations

import random

import pytest

from oracle import block_manager as BM

B = BM.BLOCK


class World:
    """A reference manager plus the physical pool model and each sequence's
    logical tokens."""

    def __init__(self, nb=64, max_blocks=64, max_seqs=16, mgr_cls=BM.BlockManagerRef):
        self.m = mgr_cls(nb, max_blocks, max_seqs)
        self.pool = [None] * (nb * B)
        self.tokens = {}

    @staticmethod
    def ident(tokens, p):
        return (p, tuple(tokens[:p + 1]))

    def add(self, seq, prompt):
        cached, slots = self.m.add_sequence(seq, list(prompt))
        self.tokens[seq] = list(prompt)
        for p in range(cached, len(prompt)):     # prefill writes only the uncached tail
            self.pool[slots[p]] = self.ident(prompt, p)
        self.check()
        return cached

    def append(self, seq, toks):
        slots, copies = self.m.append(seq, list(toks))
        for src, dst in copies:
            self.pool[dst * B:(dst + 1) * B] = self.pool[src * B:(src + 1) * B]
        for i, t in enumerate(toks):
            self.tokens[seq].append(t)
            self.pool[slots[i]] = self.ident(self.tokens[seq], len(self.tokens[seq]) - 1)
        self.check()
        return slots, copies

    def fork(self, parent, child):
        self.m.fork(parent, child)
        self.tokens[child] = list(self.tokens[parent])
        self.check()

    def free(self, seq):
        self.m.free_sequence(seq)
        del self.tokens[seq]
        self.check()

    def check(self):
        m = self.m
        for s, toks in self.tokens.items():
            table = m.table(s)
            assert m.length(s) == len(toks)
            for p in range(len(toks)):
                assert self.pool[table[p // B] * B + p % B] == self.ident(toks, p), (s, p)
        held = [0] * m.nb
        for s in self.tokens:
            for b in m.table(s):
                held[b] += 1
        assert held == m.ref
        for b in range(m.nb):
            states = [m.ref[b] > 0, b in m.lru, b in m.free]
            assert sum(states) == 1, (b, states)
        for k, b in m.cache.items():
            assert m.key[b] is not None and m.key[b][0] == k


def test_fnv1a_reference_vectors():
    # the published FNV-1a 64-bit test vectors
    assert BM.fnv1a64(b"") == 0xCBF29CE484222325
    assert BM.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert BM.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_second_request_sharing_a_200_token_system_prompt():
    """Block-granular reuse: 12 full blocks (192 of the 200 tokens) are cached;
    the 13th block mixes system and user tokens and is the second request's own."""
    w = World()
    sys_prompt = list(range(1000, 1200))
    assert w.add(0, sys_prompt + list(range(37))) == 0
    assert w.add(1, sys_prompt + list(range(50, 60))) == 192
    c = w.m.counts()
    assert c["hit_blocks"] == 12 and c["miss_blocks"] == 14 + 1
    assert w.m.table(1)[:12] == w.m.table(0)[:12] and w.m.table(1)[12] != w.m.table(0)[12]


def test_prefix_shared_by_8_sequences():
    w = World(nb=8 * 40, max_blocks=40, max_seqs=8)
    prefix = list(range(208))                    # 13 full blocks
    for s in range(8):
        w.add(s, prefix + [10_000 + s * 1000 + i for i in range(300)])
    c = w.m.counts()
    assert c["hit_blocks"] == 7 * 13
    assert c["used_blocks"] == 13 + 8 * ((208 + 300 + 15) // 16 - 13)


def test_copy_on_write_of_a_shared_partial_block():
    w = World()
    w.add(0, list(range(20)))                    # one full block + 4 tokens
    w.fork(0, 1)
    slots, copies = w.append(1, [77])
    assert len(copies) == 1 and copies[0][0] == w.m.table(0)[1]
    assert w.m.table(1)[0] == w.m.table(0)[0] and w.m.table(1)[1] != w.m.table(0)[1]
    slots, copies = w.append(0, [88])            # now the parent's block is its own
    assert copies == []
    assert w.m.counts()["cow_copies"] == 1


def test_eviction_takes_the_least_recently_released_cached_block():
    w = World(nb=6, max_blocks=6, max_seqs=6)
    w.add(0, list(range(32)))                    # blocks 0, 1 cached
    w.add(1, list(range(100, 132)))              # blocks 2, 3 cached
    w.free(1)                                    # released 3 then 2
    w.free(0)                                    # released 1 then 0
    w.add(2, list(range(200, 232)))              # free blocks 4, 5 first
    assert w.m.table(2) == [4, 5] and w.m.counts()["evictions"] == 0
    w.add(3, list(range(300, 316)))              # evicts block 3 (released first)
    assert w.m.table(3) == [3] and w.m.counts()["evictions"] == 1
    # the prefix of sequence 0 is still cached, the one of sequence 1 lost its last block
    assert w.add(4, list(range(32))) == 32


def test_out_of_blocks_changes_nothing():
    w = World(nb=4, max_blocks=8, max_seqs=4)
    w.add(0, list(range(40)))                    # 3 blocks
    before = (list(w.m.ref), set(w.m.free), dict(w.m.lru), w.m.counts())
    with pytest.raises(BM.NoBlocks):
        w.m.add_sequence(1, list(range(500, 540)))
    with pytest.raises(BM.NoBlocks):
        w.m.append(0, list(range(30)))
    assert (list(w.m.ref), set(w.m.free), dict(w.m.lru), w.m.counts()) == before
    w.check()


@pytest.mark.parametrize("seed", range(6))
def test_random_workloads_keep_every_sequence_intact(seed):
    rng = random.Random(seed)
    w = World(nb=96, max_blocks=24, max_seqs=12)
    prefixes = [[rng.randrange(50) for _ in range(rng.choice([16, 40, 64]))] for _ in range(3)]
    live = []
    for _ in range(300):
        op = rng.random()
        try:
            if op < 0.25 and len(live) < 12:
                s = next(i for i in range(12) if i not in live)
                pre = rng.choice(prefixes)[:rng.randrange(1, 65)]
                w.add(s, pre + [rng.randrange(50) for _ in range(rng.randrange(0, 40))])
                live.append(s)
            elif op < 0.65 and live:
                s = rng.choice(live)
                w.append(s, [rng.randrange(50) for _ in range(rng.randrange(1, 20))])
            elif op < 0.8 and live and len(live) < 12:
                s = rng.choice(live)
                c = next(i for i in range(12) if i not in live)
                w.fork(s, c)
                live.append(c)
            elif live:
                s = rng.choice(live)
                w.free(s)
                live.remove(s)
        except (BM.NoBlocks, ValueError):
            w.check()
    assert w.m.counts()["hit_blocks"] > 0 and w.m.counts()["cow_copies"] > 0


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

class NoCow(BM.BlockManagerRef):
    """Appends into the last block even when another table holds it."""
    def append(self, seq, tokens):
        s = self.seqs[seq]
        slots = []
        for tok in tokens:
            p = s["len"]
            if p % B == 0:
                s["table"].append(self._alloc())
                s["tail"] = []
            slots.append(s["table"][-1] * B + p % B)
            s["tail"].append(tok)
            s["len"] = p + 1
            if s["len"] % B == 0:
                s["parent"] = self._register(s["table"][-1], s["parent"], s["tail"])
                s["tail"] = []
        return slots, []


class NoParentInKey(BM.BlockManagerRef):
    def _lookup(self, parent, tokens):
        for b, k in enumerate(self.key):
            if k is not None and list(k[2]) == list(tokens) and self.cache.get(k[0]) == b:
                return b
        return None


class ForwardRelease(BM.BlockManagerRef):
    def free_sequence(self, seq):
        self.seqs[seq]["table"].reverse()
        super().free_sequence(seq)


def test_planted_missing_copy_on_write_is_caught():
    with pytest.raises(AssertionError):
        w = World(mgr_cls=NoCow)
        w.add(0, list(range(20)))
        w.fork(0, 1)
        w.append(1, [77])
        w.append(0, [88])      # both now wrote position 20 into the same slot


def test_planted_key_without_parent_is_caught():
    with pytest.raises(AssertionError):
        w = World(mgr_cls=NoParentInKey)
        w.add(0, list(range(16)) + list(range(500, 516)))
        w.add(1, list(range(500, 516)) + [1, 2, 3])   # its first block equals seq 0's second block


def test_planted_forward_release_order_is_caught():
    with pytest.raises(AssertionError):
        w = World(nb=6, max_blocks=6, max_seqs=6, mgr_cls=ForwardRelease)
        test_eviction_order_scenario(w)


def test_eviction_order_scenario(w=None):
    w = w or World(nb=6, max_blocks=6, max_seqs=6)
    w.add(0, list(range(32)))
    w.add(1, list(range(100, 132)))
    w.free(1)
    w.free(0)
    w.add(2, list(range(200, 232)))
    w.add(3, list(range(300, 316)))
    assert w.m.table(3) == [3]


def test_append_step_equals_single_appends_and_is_all_or_nothing():
    w1, w2 = World(nb=12, max_blocks=8, max_seqs=6), World(nb=12, max_blocks=8, max_seqs=6)
    for w in (w1, w2):
        w.add(0, list(range(20)))
        w.fork(0, 1)
        w.fork(0, 2)                               # three tables share the partial block
    slots, copies = w1.m.append_step([1, 2, 0], [7, 8, 9])
    singles = [w2.m.append(s, [t]) for s, t in ((1, 7), (2, 8), (0, 9))]
    assert slots == [x for sl, _ in singles for x in sl] and copies == [c for _, cp in singles for c in cp]
    assert len(copies) == 2                        # the last of the three keeps the block
    w = World(nb=4, max_blocks=8, max_seqs=4)
    w.add(0, list(range(16)))
    w.add(1, list(range(100, 116)))
    w.add(2, list(range(200, 216)))
    before = (list(w.m.ref), set(w.m.free), w.m.counts())
    with pytest.raises(BM.NoBlocks):               # three new blocks needed, one free
        w.m.append_step([0, 1, 2], [1, 2, 3])
    assert (list(w.m.ref), set(w.m.free), w.m.counts()) == before
