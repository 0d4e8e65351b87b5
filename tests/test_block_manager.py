"""The library's block manager (host C++) against the reference model.

Both follow the same deterministic policies, so on any sequence of calls they
must agree exactly: every slot, every block table, every copy-on-write pair,
every counter, and every call that runs out of blocks.  Runs on the CPU (the
manager is host code in the library)."""
from __future__ import annotations

import random

import numpy as np
import pytest

from oracle import block_manager as BM
from paged_kv_decode_27_gb300 import binding as pa


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_27_gb300 import build
    build.build()
    return pa.load_library()


class Pair:
    def __init__(self, nb, mb, ms):
        self.ref = BM.BlockManagerRef(nb, mb, ms)
        self.bm = pa.pa_bm_create(nb, mb, ms)
        self.mb = mb

    def close(self):
        pa.pa_bm_destroy(self.bm)

    def same(self, live):
        if live:
            tables, ctx = pa.pa_bm_block_tables(self.bm, live, self.mb)
            for i, s in enumerate(live):
                t = self.ref.table(s)
                assert list(tables[i, :len(t)]) == t and not tables[i, len(t):].any()
                assert ctx[i] == self.ref.length(s)
        got = pa.pa_bm_get_stats(self.bm)
        want = self.ref.counts()
        for k in want:
            assert got[k] == want[k], (k, got[k], want[k])

    def add(self, seq, prompt):
        try:
            want = self.ref.add_sequence(seq, prompt)
        except BM.NoBlocks:
            with pytest.raises(pa.PaError) as e:
                pa.pa_bm_add_sequence(self.bm, seq, prompt)
            assert e.value.code == pa.PA_ERR_NO_BLOCKS
            return False
        cached, slots = pa.pa_bm_add_sequence(self.bm, seq, prompt)
        assert cached == want[0] and list(slots) == want[1]
        return True

    def append(self, seq, toks):
        try:
            want = self.ref.append(seq, toks)
        except BM.NoBlocks:
            with pytest.raises(pa.PaError) as e:
                pa.pa_bm_append(self.bm, seq, toks)
            assert e.value.code == pa.PA_ERR_NO_BLOCKS
            return
        slots, copies = pa.pa_bm_append(self.bm, seq, toks)
        assert list(slots) == want[0] and copies == want[1]


def test_pages_scenarios_match(lib):
    p = Pair(64, 64, 8)
    sys_prompt = list(range(1000, 1200))
    assert p.add(0, sys_prompt + list(range(37)))
    assert p.add(1, sys_prompt + list(range(50, 60)))
    p.same([0, 1])
    pa.pa_bm_fork(p.bm, 1, 2)
    p.ref.fork(1, 2)
    p.append(2, [5])                      # copy-on-write of the shared partial block
    p.append(1, [6, 7, 8])
    p.same([0, 1, 2])
    assert pa.pa_bm_get_stats(p.bm)["cow_copies"] == 1
    p.close()


@pytest.mark.parametrize("seed", range(8))
def test_random_call_sequences_match(lib, seed):
    rng = random.Random(100 + seed)
    nb, mb, ms = rng.choice([(48, 16, 10), (96, 24, 12), (30, 12, 8)])
    p = Pair(nb, mb, ms)
    prefixes = [[rng.randrange(40) for _ in range(rng.choice([16, 33, 64]))] for _ in range(3)]
    live = []
    for _ in range(400):
        op = rng.random()
        if op < 0.25 and len(live) < ms:
            s = next(i for i in range(ms) if i not in live)
            prompt = rng.choice(prefixes)[:rng.randrange(1, 65)] + [rng.randrange(40) for _ in range(rng.randrange(30))]
            if (len(prompt) + 15) // 16 <= mb and p.add(s, prompt):
                live.append(s)
        elif op < 0.65 and live:
            s = rng.choice(live)
            toks = [rng.randrange(40) for _ in range(rng.randrange(1, 20))]
            if (p.ref.length(s) + len(toks) + 15) // 16 <= mb:
                p.append(s, toks)
        elif op < 0.72 and live:
            step = rng.sample(live, rng.randrange(1, len(live) + 1))
            toks = [rng.randrange(40) for _ in step]
            if all((p.ref.length(s) + 16) // 16 <= mb for s in step):
                try:
                    want = p.ref.append_step(step, toks)
                except BM.NoBlocks:
                    with pytest.raises(pa.PaError) as e:
                        pa.pa_bm_append_step(p.bm, step, toks)
                    assert e.value.code == pa.PA_ERR_NO_BLOCKS
                else:
                    slots, copies = pa.pa_bm_append_step(p.bm, step, toks)
                    assert list(slots[:len(step)]) == want[0] and copies == want[1]
        elif op < 0.8 and live and len(live) < ms:
            s = rng.choice(live)
            c = next(i for i in range(ms) if i not in live)
            p.ref.fork(s, c)
            pa.pa_bm_fork(p.bm, s, c)
            live.append(c)
        elif live:
            s = rng.choice(live)
            p.ref.free_sequence(s)
            pa.pa_bm_free_sequence(p.bm, s)
            live.remove(s)
        p.same(live)
    st = pa.pa_bm_get_stats(p.bm)
    assert st["hit_blocks"] > 0
    p.close()


def test_host_validation(lib):
    bm = pa.pa_bm_create(8, 4, 2)
    with pytest.raises(pa.PaError):
        pa.pa_bm_add_sequence(bm, 5, [1, 2])             # id out of range
    with pytest.raises(pa.PaError):
        pa.pa_bm_add_sequence(bm, 0, list(range(80)))    # longer than the table
    pa.pa_bm_add_sequence(bm, 0, [1, 2, 3])
    with pytest.raises(pa.PaError):
        pa.pa_bm_add_sequence(bm, 0, [1])                # already live
    with pytest.raises(pa.PaError):
        pa.pa_bm_append(bm, 1, [1])                      # not live
    with pytest.raises(pa.PaError):
        pa.pa_bm_fork(bm, 0, 0)
    pa.pa_bm_free_sequence(bm, 0)
    with pytest.raises(pa.PaError):
        pa.pa_bm_free_sequence(bm, 0)
    pa.pa_bm_destroy(bm)
    with pytest.raises(pa.PaError):
        pa.pa_bm_create(0, 4, 2)
