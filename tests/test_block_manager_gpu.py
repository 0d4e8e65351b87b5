"""The block manager driving the GPU path end to end.

K/V vectors are a deterministic function of the token prefix they belong to
(as a model's would be), so sequences that share a prompt prefix share
identical K/V.  Sequences are started through the manager (the prefix cache
decides which prompt tokens need prefilling), forked, and extended (with the
copy-on-write pairs copied by pa_copy_blocks); only the tokens the manager
says are new are written into the pool.  Decode over the manager's block
tables must then equal the oracle's attention over each sequence's own
logical cache, built without any paging."""
from __future__ import annotations

import hashlib

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
HKV, HQ, D = 4, 16, 128


def kv_of(prefix):
    """K and V rows [H_kv][D] of the last token of `prefix` (bf16-exact floats)."""
    seed = int.from_bytes(hashlib.sha256(np.asarray(prefix, np.int64).tobytes()).digest()[:8], "little")
    g = torch.Generator().manual_seed(seed % (1 << 63))
    kv = torch.randn((2, HKV, D), generator=g).to(torch.bfloat16)
    return kv[0], kv[1]


class Engine:
    def __init__(self, nb=256, mb=64, ms=8):
        self.bm = pa.pa_bm_create(nb, mb, ms)
        self.mb = mb
        self.kp = torch.zeros((nb, HKV, 16, D), dtype=torch.bfloat16, device=DEV)
        self.vp = torch.zeros_like(self.kp)
        self.tokens = {}

    def write(self, seq, first, slots):
        """K/V of positions first.. of `seq` into the given slots."""
        toks = self.tokens[seq]
        ks, vs = zip(*[kv_of(toks[:p + 1]) for p in range(first, len(toks))])
        pa.pa_append_kv(self.kp, self.vp, torch.as_tensor(np.asarray(slots, np.int64), device=DEV),
                        torch.stack(ks).to(DEV), torch.stack(vs).to(DEV))

    def add(self, seq, prompt):
        self.tokens[seq] = list(prompt)
        cached, slots = pa.pa_bm_add_sequence(self.bm, seq, prompt)
        if cached < len(prompt):
            self.write(seq, cached, slots[cached:])
        return cached

    def append(self, seq, toks):
        slots, copies = pa.pa_bm_append(self.bm, seq, toks)
        if copies:
            pa.pa_copy_blocks(self.kp, self.vp, torch.tensor(copies, dtype=torch.int32, device=DEV))
        first = len(self.tokens[seq])
        self.tokens[seq] += list(toks)
        self.write(seq, first, slots)
        return copies

    def fork(self, parent, child):
        pa.pa_bm_fork(self.bm, parent, child)
        self.tokens[child] = list(self.tokens[parent])

    def decode_vs_oracle(self, seqs, what):
        tables, ctx = pa.pa_bm_block_tables(self.bm, seqs, self.mb)
        g = torch.Generator().manual_seed(len(seqs))
        q = torch.randn((len(seqs), HQ, D), generator=g).to(torch.bfloat16)
        out = torch.empty((len(seqs), HQ, D), dtype=torch.bfloat16, device=DEV)
        pa.pa_decode_attention(out, q.to(DEV), self.kp, self.vp, torch.from_numpy(tables).to(DEV),
                               torch.from_numpy(ctx).to(DEV), 1.0 / np.sqrt(D), max_context_len=int(ctx.max()))
        torch.cuda.synchronize()
        ref = np.zeros((len(seqs), HQ, D))
        for i, s in enumerate(seqs):
            toks = self.tokens[s]
            assert ctx[i] == len(toks)
            kv = [kv_of(toks[:p + 1]) for p in range(len(toks))]
            k = torch.stack([a for a, _ in kv]).to(torch.float64).numpy()
            v = torch.stack([b for _, b in kv]).to(torch.float64).numpy()
            ref[i] = oracle.attend(q[i].to(torch.float64).numpy(), k, v, 1.0 / np.sqrt(D), len(toks))
        assert_close_to_ref(out, ref, torch.bfloat16, what)


def test_shared_system_prompt_fork_and_copy_on_write():
    e = Engine()
    system = list(range(1000, 1200))                      # 200 tokens: 12 full blocks cached
    assert e.add(0, system + list(range(37))) == 0
    assert e.add(1, system + list(range(50, 60))) == 192
    assert e.add(2, system + list(range(70, 75))) == 192
    e.decode_vs_oracle([0, 1, 2], "after prompts")
    e.fork(1, 3)                                          # shares sequence 1's partial last block
    assert e.append(3, [9]) != []                         # copy-on-write before writing
    assert e.append(1, [8, 7]) == []
    for s in (0, 1, 2, 3):
        e.append(s, list(range(s * 10, s * 10 + 21)))     # cross block boundaries
    e.decode_vs_oracle([0, 1, 2, 3], "after appends")
    st = pa.pa_bm_get_stats(e.bm)
    assert st["hit_blocks"] == 24 and st["cow_copies"] == 1
    assert pa.pa_device_status() == 0
    pa.pa_bm_destroy(e.bm)


def test_eviction_reuses_blocks_without_corrupting_live_sequences():
    e = Engine(nb=40, mb=20, ms=8)
    for s in range(3):                                     # fill, then release two sequences
        e.add(s, list(range(s * 500, s * 500 + 150)))
    pa.pa_bm_free_sequence(e.bm, 1)
    pa.pa_bm_free_sequence(e.bm, 2)
    del e.tokens[1], e.tokens[2]
    e.add(4, list(range(0, 150)))                          # sequence 0's prompt: fully cached
    e.add(5, list(range(9000, 9200)))                      # needs evictions
    assert pa.pa_bm_get_stats(e.bm)["evictions"] > 0
    e.decode_vs_oracle([0, 4, 5], "after evictions")
    pa.pa_bm_destroy(e.bm)


def test_copy_blocks_is_bit_exact_and_checks_ids():
    g = torch.Generator().manual_seed(7)
    kp = torch.randn((10, 2, 16, 64), generator=g).to(torch.bfloat16)
    vp = torch.randn((10, 2, 16, 64), generator=g).to(torch.bfloat16)
    kd, vd = kp.to(DEV), vp.to(DEV)
    pa.pa_copy_blocks(kd, vd, torch.tensor([[1, 7], [4, 2]], dtype=torch.int32, device=DEV))
    want_k, want_v = kp.clone(), vp.clone()
    want_k[7], want_v[7], want_k[2], want_v[2] = kp[1], vp[1], kp[4], vp[4]
    assert torch.equal(kd.cpu(), want_k) and torch.equal(vd.cpu(), want_v)
    assert pa.pa_device_status() == 0
    pa.pa_copy_blocks(kd, vd, torch.tensor([[1, 12]], dtype=torch.int32, device=DEV))
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID


class Int8Engine(Engine):
    """The same engine over an INT8 cache: K/V rows are quantised on append
    (pa_append_kv_int8) and copy-on-write copies code blocks and their scale
    rows (pa_copy_blocks_int8).  A host mirror of the four arrays follows every
    operation through the oracle: oracle.append_int8_ref for the writes, and a
    plain copy of the block's rows in all four arrays for each copy-on-write
    pair (what copying a block means)."""

    def __init__(self, nb=256, mb=64, ms=8):
        self.bm = pa.pa_bm_create(nb, mb, ms)
        self.mb = mb
        self.kp = torch.zeros((nb, HKV, 16, D), dtype=torch.int8, device=DEV)
        self.vp = torch.zeros_like(self.kp)
        self.ks = torch.zeros((nb, HKV, 16), dtype=torch.float32, device=DEV)
        self.vs = torch.zeros_like(self.ks)
        self.host = [np.zeros((nb, HKV, 16, D), np.int8), np.zeros((nb, HKV, 16, D), np.int8),
                     np.zeros((nb, HKV, 16), np.float32), np.zeros((nb, HKV, 16), np.float32)]
        self.tokens = {}

    def write(self, seq, first, slots):
        toks = self.tokens[seq]
        ks, vs = zip(*[kv_of(toks[:p + 1]) for p in range(first, len(toks))])
        kn, vn = torch.stack(ks), torch.stack(vs)
        sl = np.asarray(slots, np.int64)
        pa.pa_append_kv_int8(self.kp, self.vp, self.ks, self.vs, torch.as_tensor(sl, device=DEV), kn.to(DEV),
                             vn.to(DEV))
        self.host = list(oracle.append_int8_ref(*self.host, sl, to_np(kn), to_np(vn)))

    def append(self, seq, toks):
        slots, copies = pa.pa_bm_append(self.bm, seq, toks)
        if copies:
            pa.pa_copy_blocks_int8(self.kp, self.vp, self.ks, self.vs,
                                   torch.tensor(copies, dtype=torch.int32, device=DEV))
            for src, dst in copies:
                for a in self.host:
                    a[dst] = a[src]
        first = len(self.tokens[seq])
        self.tokens[seq] += list(toks)
        self.write(seq, first, slots)
        return copies

    def check(self, seqs, what):
        torch.cuda.synchronize()
        got = [to_np(self.kp), to_np(self.vp), self.ks.cpu().numpy(), self.vs.cpu().numpy()]
        assert all(np.array_equal(g.view(np.uint8), h.view(np.uint8)) for g, h in zip(got, self.host)), what
        tables, ctx = pa.pa_bm_block_tables(self.bm, seqs, self.mb)
        # every live sequence reads back, through its own table, the codes and
        # scales of its own tokens (nothing overwritten a shared block)
        for i, s in enumerate(seqs):
            toks = self.tokens[s]
            kv = [kv_of(toks[:p + 1]) for p in range(len(toks))]
            qk, sk = oracle.quantize_rows_int8(to_np(torch.stack([a for a, _ in kv])))
            qv, sv = oracle.quantize_rows_int8(to_np(torch.stack([b for _, b in kv])))
            for p in range(len(toks)):
                blk, off = int(tables[i, p // 16]), p % 16
                assert np.array_equal(got[0][blk, :, off], qk[p]) and np.array_equal(got[1][blk, :, off], qv[p])
                assert np.array_equal(got[2][blk, :, off], sk[p]) and np.array_equal(got[3][blk, :, off], sv[p])
        g = torch.Generator().manual_seed(len(seqs))
        q = torch.randn((len(seqs), HQ, D), generator=g).to(torch.bfloat16)
        out = torch.empty((len(seqs), HQ, D), dtype=torch.bfloat16, device=DEV)
        pa.pa_decode_attention_int8(out, q.to(DEV), self.kp, self.vp, self.ks, self.vs,
                                    torch.from_numpy(tables).to(DEV), torch.from_numpy(ctx).to(DEV),
                                    1.0 / np.sqrt(D), max_context_len=int(ctx.max()))
        torch.cuda.synchronize()
        ref = oracle.decode_int8_ref(to_np(q), *self.host, tables, ctx, 1.0 / np.sqrt(D))
        assert_close_to_ref(out, ref, torch.bfloat16, what)


def test_int8_cache_fork_and_copy_on_write():
    """Prefix sharing over an INT8 cache: a fork shares a partly filled last
    block, the next append copies it first (codes and scale rows), and every
    sequence keeps reading its own tokens' codes and scales; decode over the
    manager's tables matches the oracle over the mirrored cache."""
    e = Int8Engine()
    system = list(range(1000, 1200))
    assert e.add(0, system + list(range(37))) == 0
    assert e.add(1, system + list(range(50, 60))) == 192
    e.check([0, 1], "int8 after prompts")
    e.fork(1, 2)
    assert e.append(2, [9]) != []                         # copy-on-write of the shared last block
    assert e.append(1, [8, 7]) == []
    for s in (0, 1, 2):
        e.append(s, list(range(s * 10, s * 10 + 21)))
    e.check([0, 1, 2], "int8 after fork and appends")
    assert pa.pa_bm_get_stats(e.bm)["cow_copies"] == 1
    assert pa.pa_device_status() == 0
    pa.pa_bm_destroy(e.bm)


def test_copy_blocks_int8_is_bit_exact_and_checks_ids():
    g = torch.Generator().manual_seed(8)
    kc = torch.randint(-127, 128, (10, 2, 16, 64), generator=g, dtype=torch.int16).to(torch.int8)
    vc = torch.randint(-127, 128, (10, 2, 16, 64), generator=g, dtype=torch.int16).to(torch.int8)
    ks, vs = torch.rand((10, 2, 16), generator=g), torch.rand((10, 2, 16), generator=g)
    d = [t.to(DEV) for t in (kc, vc, ks, vs)]
    pa.pa_copy_blocks_int8(*d, torch.tensor([[1, 7], [4, 2]], dtype=torch.int32, device=DEV))
    for got, src in zip(d, (kc, vc, ks, vs)):
        want = src.clone()
        want[7], want[2] = src[1], src[4]
        assert torch.equal(got.cpu(), want)
    assert pa.pa_device_status() == 0
    pa.pa_copy_blocks_int8(*d, torch.tensor([[1, 12]], dtype=torch.int32, device=DEV))
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID
