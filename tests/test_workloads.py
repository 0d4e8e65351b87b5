"""Structure of the seeded synthetic workloads (CPU only)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from paged_kv_decode_27_gb300 import workloads as W


def _used_blocks(wl: W.Workload, rows, ctx):
    bt = wl.block_tables[rows]
    used = []
    for s in range(bt.shape[0]):
        nb = (int(ctx[s]) + 15) // 16
        used.append(bt[s, :nb].tolist())
    return used


def test_tiny_layout():
    wl = W.tiny_fp32()
    assert wl.k_pool.shape == (16, 2, 16, 64) and wl.k_pool.dtype == torch.float32
    assert wl.ctx0.tolist() == [17, 40]
    used = _used_blocks(wl, wl.decode_rows, wl.ctx0)
    assert [len(u) for u in used] == [2, 3]
    flat = sum(used, [])
    assert len(set(flat)) == 5 and all(0 <= b < 16 for b in flat)
    assert wl.scale == 1.0 / 8.0
    st = wl.step(0)
    # the appended token is the last position of each sequence
    for s, c in enumerate([17, 40]):
        slot = int(st.slot_mapping[s])
        assert slot // 16 == used[s][(c - 1) // 16] and slot % 16 == (c - 1) % 16


def test_step_determinism():
    a = W.tiny_fp32().step(0)
    b = W.tiny_fp32().step(0)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_new, b.k_new)
    assert torch.equal(a.slot_mapping, b.slot_mapping)


@pytest.mark.slow
def test_llama3_8b_shape_and_pool():
    wl = W.llama3_8b_decode()
    assert (wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.num_decode_seqs) == (32, 8, 128, 64)
    c = wl.ctx0
    assert int(c.min()) >= 512 and int(c.max()) <= 8192
    # log-uniform: the median sits near the geometric mean 2048
    assert 1000 < float(c.float().median()) < 4000
    need = sum((int(x) + wl.steps - 1 + 15) // 16 for x in c)
    assert wl.num_blocks == math.ceil(1.25 * need)
    flat = sum(_used_blocks(wl, wl.decode_rows, c + wl.steps - 1), [])
    assert len(set(flat)) == len(flat), "private blocks must not be shared"
    # pool bytes: [N][8][16][128] bf16 = 32 KiB per block for K
    assert wl.k_pool.element_size() * wl.k_pool[0].numel() == 32 * 1024
    last = wl.step(wl.steps - 1)
    assert torch.equal(last.context_lens, (c + wl.steps - 1).to(torch.int32))


@pytest.mark.slow
def test_prefix_shared_tables():
    wl = W.prefix_shared_8k()
    bt = wl.block_tables
    assert bt.shape == (8, 512)
    assert (bt[:, :13] == bt[0, :13]).all()
    priv = bt[:, 13:].reshape(-1).tolist()
    assert len(set(priv)) == len(priv)
    assert not set(priv) & set(bt[0, :13].tolist())
    st = wl.step(0)
    # the appended token lands in a private block
    assert all(int(s) // 16 in set(priv) for s in st.slot_mapping)


@pytest.mark.slow
def test_mixed_step_slots_cover_prompts_then_decodes():
    wl = W.mixed_mistral7b()
    st = wl.step(0)
    assert st.slot_mapping.numel() == 512 + 1024 + 1536 + 2048 + 60
    assert st.cu_q_lens.tolist() == [0, 512, 1536, 3072, 5120]
    assert st.q_prefill.shape == (5120, 32, 128) and st.q.shape == (60, 32, 128)
    assert len(set(st.slot_mapping.tolist())) == st.slot_mapping.numel()
    assert int(wl.ctx0.min()) >= 256 and int(wl.ctx0.max()) <= 4096


def test_small_random_zero_context_skips_append():
    wl = W.small_random(1, 3, 10, 4, 2, 8, ctx=[3, 0, 9])
    st = wl.step(0)
    assert int(st.slot_mapping[1]) == -1
    assert int(st.slot_mapping[0]) >= 0 and int(st.slot_mapping[2]) >= 0


def test_byte_accounting():
    wl = W.tiny_fp32()
    # KV: (17+40) tokens * 2 (K,V) * 2 heads * 64 * 4 B; q,out: 2*2*4*64*4; ids: 5 blocks + 2 lens
    assert wl.decode_bytes(0) == 57 * 2 * 2 * 64 * 4 + 2 * 2 * 4 * 64 * 4 + 4 * 5 + 4 * 2


def test_int8_cache_draw():
    wl = W.small_random(3, 4, 300, 8, 2, 64, kv="int8")
    assert wl.kv_int8 and wl.k_pool.dtype == torch.int8 and wl.v_pool.dtype == torch.int8
    assert wl.k_scales.shape == wl.k_pool.shape[:3] and wl.k_scales.dtype == torch.float32
    assert int(wl.k_pool.min()) >= -127 and int(wl.k_pool.max()) <= 127
    assert float(wl.k_scales.min()) >= 2.0 / 127 and float(wl.v_scales.max()) <= 4.0 / 127
    # the same tables and step draws as the float cache of the same seed
    wf = W.small_random(3, 4, 300, 8, 2, 64)
    assert torch.equal(wf.block_tables, wl.block_tables) and torch.equal(wf.ctx0, wl.ctx0)
    assert torch.equal(wf.step(0).q, wl.step(0).q) and wl.step(0).k_new.dtype == torch.bfloat16
    # bytes: D codes + a 4-byte scale per (token, head) row, for K and V
    ctx = wl.ctx0.to(torch.int64)
    assert wl.decode_bytes(0) == (int(ctx.sum()) * 2 * 2 * (64 + 4) + 2 * 4 * 8 * 64 * 2
                                  + 4 * int(((ctx + 15) // 16).sum()) + 4 * 4)
