"""pa_verify_attention (speculative-decoding verification, q_len query
positions per sequence, causal) on the GPU against the float64 oracle.

The oracle is the prompt-pass definition over a cached prefix: query i of a
sequence with context c and q_len n sits at position c - n + i and sees keys
0 .. c - n + i.  Bar: |gpu - ref| <= 2e-2 + 1e-2 |ref| (bf16/fp16 inputs)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, fill_unused_with_nan, run_decode
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu


def _verify(wl, q, ctx, part=0, kp=None, vp=None):
    kp = wl.k_pool.to(DEV) if kp is None else kp
    vp = wl.v_pool.to(DEV) if vp is None else vp
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    pa.pa_verify_attention(out, q.to(DEV), kp, vp, wl.decode_block_tables.contiguous().to(DEV), ctx.to(DEV),
                           wl.scale, max_context_len=int(ctx.max()), partition_size=part)
    torch.cuda.synchronize()
    return out


def _ref(wl, q, ctx, seqs=None):
    S, n = q.shape[0], q.shape[1]
    cu = np.arange(S + 1) * n
    rows = None if seqs is None else [s * n + i for s in seqs for i in range(n)]
    r = oracle.prefill_ref(to_np(q.reshape(S * n, q.shape[2], q.shape[3])), to_np(wl.k_pool), to_np(wl.v_pool),
                           wl.decode_block_tables.contiguous().numpy(), cu, ctx.numpy(), wl.scale, rows=rows)
    return r.reshape(q.shape)


@pytest.mark.parametrize("hq,hkv,q_len,d,dtype", [
    (32, 8, 5, 128, torch.bfloat16),    # G 4 x 5 positions: 20 columns (three 8-column tiles)
    (32, 4, 4, 128, torch.bfloat16),    # G 8 x 4: 32 columns (four tiles)
    (8, 8, 5, 128, torch.float16),      # G 1 x 5: one tile
    (16, 8, 5, 128, torch.bfloat16),    # G 2 x 5: 10 columns (the 16-column tensor-core kernel)
    (32, 8, 2, 128, torch.bfloat16),    # G 4 x 2: 8 columns, the narrowest softmax
    (32, 8, 8, 128, torch.float16),     # G 4 x 8: 32 columns
    (16, 8, 5, 64, torch.bfloat16),     # G 2 x 5: two tiles, D 64
    (12, 4, 8, 64, torch.float16),      # G 3 x 8: 24 columns, D 64
    (32, 8, 1, 128, torch.bfloat16),    # q_len 1 is decode
])
def test_verify_shapes(hq, hkv, q_len, d, dtype):
    wl = W.small_random(90 + hq + q_len + d, 5, 600, hq, hkv, d, dtype)
    ctx = wl.ctx0.clamp(min=q_len)
    q = wl.verify_queries(0, q_len)
    ref = _ref(wl, q, ctx)
    for part in (0, 16, 64, 512):
        out = _verify(wl, q, ctx, part)
        assert_close_to_ref(out, ref, dtype, f"verify G={hq // hkv} q_len={q_len} part={part}")
    assert pa.pa_device_status() == 0


@pytest.mark.parametrize("ctx", [[5, 6, 15, 16, 17, 20, 21], [31, 32, 33, 64, 65, 255, 256, 257]])
def test_verify_ragged_contexts(ctx):
    """The causal edge falls at every offset of a 16-token block, and at block
    and partition boundaries."""
    wl = W.small_random(97, len(ctx), 0, 32, 8, 128, torch.bfloat16, ctx=ctx)
    ctx_t = torch.tensor(ctx, dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    ref = _ref(wl, q, ctx_t)
    for part in (0, 16, 32):
        assert_close_to_ref(_verify(wl, q, ctx_t, part), ref, wl.dtype, f"verify ragged part={part}")


def test_verify_q_len_1_is_decode_bit_for_bit():
    wl = W.small_random(98, 6, 900, 32, 8, 128, torch.bfloat16)
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    for part in (0, 64):
        dec = run_decode(wl, st, kp, vp, partition_size=part)
        ver = _verify(wl, st.q.unsqueeze(1), st.context_lens, part, kp, vp)
        assert torch.equal(ver[:, 0], dec)


def test_verify_rows_match_decode_at_each_position():
    """Consistency check, not parity evidence (both sides are GPU paths): row i
    of a verification pass equals a decode of the same query with the context
    cut at its position, within the bf16 bar.  Parity of each path against the
    oracle is tested separately."""
    wl = W.small_random(99, 3, 0, 32, 8, 128, torch.bfloat16, ctx=[40, 130, 700])
    ctx = torch.tensor([40, 130, 700], dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    ver = _verify(wl, q, ctx)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    for i in range(5):
        st = W.StepInputs(slot_mapping=torch.full((3,), -1, dtype=torch.int64),
                          k_new=torch.empty((3, 8, 128), dtype=torch.bfloat16),
                          v_new=torch.empty((3, 8, 128), dtype=torch.bfloat16),
                          q=q[:, i].contiguous(), context_lens=ctx - 5 + i + 1)
        dec = run_decode(wl, st, kp, vp)
        assert torch.max(torch.abs(dec.float() - ver[:, i].float())).item() < 2e-2


def test_verify_stale_slots_never_leak():
    wl = W.small_random(100, 5, 300, 32, 8, 128, torch.bfloat16)
    ctx = wl.ctx0.clamp(min=5)
    fill_unused_with_nan(wl, ctx)
    q = wl.verify_queries(0, 5)
    ref = _ref(wl, q, ctx)
    assert np.isfinite(ref).all()
    for part in (0, 16):
        out = _verify(wl, q, ctx, part)
        assert torch.isfinite(out.float()).all()
        assert_close_to_ref(out, ref, wl.dtype, f"verify NaN canary part={part}")


def test_verify_short_contexts_give_zero_leading_rows():
    """A context shorter than q_len: the queries before position 0 see no key."""
    wl = W.small_random(101, 3, 0, 8, 2, 64, torch.bfloat16, ctx=[3, 0, 9])
    ctx = torch.tensor([3, 0, 9], dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    out = _verify(wl, q, ctx)
    assert int(out[0, :2].count_nonzero()) == 0 and int(out[1].count_nonzero()) == 0
    assert_close_to_ref(out, _ref(wl, q, ctx), wl.dtype, "short contexts")


def test_verify_llama3_8b_full_size():
    """Batch 64, D 128, K = 4 drafts (q_len 5) in the benchmark's launch
    configuration (automatic partition): every row against the oracle."""
    wl = W.llama3_8b_decode(steps=1)
    ctx = wl.ctx0
    q = wl.verify_queries(0, 5)
    out = _verify(wl, q, ctx)
    ref = _ref(wl, q, ctx)
    assert_close_to_ref(out, ref, wl.dtype, "verify llama3-8b")
    assert pa.pa_device_status() == 0


def test_verify_d128_empty_and_short_contexts():
    """Head dim 128 (the tensor-core kernel): a context of 0 owns no tile and
    its rows are zero; a context shorter than q_len zeroes the leading rows."""
    ctx_l = [3, 0, 9, 0, 130, 1]
    wl = W.small_random(102, len(ctx_l), 0, 32, 8, 128, torch.bfloat16, ctx=ctx_l)
    ctx = torch.tensor(ctx_l, dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    out = _verify(wl, q, ctx)
    assert int(out[1].count_nonzero()) == 0 and int(out[3].count_nonzero()) == 0
    assert int(out[0, :2].count_nonzero()) == 0 and int(out[5, :4].count_nonzero()) == 0
    assert_close_to_ref(out, _ref(wl, q, ctx), wl.dtype, "empty and short contexts, D 128")
    assert pa.pa_device_status() == 0


@pytest.mark.parametrize("part", [0, 128, 1024])
def test_verify_many_segments_per_cta(part):
    """Ninety mostly short sequences: every CTA of the persistent launch walks
    many (sequence, KV head) segments, long ones are split over several CTAs
    and merged."""
    g = torch.Generator().manual_seed(7)
    ctx_l = [int(x) for x in torch.randint(1, 400, (88,), generator=g)] + [3000, 5000]
    wl = W.small_random(103, len(ctx_l), 0, 32, 8, 128, torch.bfloat16, ctx=ctx_l)
    ctx = torch.tensor(ctx_l, dtype=torch.int32).clamp(min=5)
    q = wl.verify_queries(0, 5)
    out = _verify(wl, q, ctx, part)
    ref = _ref(wl, q, ctx)
    assert_close_to_ref(out, ref, wl.dtype, f"many segments part={part}")
    assert pa.pa_device_status() == 0


def test_verify_d128_bad_block_id_is_reported():
    wl = W.small_random(104, 3, 0, 32, 8, 128, torch.bfloat16, ctx=[200, 300, 90])
    ctx = torch.tensor([200, 300, 90], dtype=torch.int32)
    bt = wl.decode_block_tables.clone()
    bt[1, 3] = wl.num_blocks + 1000
    bt[2, 0] = -7
    q = wl.verify_queries(0, 5)
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    pa.pa_verify_attention(out, q.to(DEV), wl.k_pool.to(DEV), wl.v_pool.to(DEV), bt.to(DEV), ctx.to(DEV),
                           wl.scale, max_context_len=300)
    torch.cuda.synchronize()
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID
    # sequence 0 is untouched by the bad entries
    ref = _ref(wl, q, ctx, seqs=[0])
    assert_close_to_ref(out[:1], ref[:1], wl.dtype, "good row next to bad ones, D 128")
