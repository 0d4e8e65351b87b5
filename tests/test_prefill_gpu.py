"""pa_prefill_attention (causal prompt pass over the pool) against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, fill_unused_with_nan, oracle_append, run_append, run_decode
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu


def _run_prefill(wl, q, cu, ctx, kp, vp, bt):
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    qlens = (cu[1:] - cu[:-1])
    pa.pa_prefill_attention(out, q.to(DEV), kp, vp, bt.contiguous().to(DEV), cu.to(DEV), ctx.to(DEV), wl.scale,
                            max_q_len=int(qlens.max()), max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    return out


def _case(seed, qlens, prior, hq=32, hkv=8, d=128, dtype=torch.bfloat16):
    ctx = [a + b for a, b in zip(qlens, prior)]
    wl = W.small_random(seed, len(ctx), 0, hq, hkv, d, dtype, ctx=ctx)
    g = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((sum(qlens), hq, d), generator=g).to(dtype)
    cu = torch.tensor([0] + list(np.cumsum(qlens)), dtype=torch.int32)
    return wl, q, cu, torch.tensor(ctx, dtype=torch.int32)


@pytest.mark.parametrize("qlens,prior", [
    ([1, 15, 16, 17, 63, 64, 65, 130], [0] * 8),
    ([5, 64, 100], [40, 3, 200]),          # cached prefix before the prompt
    ([257], [0]),
])
@pytest.mark.parametrize("hq,hkv,d,dtype", [(32, 8, 128, torch.bfloat16), (8, 8, 64, torch.bfloat16),
                                            (16, 2, 64, torch.float16),
                                            (12, 4, 128, torch.float16)])   # odd group: one tile per item
def test_prefill_small(qlens, prior, hq, hkv, d, dtype):
    wl, q, cu, ctx = _case(50 + sum(qlens) + d, qlens, prior, hq, hkv, d, dtype)
    fill_unused_with_nan(wl, ctx)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    out = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
    ref = oracle.prefill_ref(to_np(q), to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy(), cu.numpy(),
                             ctx.numpy(), wl.scale)
    assert_close_to_ref(out, ref, dtype, "prefill")
    assert pa.pa_device_status() == 0


def test_prefill_rows_match_gpu_decode():
    """Consistency check, not parity evidence (both sides are GPU paths): row i
    of the prompt pass and a decode of the same query at context position+1
    agree within the bf16 bar of each other.  Parity of each path against the
    oracle is tested separately."""
    wl, q, cu, ctx = _case(60, [200], [0])
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    out = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
    for i in (0, 15, 16, 63, 64, 199):
        st = W.StepInputs(slot_mapping=torch.full((1,), -1, dtype=torch.int64),
                          k_new=torch.empty((1, 8, 128), dtype=torch.bfloat16),
                          v_new=torch.empty((1, 8, 128), dtype=torch.bfloat16),
                          q=q[i:i + 1].clone(), context_lens=torch.tensor([i + 1], dtype=torch.int32))
        dec = run_decode(wl, st, kp, vp)
        assert torch.max(torch.abs(dec[0].float() - out[i].float())).item() < 2e-2


def test_mixed_mistral7b_prefill_every_row():
    """The four prompts (512..2048) of the mixed continuous-batching step in the
    benchmark's launch configuration: every one of the 5120 query rows (so
    every 128-row tile, both tiles of every tile pair, every causal tail)
    against the oracle."""
    wl = W.mixed_mistral7b()
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    k_np, v_np = oracle_append(wl, st)
    out = _run_prefill(wl, st.q_prefill, st.cu_q_lens, st.prefill_context_lens, kp, vp, wl.prefill_block_tables)
    ref = oracle.prefill_ref(to_np(st.q_prefill), k_np, v_np, wl.prefill_block_tables.numpy(),
                             st.cu_q_lens.numpy(), st.prefill_context_lens.numpy(), wl.scale)
    assert_close_to_ref(out, ref, wl.dtype, "mixed prefill")
    assert pa.pa_device_status() == 0


def test_prefill_schedule_counters_wrap():
    """Items are handed out at run time from one of 1024 per-launch counter
    pairs, each set back to zero by its launch's last CTA.  1100 launches
    wrap every pair at least once; the last output equals the first bit for
    bit (an item's arithmetic does not depend on the CTA that runs it), and
    the first matches the oracle."""
    wl, q, cu, ctx = _case(71, [130, 257, 40], [0, 16, 300])
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    first = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
    ref = oracle.prefill_ref(to_np(q), to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy(), cu.numpy(),
                             ctx.numpy(), wl.scale)
    assert_close_to_ref(first, ref, wl.dtype, "prefill, first launch")
    out = torch.empty_like(first)
    qd, btd, cud, ctxd = q.to(DEV), wl.block_tables.contiguous().to(DEV), cu.to(DEV), ctx.to(DEV)
    for _ in range(1100):
        pa.pa_prefill_attention(out, qd, kp, vp, btd, cud, ctxd, wl.scale, max_q_len=257,
                                max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    assert pa.pa_device_status() == 0


def test_prefill_concurrent_launches_on_two_streams():
    """Two prompt passes in flight at once on two streams draw different
    counter pairs: each stays equal to its own single-stream result."""
    cases = [_case(72, [300, 17], [0, 64]), _case(73, [129, 200, 64], [5, 0, 128], hq=16, hkv=2, d=64,
                                                                           dtype=torch.float16)]
    runs = []
    for wl, q, cu, ctx in cases:
        kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
        ref = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
        runs.append((wl, q.to(DEV), cu.to(DEV), ctx.to(DEV), kp, vp, wl.block_tables.contiguous().to(DEV), ref,
                     int((cu[1:] - cu[:-1]).max()), int(ctx.max())))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(r[7]) for r in runs]
    for _ in range(50):
        for (wl, q, cu, ctx, kp, vp, bt, _ref, mq, mc), st, o in zip(runs, streams, outs):
            with torch.cuda.stream(st):
                pa.pa_prefill_attention(o, q, kp, vp, bt, cu, ctx, wl.scale, max_q_len=mq, max_context_len=mc,
                                        stream=st)
    torch.cuda.synchronize()
    for r, o in zip(runs, outs):
        assert torch.equal(o, r[7])
    assert pa.pa_device_status() == 0


def test_prefill_many_sequences_unsorted_order():
    """More (sequence, query tile) pairs than the sorted work list holds (384):
    the items run in the fallback order over (tile, sequence, head group),
    and the run-time schedule skips the items past each prompt.  400 short
    prompts with cached prefixes, every row against the oracle."""
    g = torch.Generator().manual_seed(74)
    qlens = torch.randint(1, 150, (400,), generator=g).tolist()
    prior = torch.randint(0, 40, (400,), generator=g).tolist()
    wl, q, cu, ctx = _case(74, qlens, prior, hq=8, hkv=2, d=64, dtype=torch.bfloat16)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    out = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
    ref = oracle.prefill_ref(to_np(q), to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy(), cu.numpy(),
                             ctx.numpy(), wl.scale)
    assert_close_to_ref(out, ref, wl.dtype, "prefill, 400 sequences")
    assert pa.pa_device_status() == 0


def test_prefill_output_only_16_byte_aligned():
    """The epilogue stores whole 32-byte sectors when the output is 32-byte
    aligned and 16-byte vectors otherwise: an output view 16 bytes past an
    aligned base takes the second path and equals the first bit for bit."""
    wl, q, cu, ctx = _case(75, [200, 64, 1], [0, 30, 7])
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    aligned = _run_prefill(wl, q, cu, ctx, kp, vp, wl.block_tables)
    assert aligned.data_ptr() % 32 == 0
    base = torch.empty(aligned.numel() + 8, dtype=aligned.dtype, device=DEV)
    shifted = base[8:].view(aligned.shape)
    assert shifted.data_ptr() % 32 == 16
    pa.pa_prefill_attention(shifted, q.to(DEV), kp, vp, wl.block_tables.contiguous().to(DEV), cu.to(DEV),
                            ctx.to(DEV), wl.scale, max_q_len=200, max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    assert torch.equal(shifted, aligned)
    assert pa.pa_device_status() == 0
