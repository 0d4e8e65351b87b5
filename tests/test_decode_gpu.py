"""pa_decode_attention on the GPU against the float64 oracle.

Bar: fp32 inputs max-abs 1e-5; bf16/fp16 inputs |gpu - ref| <= 2e-2 + 1e-2 |ref|
(fp32 accumulation inside, one rounding of the output)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, fill_unused_with_nan, oracle_append, oracle_decode, run_append, run_decode
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu


def _step_and_check(wl, t=0, partitions=(0,), seqs=None, k_np=None, v_np=None, kp=None, vp=None):
    st = wl.step(t)
    if kp is None:
        kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    k_np, v_np = oracle_append(wl, st, k_np, v_np)
    ref = oracle_decode(wl, st, k_np, v_np, seqs=seqs)
    for part in partitions:
        out = run_decode(wl, st, kp, vp, partition_size=part)
        if seqs is None:
            assert_close_to_ref(out, ref, wl.dtype, f"{wl.name} t={t} partition={part}")
        else:
            idx = list(seqs)
            assert_close_to_ref(out[idx], ref[idx], wl.dtype, f"{wl.name} t={t} partition={part}")
    assert pa.pa_device_status() == 0
    return kp, vp, k_np, v_np


def test_tiny_fp32_all_partitions():
    _step_and_check(W.tiny_fp32(), partitions=(0, 16, 32, 48, 2048))


def test_llama32_1b_steps():
    wl = W.llama32_1b_decode(steps=4)
    kp = vp = k_np = v_np = None
    for t in range(4):
        kp, vp, k_np, v_np = _step_and_check(wl, t, (0, 256), kp=kp, vp=vp, k_np=k_np, v_np=v_np)


def test_llama3_8b_full_size():
    """The batch-64, D=128 workload in the launch configuration the benchmark
    times (automatic partition): every output row of two consecutive steps
    against the oracle."""
    wl = W.llama3_8b_decode(steps=2)
    kp = vp = k_np = v_np = None
    for t in range(2):
        kp, vp, k_np, v_np = _step_and_check(wl, t, (0,), kp=kp, vp=vp, k_np=k_np, v_np=v_np)


def test_prefix_shared_8k_split_k():
    """All 8 sequences of 8192 tokens (13 shared blocks), automatic, 2048- and
    64-token partitions (4 and 128 partials merged per row)."""
    wl = W.prefix_shared_8k()
    _step_and_check(wl, 0, (0, 2048, 64))


@pytest.mark.parametrize("batch", [1, 4])
def test_llama3_8b_long_context_small_batch(batch):
    """Batch 1 and batch 4 at contexts near 8192 (the small-batch end of the
    decode range, where split-K carries all the parallelism): every row, two
    steps, the automatic partition and two forced ones."""
    wl = W.llama3_8b_long(batch, steps=2)
    kp = vp = k_np = v_np = None
    for t in range(2):
        kp, vp, k_np, v_np = _step_and_check(wl, t, (0, 128, 2048), kp=kp, vp=vp, k_np=k_np, v_np=v_np)


def test_prefix_shared_identical_tails_give_identical_outputs():
    """Sequences whose private blocks hold the same data and whose queries are
    equal must produce bit-identical rows (the shared prefix is read through
    every table)."""
    wl = W.prefix_shared_8k()
    bt = wl.block_tables
    for s in range(1, 8):
        wl.k_pool[bt[s, 13:]] = wl.k_pool[bt[0, 13:]]
        wl.v_pool[bt[s, 13:]] = wl.v_pool[bt[0, 13:]]
    st = wl.step(0)
    st.q[:] = st.q[0]
    st.k_new[:] = st.k_new[0]
    st.v_new[:] = st.v_new[0]
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    out = run_decode(wl, st, kp, vp)
    for s in range(1, 8):
        assert torch.equal(out[s], out[0])


def test_mixed_step_decode_part():
    """The 60 decode sequences of the mixed continuous-batching step, every row."""
    wl = W.mixed_mistral7b()
    _step_and_check(wl, 0, (0,))


@pytest.mark.parametrize("ctx", [[1, 15, 16, 17, 31, 32, 33], [63, 64, 65, 127, 128, 129, 255, 256, 257]])
@pytest.mark.parametrize("part", [0, 16, 64, 128])
def test_ragged_block_and_partition_boundaries(ctx, part):
    wl = W.small_random(21, len(ctx), 0, 32, 8, 128, torch.bfloat16, ctx=ctx)
    _step_and_check(wl, 0, (part,))


@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (8, 8, 128, torch.bfloat16), (4, 2, 64, torch.bfloat16), (16, 2, 128, torch.bfloat16),
    (12, 4, 64, torch.float16), (32, 8, 128, torch.float16), (8, 1, 64, torch.float32),
    (6, 2, 128, torch.float32), (16, 2, 64, torch.float32)])
def test_group_sizes_dims_dtypes(hq, hkv, d, dtype):
    wl = W.small_random(30 + hq + d, 5, 700, hq, hkv, d, dtype)
    _step_and_check(wl, 0, (0, 64, 512))


def test_zero_context_rows_are_zero():
    wl = W.small_random(40, 4, 0, 8, 2, 128, torch.bfloat16, ctx=[50, 0, 300, 0])
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    for part in (0, 16):
        out = run_decode(wl, st, kp, vp, partition_size=part)
        assert int(out[1].count_nonzero()) == 0 and int(out[3].count_nonzero()) == 0
        k_np, v_np = oracle_append(wl, st)
        assert_close_to_ref(out, oracle_decode(wl, st, k_np, v_np), wl.dtype, "zero ctx")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_stale_nan_slots_never_leak(dtype):
    """Every slot outside the contexts holds NaN (partial last blocks included)."""
    wl = W.small_random(41, 6, 200, 16, 4, 128 if dtype != torch.float32 else 64, dtype)
    st = wl.step(0)
    fill_unused_with_nan(wl, st.context_lens)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    k_np, v_np = oracle_append(wl, st)
    ref = oracle_decode(wl, st, k_np, v_np)
    assert np.isfinite(ref).all()
    for part in (0, 16, 48):
        out = run_decode(wl, st, kp, vp, partition_size=part)
        assert torch.isfinite(out.float()).all()
        assert_close_to_ref(out, ref, dtype, f"nan canary part={part}")


def test_long_context_16k_boundaries():
    ctx = [16383, 16384, 16385, 1]
    wl = W.small_random(42, 4, 0, 32, 8, 128, torch.bfloat16, ctx=ctx)
    _step_and_check(wl, 0, (0, 2048), seqs=[0, 1, 2, 3])


def test_partition_choice_does_not_change_results_beyond_rounding():
    wl = W.small_random(43, 8, 3000, 32, 8, 128, torch.bfloat16)
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    outs = [run_decode(wl, st, kp, vp, partition_size=p).float() for p in (16, 128, 512, 2048)]
    for o in outs[1:]:
        assert torch.max(torch.abs(o - outs[0])).item() < 2e-2


def test_bad_block_id_is_reported_not_dereferenced():
    wl = W.small_random(44, 3, 100, 8, 2, 128, torch.bfloat16, ctx=[40, 90, 17])
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    bt = wl.decode_block_tables.clone()
    bt[1, 2] = wl.num_blocks + 1000
    bt[2, 0] = -7
    out = torch.empty(st.q.shape, dtype=st.q.dtype, device=DEV)
    pa.pa_decode_attention(out, st.q.to(DEV), kp, vp, bt.to(DEV), st.context_lens.to(DEV), wl.scale,
                           max_context_len=90)
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID
    # sequence 0 is untouched by the bad entries
    k_np, v_np = to_np(wl.k_pool), to_np(wl.v_pool)
    ref = oracle_decode(wl, st, k_np, v_np, seqs=[0])
    assert_close_to_ref(out[:1], ref[:1], wl.dtype, "good row next to bad ones")


def test_context_above_host_bound_is_clamped_and_reported():
    wl = W.small_random(45, 2, 100, 8, 2, 64, torch.bfloat16, ctx=[40, 90])
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    out = torch.empty(st.q.shape, dtype=st.q.dtype, device=DEV)
    # host says 64 but sequence 1 has 90: the kernels clamp to 64 and flag it
    pa.pa_decode_attention(out, st.q.to(DEV), kp, vp, wl.decode_block_tables.contiguous().to(DEV),
                           st.context_lens.to(DEV), wl.scale, max_context_len=64, partition_size=16)
    assert pa.pa_device_status() & pa.PA_DEV_BAD_CONTEXT
    assert torch.isfinite(out.float()).all()
