"""pa_decode_step: the append fused into the decode launch.

After the call the pools must equal the oracle's append of every sequence's
new token at position context - 1, byte for byte, and the output must equal
pa_append_kv followed by pa_decode_attention bit for bit (same arithmetic),
hence the oracle within the decode bar."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, oracle_append, oracle_decode, run_append, run_decode
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu


def _step(wl, st, kp, vp, part=0):
    out = torch.empty(st.q.shape, dtype=st.q.dtype, device=DEV)
    pa.pa_decode_step(out, st.q.to(DEV), kp, vp, st.k_new.to(DEV), st.v_new.to(DEV),
                      wl.decode_block_tables.contiguous().to(DEV), st.context_lens.to(DEV), wl.scale,
                      max_context_len=int(st.context_lens.max()), partition_size=part)
    torch.cuda.synchronize()
    return out


def _same_bytes(gpu, ref):
    return np.array_equal(to_np(gpu).view(np.uint8), ref.view(np.uint8))


@pytest.mark.parametrize("factory,parts", [(W.tiny_fp32, (0, 16)),
                                           (lambda: W.small_random(150, 6, 900, 32, 8, 128, torch.bfloat16),
                                            (0, 16, 64)),
                                           (lambda: W.small_random(151, 5, 400, 16, 4, 64, torch.float16), (0, 32))])
def test_fused_step_equals_append_then_decode(factory, parts):
    wl = factory()
    st = wl.step(0)
    k_ref, v_ref = oracle_append(wl, st)
    ref = oracle_decode(wl, st, k_ref, v_ref)
    for part in parts:
        kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
        out = _step(wl, st, kp, vp, part)
        assert _same_bytes(kp, k_ref) and _same_bytes(vp, v_ref)
        kp2, vp2 = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
        run_append(wl, st, kp2, vp2)
        sep = run_decode(wl, st, kp2, vp2, partition_size=part)
        assert torch.equal(out, sep)
        assert_close_to_ref(out, ref, wl.dtype, f"decode step part={part}")
    assert pa.pa_device_status() == 0


def test_empty_contexts_append_nothing():
    wl = W.small_random(152, 4, 0, 8, 2, 128, torch.bfloat16, ctx=[50, 0, 300, 0])
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    out = _step(wl, st, kp, vp)
    k_ref, v_ref = oracle_append(wl, st)          # slots -1 for the empty contexts
    assert _same_bytes(kp, k_ref) and _same_bytes(vp, v_ref)
    assert int(out[1].count_nonzero()) == 0 and int(out[3].count_nonzero()) == 0


def test_llama3_8b_steps_keep_the_pool_and_match_the_oracle():
    """Three consecutive batch-64 steps through the fused call (automatic
    partition, as the benchmark runs it); pools bit-exact after each step,
    every output row against the oracle."""
    wl = W.llama3_8b_decode(steps=3)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    k_np, v_np = to_np(wl.k_pool), to_np(wl.v_pool)
    for t in range(3):
        st = wl.step(t)
        out = _step(wl, st, kp, vp)
        k_np, v_np = oracle_append(wl, st, k_np, v_np)
        assert _same_bytes(kp, k_np) and _same_bytes(vp, v_np)
        ref = oracle_decode(wl, st, k_np, v_np)
        assert_close_to_ref(out, ref, wl.dtype, f"llama3 step {t}")
    assert pa.pa_device_status() == 0


@pytest.mark.parametrize("batch", [1, 4])
def test_long_context_small_batch_steps(batch):
    """The fused step at batch 1 and 4 with contexts near 8192: pools bit-exact,
    every row within the bar, two steps."""
    wl = W.llama3_8b_long(batch, steps=2)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    k_np, v_np = to_np(wl.k_pool), to_np(wl.v_pool)
    for t in range(2):
        st = wl.step(t)
        out = _step(wl, st, kp, vp)
        k_np, v_np = oracle_append(wl, st, k_np, v_np)
        assert _same_bytes(kp, k_np) and _same_bytes(vp, v_np)
        assert_close_to_ref(out, oracle_decode(wl, st, k_np, v_np), wl.dtype, f"batch {batch} step {t}")
    assert pa.pa_device_status() == 0
