"""pa_append_kv on the GPU: bit-exact against the oracle's indexed copy."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, oracle_append, run_append
from _util import to_np

pytestmark = pytest.mark.gpu


def _same_bytes(gpu: torch.Tensor, ref: np.ndarray) -> bool:
    return np.array_equal(to_np(gpu).view(np.uint8), ref.view(np.uint8))


@pytest.mark.parametrize("factory", [W.tiny_fp32, W.llama32_1b_decode, W.prefix_shared_8k, W.mixed_mistral7b])
def test_append_bit_exact(factory):
    wl = factory()
    st = wl.step(0)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    run_append(wl, st, kp, vp)
    k_ref, v_ref = oracle_append(wl, st)
    torch.cuda.synchronize()
    assert _same_bytes(kp, k_ref) and _same_bytes(vp, v_ref)
    assert pa.pa_device_status() == 0


def test_append_bit_exact_llama3_8b_all_steps():
    """Batch 64, D=128: several steps in a row, each compared with the oracle
    applied to the previous oracle state."""
    wl = W.llama3_8b_decode(steps=3)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    k_ref, v_ref = to_np(wl.k_pool), to_np(wl.v_pool)
    for t in range(3):
        st = wl.step(t)
        run_append(wl, st, kp, vp)
        k_ref, v_ref = oracle_append(wl, st, k_ref, v_ref)
    torch.cuda.synchronize()
    assert _same_bytes(kp, k_ref) and _same_bytes(vp, v_ref)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 128)])
def test_append_canary_negative_and_out_of_range_slots(dtype, d):
    g = torch.Generator().manual_seed(11)
    n_blk, hkv, T = 9, 3, 40
    kp = torch.empty((n_blk, hkv, 16, d), dtype=dtype)
    kp.view(torch.uint8).fill_(0xA5)
    vp = kp.clone()
    slots = torch.randperm(n_blk * 16, generator=g)[:T].to(torch.int64)
    slots[5] = -1
    slots[17] = -100
    k_new = torch.randn((T, hkv, d), generator=g).to(dtype)
    v_new = torch.randn((T, hkv, d), generator=g).to(dtype)
    ref_k, ref_v = __import__("oracle").append_ref(to_np(kp), to_np(vp), slots.numpy(), to_np(k_new),
                                                   to_np(v_new))
    kd, vd = kp.to(DEV), vp.to(DEV)
    pa.pa_append_kv(kd, vd, slots.to(DEV), k_new.to(DEV), v_new.to(DEV))
    torch.cuda.synchronize()
    assert _same_bytes(kd, ref_k) and _same_bytes(vd, ref_v)
    assert pa.pa_device_status() == 0
    # a slot past the pool is skipped by the kernel and reported
    bad = slots.clone()
    bad[0] = n_blk * 16 + 3
    kd2, vd2 = kp.to(DEV), vp.to(DEV)
    pa.pa_append_kv(kd2, vd2, bad.to(DEV), k_new.to(DEV), v_new.to(DEV))
    assert pa.pa_device_status() & pa.PA_DEV_BAD_SLOT
    rk, _ = __import__("oracle").append_ref(to_np(kp), to_np(vp), torch.where(bad >= n_blk * 16, -1, bad).numpy(),
                                            to_np(k_new), to_np(v_new))
    assert _same_bytes(kd2, rk)


def test_append_empty_is_a_no_op():
    kp = torch.zeros((2, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device=DEV)
    pa.pa_append_kv(kp, vp, torch.empty((0,), dtype=torch.int64, device=DEV), e, e)
    assert int(kp.count_nonzero()) == 0
