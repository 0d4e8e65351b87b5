"""RoPE fused into the append, on the GPU, against the float64 oracle.

Every expected value here is computed from oracle inputs alone: the oracle
builds its own (cos, sin) table (``oracle.rope_cache_ref``) and never sees the
table the GPU built.

Bars, from the arithmetic:
  * table: float64 angle and trigonometry on both sides, rounded once to
    float32: |gpu - ref| <= 1 ulp of float32 at |ref| plus the float64 error of
    the angle itself (pow is within 2 ulp on either side, so the angle p * f
    may differ by 4 * 2^-52 * p * f, which moves cos / sin by as much in
    absolute terms -- visible only next to their zeros);
  * rotation: the GPU computes fp32 a*c - b*s (one fused multiply-add) on ITS
    table, then rounds once to the element type; the oracle rotates exactly
    in float64 on the oracle's table.  The two tables differ by at most the
    table bar above, |dc|, |ds| <= 2^-23 + 4 * 2^-52 * p * f (cos and sin lie
    in [-1, 1], where a float32 ulp is at most 2^-23), which moves the exact
    rotation by at most that much times (|a| + |b|).  So
    |gpu - ref| <= e + half an ulp of the element type at |ref| + e, with
    e = (2^-22 + 2^-23 + 4 * 2^-52 * p * f_max) (|a| + |b|), the first term
    being the fp32 arithmetic;
  * V rows: bit-exact copies, untouched slots untouched.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import DEV, run_decode
from _util import assert_close_to_ref, to_f64, to_np

pytestmark = pytest.mark.gpu


def gpu_cache(max_pos, d, theta):
    cs = torch.empty((max_pos, d // 2, 2), dtype=torch.float32, device=DEV)
    pa.pa_rope_cache(cs, theta)
    torch.cuda.synchronize()
    return cs


def rotation_bound(x: torch.Tensor, ref: np.ndarray, max_angle: float) -> np.ndarray:
    """e + half an ulp of the element type at |ref| + e, with
    e = (2^-22 + 2^-23 + 4 * 2^-52 * max_angle) (|a| + |b|) per pair: the fp32
    arithmetic plus the largest difference between the GPU's table and the
    oracle's (max_angle bounds p * f over the rows checked)."""
    a = np.abs(to_f64(x))
    h = a.shape[-1] // 2
    pair = np.concatenate([a[..., :h] + a[..., h:]] * 2, axis=-1)
    e = (2.0 ** -22 + 2.0 ** -23 + 4 * 2.0 ** -52 * max_angle) * pair
    mant = {torch.float32: 23, torch.bfloat16: 7, torch.float16: 10}[x.dtype]
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref) + e, 1e-30))) - mant)
    return e + 0.5 * ulp + 1e-30


@pytest.mark.parametrize("d,theta", [(128, 10000.0), (128, 500000.0), (64, 10000.0)])
def test_cache_matches_oracle(d, theta):
    cs = gpu_cache(9000, d, theta).cpu().numpy()
    ref = oracle.rope_cache_ref(9000, d, theta)
    diff = np.abs(cs.astype(np.float64) - ref.astype(np.float64))
    angle = np.arange(9000, dtype=np.float64)[:, None] * oracle.rope_inv_freq(d, theta)[None, :]
    bound = np.spacing(np.abs(ref)).astype(np.float64) + 4 * 2.0 ** -52 * angle[..., None]
    assert np.all(diff <= bound)
    assert np.mean(cs == ref) > 0.999


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 128),
                                     (torch.bfloat16, 64)])
def test_append_rope_rotates_k_and_copies_v(dtype, d):
    g = torch.Generator().manual_seed(120 + d)
    nb, hkv, T = 12, 4, 40
    kp = torch.empty((nb, hkv, 16, d), dtype=dtype)
    kp.view(torch.uint8).fill_(0x5A)
    vp = kp.clone()
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[7] = -1
    pos = torch.randint(0, 8192, (T,), generator=g, dtype=torch.int32)
    pos[0] = 0
    k_new = (torch.randn((T, hkv, d), generator=g) * 3).to(dtype)
    v_new = torch.randn((T, hkv, d), generator=g).to(dtype)
    cs = gpu_cache(8192, d, 10000.0)
    kd, vd = kp.to(DEV), vp.to(DEV)
    pa.pa_append_kv_rope(kd, vd, slots.to(DEV), pos.to(DEV), k_new.to(DEV), v_new.to(DEV), cs)
    torch.cuda.synchronize()
    assert pa.pa_device_status() == 0
    k_rot, v_ref = oracle.append_rope_ref(to_np(vp), slots.numpy(), pos.numpy(), to_np(k_new), to_np(v_new),
                                          oracle.rope_cache_ref(8192, d, 10000.0))
    assert np.array_equal(to_np(vd).view(np.uint8), v_ref.view(np.uint8))
    kg = kd.cpu()
    written = torch.zeros((nb, 16), dtype=torch.bool)
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        b, o = divmod(s, 16)
        written[b, o] = True
        got = to_f64(kg[b, :, o])
        err = np.abs(got - k_rot[t])
        assert np.all(err <= rotation_bound(k_new[t], k_rot[t], float(pos[t]))), (t, float(err.max()))
    # position 0 is the identity: that row is copied exactly
    b0, o0 = divmod(int(slots[0]), 16)
    assert torch.equal(kg[b0, :, o0], k_new[0])
    keep = ~written
    assert torch.equal(kg.permute(0, 2, 1, 3)[keep].view(torch.uint8), kp.permute(0, 2, 1, 3)[keep].view(torch.uint8))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_apply_rope_in_place(dtype):
    g = torch.Generator().manual_seed(130)
    T, H, d = 33, 32, 128
    x = (torch.randn((T, H, d), generator=g) * 2).to(dtype)
    pos = torch.randint(0, 4096, (T,), generator=g, dtype=torch.int32)
    cs = gpu_cache(4096, d, 500000.0)
    xd = x.to(DEV)
    pa.pa_apply_rope(xd, pos.to(DEV), cs)
    torch.cuda.synchronize()
    ref = oracle.rope_rotate_ref(to_np(x), pos.numpy(), oracle.rope_cache_ref(4096, d, 500000.0))
    assert np.all(np.abs(to_f64(xd) - ref) <= rotation_bound(x, ref, 4095.0))


def test_bad_position_is_skipped_and_reported():
    kd = torch.zeros((4, 2, 16, 64), dtype=torch.bfloat16, device=DEV)
    vd = torch.zeros_like(kd)
    kn = torch.ones((2, 2, 64), dtype=torch.bfloat16, device=DEV)
    cs = gpu_cache(100, 64, 10000.0)
    slots = torch.tensor([3, 9], dtype=torch.int64, device=DEV)
    pos = torch.tensor([5, 100], dtype=torch.int32, device=DEV)
    pa.pa_append_kv_rope(kd, vd, slots, pos, kn, kn, cs)
    assert pa.pa_device_status() & pa.PA_DEV_BAD_POSITION
    assert int(kd[0, :, 9].count_nonzero()) == 0 and int(kd[0, :, 3].count_nonzero()) > 0
    assert int(vd[0, :, 9].count_nonzero()) == 2 * 64     # V is still written


def _rope_decode(wl, shift, cs):
    """Fill every context position of every sequence through the RoPE append,
    rotate the decode queries at position ctx - 1 (+ shift), decode."""
    g = torch.Generator().manual_seed(140)
    bt = wl.decode_block_tables
    ctx = wl.ctx0
    slots = torch.cat([bt[s, torch.arange(int(c)) // 16].to(torch.int64) * 16 + torch.arange(int(c)) % 16
                       for s, c in enumerate(ctx)])
    pos = torch.cat([torch.arange(int(c), dtype=torch.int32) for c in ctx]) + shift
    kn = torch.randn((slots.numel(), wl.num_kv_heads, wl.head_dim), generator=g).to(wl.dtype)
    vn = torch.randn((slots.numel(), wl.num_kv_heads, wl.head_dim), generator=g).to(wl.dtype)
    q = torch.randn((len(ctx), wl.num_q_heads, wl.head_dim), generator=g).to(wl.dtype)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    pa.pa_append_kv_rope(kp, vp, slots.to(DEV), pos.to(DEV), kn.to(DEV), vn.to(DEV), cs)
    qd = q.to(DEV)
    pa.pa_apply_rope(qd, (ctx - 1 + shift).to(torch.int32).to(DEV), cs)
    st = W.StepInputs(slot_mapping=torch.full((len(ctx),), -1, dtype=torch.int64), k_new=kn[:1], v_new=vn[:1],
                      q=qd.cpu(), context_lens=ctx)
    out = run_decode(wl, st, kp, vp)
    return out, (slots, pos, kn, vn, q, kp, vp)


def test_decode_over_rotated_cache_matches_oracle_and_depends_on_relative_positions():
    wl = W.small_random(141, 4, 0, 16, 4, 128, torch.bfloat16, ctx=[17, 100, 333, 64])
    cs = gpu_cache(8192, 128, 10000.0)
    out0, (slots, pos, kn, vn, q, kp, vp) = _rope_decode(wl, 0, cs)
    # oracle: its own table, rotation in float64, decode over the rotated cache
    csn = oracle.rope_cache_ref(8192, 128, 10000.0)
    k_rot = oracle.rope_rotate_ref(to_np(kn), pos.numpy(), csn)
    q_rot = oracle.rope_rotate_ref(to_np(q), (wl.ctx0 - 1).numpy(), csn)
    k_pool = oracle.as_f64(to_np(wl.k_pool)).copy()
    v_pool = oracle.as_f64(to_np(wl.v_pool)).copy()
    for t, s in enumerate(slots.tolist()):
        k_pool[s // 16, :, s % 16] = k_rot[t]
        v_pool[s // 16, :, s % 16] = to_f64(vn[t])
    ref = oracle.decode_ref(q_rot, k_pool, v_pool, wl.decode_block_tables.numpy(), wl.ctx0.numpy(), wl.scale)
    assert_close_to_ref(out0, ref, wl.dtype, "decode over RoPE cache")
    # every position shifted by the same amount: scores depend on differences only
    wl2 = W.small_random(141, 4, 0, 16, 4, 128, torch.bfloat16, ctx=[17, 100, 333, 64])
    out1, _ = _rope_decode(wl2, 1234, cs)
    assert torch.max(torch.abs(out1.float() - out0.float())).item() < 2e-2
