"""INT8 KV cache on the GPU against the float64 oracle.

Append: codes and scales bit-exact (the quantiser's float32 decisions are
single IEEE operations on both sides).  Decode: the output against the oracle's
attention over the dequantised cache, |gpu - ref| <= 2e-2 + 1e-2 |ref| (fp32
accumulation inside, one rounding of the bf16/fp16 output)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _gpu import oracle_append
from _util import assert_close_to_ref, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


class Cache:
    """Device copy of a workload's INT8 cache plus the oracle's host state."""

    def __init__(self, wl: W.Workload):
        self.kc, self.vc = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
        self.ks, self.vs = wl.k_scales.to(DEV), wl.v_scales.to(DEV)
        self.host = [to_np(wl.k_pool), to_np(wl.v_pool), wl.k_scales.numpy().copy(), wl.v_scales.numpy().copy()]

    def append(self, st: W.StepInputs):
        pa.pa_append_kv_int8(self.kc, self.vc, self.ks, self.vs, st.slot_mapping.to(DEV), st.k_new.to(DEV),
                             st.v_new.to(DEV))
        self.host = list(oracle.append_int8_ref(*self.host, st.slot_mapping.numpy(), to_np(st.k_new),
                                                to_np(st.v_new)))

    def decode(self, wl, st, part=0, max_ctx=None):
        out = torch.empty(st.q.shape, dtype=st.q.dtype, device=DEV)
        mc = int(st.context_lens.max()) if max_ctx is None else max_ctx
        pa.pa_decode_attention_int8(out, st.q.to(DEV), self.kc, self.vc, self.ks, self.vs,
                                    wl.decode_block_tables.contiguous().to(DEV), st.context_lens.to(DEV), wl.scale,
                                    max_context_len=mc, partition_size=part)
        torch.cuda.synchronize()
        return out

    def ref(self, wl, st, seqs=None):
        return oracle.decode_int8_ref(to_np(st.q), *self.host, wl.decode_block_tables.contiguous().numpy(),
                                      st.context_lens.numpy(), wl.scale, seqs=seqs)

    def same_as_oracle(self):
        torch.cuda.synchronize()
        got = [to_np(self.kc), to_np(self.vc), self.ks.cpu().numpy(), self.vs.cpu().numpy()]
        return all(np.array_equal(g.view(np.uint8), h.view(np.uint8)) for g, h in zip(got, self.host))


def _check(wl, st, cache, parts=(0,), seqs=None):
    ref = cache.ref(wl, st, seqs=seqs)
    for part in parts:
        out = cache.decode(wl, st, part)
        idx = list(range(out.shape[0])) if seqs is None else list(seqs)
        assert_close_to_ref(out[idx], ref[idx], wl.dtype, f"{wl.name} int8 partition={part}")
    assert pa.pa_device_status() == 0


# ---------------------------------------------------------------------------
# append: quantise on write
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.bfloat16), (128, torch.float16),
                                     (64, torch.float16)])
def test_append_int8_bit_exact(d, dtype):
    wl = W.small_random(60 + d, 6, 300, 16, 4, d, dtype, kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    assert cache.same_as_oracle()
    assert pa.pa_device_status() == 0


def test_append_int8_special_rows():
    """Zero rows, exact ties (x / s = k + 1/2 with s exact), a single nonzero,
    tiny (subnormal scale) and huge magnitudes, padding and out-of-range slots."""
    hkv, d, T = 2, 128, 8
    g = torch.Generator().manual_seed(61)
    nb = 4
    kc = torch.randint(-127, 128, (nb, hkv, 16, d), generator=g, dtype=torch.int16).to(torch.int8)
    vc = kc.clone()
    ks = torch.full((nb, hkv, 16), 7.0)
    vs = ks.clone()
    x = torch.randn((T, hkv, d), generator=g)
    x[0] = 0.0
    x[1, 0] = 127.0
    x[1, 0, 1:] = torch.arange(1, d, dtype=torch.float32) * 0.5 - 32.0    # many .5 ties with s = 1
    x[2] = 0.0
    x[2, 1, 5] = -3.0
    x[3] *= 1e-38                                                     # scale underflows to a subnormal
    x[4] *= 3e4
    xk = x.to(torch.bfloat16)
    xv = (x * 0.5).to(torch.bfloat16)
    slots = torch.tensor([0, 17, 33, 50, 63, -1, 5, 40], dtype=torch.int64)
    wl = W.Workload(name="special", config_id=0, dtype=torch.bfloat16, num_q_heads=2, num_kv_heads=hkv,
                    head_dim=d, scale=0.1, steps=1, k_pool=kc, v_pool=vc,
                    block_tables=torch.zeros((1, 1), dtype=torch.int32), ctx0=torch.zeros(1, dtype=torch.int32),
                    decode_rows=slice(0, 1), k_scales=ks, v_scales=vs)
    cache = Cache(wl)
    st = W.StepInputs(slot_mapping=slots, k_new=xk, v_new=xv, q=torch.zeros((1, 2, d), dtype=torch.bfloat16),
                      context_lens=torch.zeros(1, dtype=torch.int32))
    cache.append(st)
    assert cache.same_as_oracle()
    assert pa.pa_device_status() == 0
    # a slot past the pool is skipped and reported
    bad = slots.clone()
    bad[2] = nb * 16 + 1
    pa.pa_append_kv_int8(cache.kc, cache.vc, cache.ks, cache.vs, bad.to(DEV), xk.to(DEV), xv.to(DEV))
    assert pa.pa_device_status() & pa.PA_DEV_BAD_SLOT


def _near_tie_rows(dtype, amaxes, d):
    """One row per amax A: A itself and the d - 1 values of `dtype` in
    [-A, A] whose quotient by s = float32(A / 127) lies closest to a
    half-integer (where the rounding of x / s decides the code), so that the
    quantiser's rounding test meets values on both sides of its margin."""
    if dtype == torch.float16:
        every = torch.arange(0, 0x7c00, dtype=torch.int32).to(torch.int16).view(torch.float16)
    else:
        every = torch.arange(0, 0x7f80, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    vals = every.double().numpy()
    rows = []
    for a in amaxes:
        a = float(torch.tensor(a, dtype=dtype).double())
        sc = np.float64(np.float32(np.float32(a) / np.float32(127)))
        cand = np.concatenate([vals[vals <= a], -vals[(vals > 0) & (vals <= a)]])
        q = cand / sc
        dist = np.abs(q - np.floor(q) - 0.5)
        pick = cand[np.argsort(dist, kind="stable")[:d - 1]]
        rows.append(np.concatenate([[a], pick]))
    return torch.tensor(np.array(rows)).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_append_int8_near_ties(dtype):
    """Codes of values whose x / s sits within a few ulps of k + 1/2 for
    inexact scales: bit-exact against the oracle's float32 division."""
    hkv, d = 2, 128
    amaxes = [100.0, 77.3, 1.7, 0.013, 3.1e-4, 6.0e-5, 5.5e4]
    rows = _near_tie_rows(dtype, amaxes, d)               # [len(amaxes)][d]
    T = len(amaxes)
    xk = torch.zeros((T, hkv, d), dtype=dtype)
    xk[:, 0] = rows
    xk[:, 1] = rows.flip(1)
    xv = torch.roll(xk, 1, dims=0)
    nb = 2
    kc = torch.zeros((nb, hkv, 16, d), dtype=torch.int8)
    ks = torch.zeros((nb, hkv, 16))
    wl = W.Workload(name="near_ties", config_id=0, dtype=dtype, num_q_heads=2, num_kv_heads=hkv,
                    head_dim=d, scale=0.1, steps=1, k_pool=kc, v_pool=kc.clone(),
                    block_tables=torch.zeros((1, 1), dtype=torch.int32), ctx0=torch.zeros(1, dtype=torch.int32),
                    decode_rows=slice(0, 1), k_scales=ks, v_scales=ks.clone())
    cache = Cache(wl)
    st = W.StepInputs(slot_mapping=torch.arange(T, dtype=torch.int64) * 3, k_new=xk, v_new=xv,
                      q=torch.zeros((1, 2, d), dtype=dtype), context_lens=torch.zeros(1, dtype=torch.int32))
    cache.append(st)
    assert cache.same_as_oracle()
    assert pa.pa_device_status() == 0


def test_append_int8_llama3_8b_steps():
    wl = W.llama3_8b_decode(steps=3, kv="int8")
    cache = Cache(wl)
    for t in range(3):
        cache.append(wl.step(t))
    assert cache.same_as_oracle()


# ---------------------------------------------------------------------------
# decode over the dequantised cache
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv,d,dtype", [
    (32, 8, 128, torch.bfloat16), (8, 8, 128, torch.bfloat16), (16, 2, 128, torch.float16),
    (32, 8, 64, torch.bfloat16), (12, 4, 64, torch.float16), (8, 1, 64, torch.bfloat16)])
def test_decode_int8_group_sizes_dims_dtypes(hq, hkv, d, dtype):
    wl = W.small_random(70 + hq + d, 5, 700, hq, hkv, d, dtype, kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    _check(wl, st, cache, parts=(0, 16, 64, 512))


@pytest.mark.parametrize("ctx", [[1, 15, 16, 17, 31, 32, 33], [63, 64, 65, 127, 128, 129, 255, 256, 257]])
@pytest.mark.parametrize("part", [0, 16, 128])
def test_decode_int8_ragged_boundaries(ctx, part):
    wl = W.small_random(81, len(ctx), 0, 32, 8, 128, torch.bfloat16, ctx=ctx, kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    _check(wl, st, cache, parts=(part,))


def test_decode_int8_stale_slots_never_leak():
    """Scales of every slot outside the contexts are NaN and their codes are
    +-127: none of it may reach the output."""
    wl = W.small_random(82, 6, 200, 16, 4, 128, torch.bfloat16, kv="int8")
    st = wl.step(0)
    used = set()
    bt = wl.block_tables
    for s in range(bt.shape[0]):
        for p in range(int(st.context_lens[s])):
            used.add(int(bt[s, p // 16]) * 16 + p % 16)
    for slot in range(wl.num_blocks * 16):
        if slot not in used:
            b, o = divmod(slot, 16)
            wl.k_scales[b, :, o] = float("nan")
            wl.v_scales[b, :, o] = float("nan")
            wl.k_pool[b, :, o] = 127
            wl.v_pool[b, :, o] = -127
    cache = Cache(wl)
    cache.append(st)
    ref = cache.ref(wl, st)
    assert np.isfinite(ref).all()
    for part in (0, 16, 48):
        out = cache.decode(wl, st, part)
        assert torch.isfinite(out.float()).all()
        assert_close_to_ref(out, ref, wl.dtype, f"int8 stale slots part={part}")


def test_decode_int8_zero_context_rows_are_zero():
    wl = W.small_random(83, 4, 0, 8, 2, 128, torch.bfloat16, ctx=[50, 0, 300, 0], kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    for part in (0, 16):
        out = cache.decode(wl, st, part)
        assert int(out[1].count_nonzero()) == 0 and int(out[3].count_nonzero()) == 0
    _check(wl, st, cache, parts=(0, 16))


@pytest.mark.parametrize("kscale,vscale,qscale", [(1e-6, 1e-6, 1.0), (300.0, 1e4, 1.0), (0.02, 0.02, 1e3),
                                                  (0.02, 0.02, 1e-3)])
def test_decode_int8_value_ranges(kscale, vscale, qscale):
    """Scales and query magnitudes far from 1: the fp16 operands inside must
    neither overflow nor lose the small rows."""
    wl = W.small_random(84, 4, 600, 16, 4, 128, torch.bfloat16, kv="int8")
    wl.k_scales.mul_(kscale * 127 / 3)
    wl.v_scales.mul_(vscale * 127 / 3)
    st = wl.step(0)
    st.q = (st.q.float() * qscale).to(torch.bfloat16)
    st.slot_mapping[:] = -1          # keep the drawn cache as it is
    cache = Cache(wl)
    ref = cache.ref(wl, st)
    for part in (0, 64):
        out = cache.decode(wl, st, part)
        # the bar is relative to the output's own magnitude
        mag = max(float(np.max(np.abs(ref))), 1e-30)
        err = float(torch.max(torch.abs(out.double().cpu() - torch.from_numpy(ref))))
        assert err <= 1e-2 * mag + 2e-2 * min(mag, 1.0), (err, mag)


def test_decode_int8_llama3_8b_full_size():
    """The batch-64, D=128 workload over an INT8 cache in the launch
    configuration the benchmark times (automatic partition), two steps with
    the quantising append before each, every row against the oracle."""
    wl = W.llama3_8b_decode(steps=2, kv="int8")
    cache = Cache(wl)
    for t in range(2):
        st = wl.step(t)
        cache.append(st)
        _check(wl, st, cache, parts=(0,))


def test_decode_int8_llama32_1b():
    wl = W.llama32_1b_decode(steps=2, kv="int8")
    cache = Cache(wl)
    for t in range(2):
        st = wl.step(t)
        cache.append(st)
        _check(wl, st, cache, parts=(0, 256))


def test_int8_cache_tracks_the_float_cache():
    """End to end: the same bf16 rows appended into a float cache and into an
    INT8 cache give decode outputs within the quantisation error of each
    other (|dv| <= s_v / 2 per element moves the output by at most that)."""
    wl = W.small_random(85, 4, 0, 16, 4, 128, torch.bfloat16, ctx=[40, 100, 250, 16])
    wq = W.small_random(85, 4, 0, 16, 4, 128, torch.bfloat16, ctx=[40, 100, 250, 16], kv="int8")
    # write every context position of both caches from the same bf16 rows
    g = torch.Generator().manual_seed(86)
    bt = wl.decode_block_tables
    slots = torch.cat([bt[s, torch.arange(c) // 16].to(torch.int64) * 16 + torch.arange(c) % 16
                       for s, c in enumerate([40, 100, 250, 16])])
    kn = (torch.randn((slots.numel(), 4, 128), generator=g) * 0.1).to(torch.bfloat16)
    vn = torch.randn((slots.numel(), 4, 128), generator=g).to(torch.bfloat16)
    kp, vp = wl.k_pool.to(DEV), wl.v_pool.to(DEV)
    pa.pa_append_kv(kp, vp, slots.to(DEV), kn.to(DEV), vn.to(DEV))
    cache = Cache(wq)
    st = W.StepInputs(slot_mapping=slots, k_new=kn, v_new=vn, q=wl.step(0).q,
                      context_lens=torch.tensor([40, 100, 250, 16], dtype=torch.int32))
    cache.append(st)
    out_f = torch.empty(st.q.shape, dtype=torch.bfloat16, device=DEV)
    pa.pa_decode_attention(out_f, st.q.to(DEV), kp, vp, bt.contiguous().to(DEV), st.context_lens.to(DEV), wl.scale,
                           max_context_len=250)
    out_q = cache.decode(wq, st)
    smax = float(cache.vs.max())
    assert float(torch.max(torch.abs(out_f.float() - out_q.float()))) <= smax + 0.05


# ---------------------------------------------------------------------------
# verification pass (q_len query tokens per sequence, causal) over the cache
# ---------------------------------------------------------------------------

def _verify8(wl, cache, q, ctx, part=0, max_ctx=None):
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    mc = int(ctx.max()) if max_ctx is None else max_ctx
    pa.pa_verify_attention_int8(out, q.to(DEV), cache.kc, cache.vc, cache.ks, cache.vs,
                                wl.decode_block_tables.contiguous().to(DEV), ctx.to(DEV), wl.scale,
                                max_context_len=mc, partition_size=part)
    torch.cuda.synchronize()
    return out


def _verify8_ref(wl, cache, q, ctx, seqs=None):
    return oracle.verify_int8_ref(to_np(q), *cache.host, wl.decode_block_tables.contiguous().numpy(),
                                  ctx.numpy(), wl.scale, seqs=seqs)


@pytest.mark.parametrize("hq,hkv,q_len,d,dtype", [
    (32, 8, 5, 128, torch.bfloat16),    # G 4 x 5: 20 columns, three 8-column tiles
    (32, 4, 4, 128, torch.bfloat16),    # G 8 x 4: 32 columns, four tiles
    (8, 8, 5, 128, torch.float16),      # G 1 x 5: one tile, masked
    (16, 8, 4, 128, torch.bfloat16),    # G 2 x 4: exactly one tile
    (32, 8, 3, 128, torch.float16),     # G 4 x 3: two tiles, a ragged second one
    (16, 8, 5, 64, torch.bfloat16),     # G 2 x 5: two tiles, D 64
    (12, 4, 8, 64, torch.float16),      # G 3 x 8: three tiles, D 64
    (32, 8, 8, 64, torch.bfloat16),     # G 4 x 8: four tiles, D 64
])
def test_verify_int8_shapes(hq, hkv, q_len, d, dtype):
    wl = W.small_random(120 + hq + q_len + d, 5, 600, hq, hkv, d, dtype, kv="int8")
    cache = Cache(wl)
    ctx = wl.ctx0.clamp(min=q_len)
    q = wl.verify_queries(0, q_len)
    ref = _verify8_ref(wl, cache, q, ctx)
    for part in (0, 16, 64, 512):
        out = _verify8(wl, cache, q, ctx, part)
        assert_close_to_ref(out, ref, dtype, f"int8 verify G={hq // hkv} q_len={q_len} part={part}")
    assert pa.pa_device_status() == 0


@pytest.mark.parametrize("ctx", [[1, 2, 4, 5, 6, 15, 16, 17, 20, 21], [31, 32, 33, 64, 65, 255, 256, 257]])
def test_verify_int8_ragged_contexts(ctx):
    """The causal edge at every offset of a 16-token block and at partition
    boundaries; contexts shorter than q_len give zero rows for the queries
    before position 0."""
    wl = W.small_random(131, len(ctx), 0, 32, 8, 128, torch.bfloat16, ctx=ctx, kv="int8")
    cache = Cache(wl)
    ctx_t = torch.tensor(ctx, dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    ref = _verify8_ref(wl, cache, q, ctx_t)
    for part in (0, 16, 32):
        out = _verify8(wl, cache, q, ctx_t, part)
        assert_close_to_ref(out, ref, wl.dtype, f"int8 verify ragged part={part}")
        for s, c in enumerate(ctx):
            if c < 5:   # queries 0 .. 4 - c sit before position 0
                assert int(out[s, :5 - c].count_nonzero()) == 0
    assert pa.pa_device_status() == 0


def test_verify_int8_q_len_1_is_decode_bit_for_bit():
    wl = W.small_random(132, 6, 900, 32, 8, 128, torch.bfloat16, kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    for part in (0, 64):
        dec = cache.decode(wl, st, part)
        ver = _verify8(wl, cache, st.q[:, None], st.context_lens, part)
        assert torch.equal(ver[:, 0], dec)


def test_verify_int8_last_query_is_the_decode_of_the_whole_context():
    """Query q_len - 1 sits at position c - 1 and sees the whole context, as
    the decode query does: with the same q row both agree within the bar."""
    wl = W.small_random(133, 6, 900, 32, 8, 128, torch.bfloat16, kv="int8")
    cache = Cache(wl)
    ctx = wl.ctx0.clamp(min=5)
    q = wl.verify_queries(0, 5)
    ver = _verify8(wl, cache, q, ctx)
    st = W.StepInputs(slot_mapping=torch.full((6,), -1, dtype=torch.int64), k_new=None, v_new=None,
                      q=q[:, 4].contiguous(), context_lens=ctx)
    dec = cache.decode(wl, st)
    assert_close_to_ref(ver[:, 4], dec.double().cpu().numpy(), wl.dtype, "last verify query vs decode")


def test_verify_int8_zero_contexts_and_bad_block_id():
    wl = W.small_random(134, 4, 0, 32, 8, 128, torch.bfloat16, ctx=[40, 0, 100, 0], kv="int8")
    cache = Cache(wl)
    ctx = torch.tensor([40, 0, 100, 0], dtype=torch.int32)
    q = wl.verify_queries(0, 5)
    out = _verify8(wl, cache, q, ctx, 16)
    assert int(out[1].count_nonzero()) == 0 and int(out[3].count_nonzero()) == 0
    assert_close_to_ref(out, _verify8_ref(wl, cache, q, ctx), wl.dtype, "int8 verify zero contexts")
    assert pa.pa_device_status() == 0
    # a block id past the pool is skipped (its keys weigh nothing) and reported
    bt = wl.decode_block_tables.contiguous().clone()
    bt[2, 1] = wl.k_pool.shape[0] + 7
    out2 = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    pa.pa_verify_attention_int8(out2, q.to(DEV), cache.kc, cache.vc, cache.ks, cache.vs, bt.to(DEV), ctx.to(DEV),
                                wl.scale, max_context_len=100, partition_size=16)
    torch.cuda.synchronize()
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID
    assert torch.equal(out2[0], out[0])       # other sequences unaffected


def test_verify_int8_llama3_8b_full_size():
    """The batch-64, D=128 verification of 4 drafts (q_len 5) over an INT8
    cache in the launch configuration the benchmark times (automatic
    partition), after the quantising append, every row against the oracle."""
    wl = W.llama3_8b_verify(steps=1, kv="int8")
    st = wl.step(0)
    cache = Cache(wl)
    cache.append(st)
    q = wl.verify_queries(0, 5)
    out = _verify8(wl, cache, q, st.context_lens, max_ctx=wl.max_context_len(0))
    ref = _verify8_ref(wl, cache, q, st.context_lens)
    assert_close_to_ref(out, ref, wl.dtype, "int8 verify llama3-8b")
    assert pa.pa_device_status() == 0


# ---------------------------------------------------------------------------
# prompt pass (causal over each prompt and its cached prefix) over the cache
# ---------------------------------------------------------------------------

def _nan_unused_scales(wl, ctx):
    """Every scale slot that no sequence's context covers becomes NaN, so a
    read past a context (or of a block outside it) shows up in the output."""
    used = set()
    for s in range(wl.block_tables.shape[0]):
        for p in range(int(ctx[s])):
            used.add((int(wl.block_tables[s, p // 16]), p % 16))
    for sc in (wl.k_scales, wl.v_scales):
        for b in range(sc.shape[0]):
            for o in range(16):
                if (b, o) not in used:
                    sc[b, :, o] = float("nan")


def _prefill8(wl, cache, q, cu, ctx, bt=None):
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    qlens = cu[1:] - cu[:-1]
    bt = wl.block_tables if bt is None else bt
    pa.pa_prefill_attention_int8(out, q.to(DEV), cache.kc, cache.vc, cache.ks, cache.vs, bt.contiguous().to(DEV),
                                 cu.to(DEV), ctx.to(DEV), wl.scale, max_q_len=int(qlens.max()),
                                 max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    return out


def _prefill8_case(seed, qlens, prior, hq, hkv, d, dtype):
    ctx = [a + b for a, b in zip(qlens, prior)]
    wl = W.small_random(seed, len(ctx), 0, hq, hkv, d, dtype, ctx=ctx, kv="int8")
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
                                            (16, 2, 64, torch.float16), (12, 4, 128, torch.float16)])
def test_prefill_int8_small(qlens, prior, hq, hkv, d, dtype):
    """Ragged prompts, cached prefixes, every 16-token block edge; the scales
    of every slot outside the contexts are NaN."""
    wl, q, cu, ctx = _prefill8_case(140 + sum(qlens) + d + hq, qlens, prior, hq, hkv, d, dtype)
    _nan_unused_scales(wl, ctx)
    cache = Cache(wl)
    out = _prefill8(wl, cache, q, cu, ctx)
    ref = oracle.prefill_int8_ref(to_np(q), *cache.host, wl.block_tables.numpy(), cu.numpy(), ctx.numpy(),
                                  wl.scale)
    assert_close_to_ref(out, ref, dtype, f"int8 prefill G={hq // hkv} d={d}")
    assert pa.pa_device_status() == 0


def test_prefill_int8_bad_block_id_is_reported():
    wl, q, cu, ctx = _prefill8_case(150, [40, 70, 33], [0, 30, 0], 32, 8, 128, torch.bfloat16)
    cache = Cache(wl)
    out = _prefill8(wl, cache, q, cu, ctx)
    assert pa.pa_device_status() == 0
    bt = wl.block_tables.clone()
    bt[1, 2] = wl.k_pool.shape[0] + 5
    out2 = _prefill8(wl, cache, q, cu, ctx, bt)
    assert pa.pa_device_status() & pa.PA_DEV_BAD_BLOCK_ID
    assert torch.equal(out2[:40], out[:40]) and torch.equal(out2[110:], out[110:])   # sequences 0 and 2


def test_prefill_int8_workspace_only_16_byte_aligned():
    """The dequantisation stores whole 32-byte sectors when the workspace is
    32-byte aligned and 16-byte vectors otherwise: a workspace view 16 bytes
    past an aligned base gives the same output bit for bit."""
    wl, q, cu, ctx = _prefill8_case(154, [70, 130], [20, 0], 32, 8, 128, torch.bfloat16)
    cache = Cache(wl)
    ref = _prefill8(wl, cache, q, cu, ctx)
    need = pa.pa_prefill_int8_workspace_size(len(ctx), int(ctx.max()), cache.kc)
    base = torch.empty(need + 32, dtype=torch.uint8, device=DEV)
    ws = base[16:16 + need]
    assert ws.data_ptr() % 32 == 16
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    qlens = cu[1:] - cu[:-1]
    pa.pa_prefill_attention_int8(out, q.to(DEV), cache.kc, cache.vc, cache.ks, cache.vs,
                                 wl.block_tables.contiguous().to(DEV), cu.to(DEV), ctx.to(DEV), wl.scale,
                                 max_q_len=int(qlens.max()), max_context_len=int(ctx.max()), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert pa.pa_device_status() == 0


def test_prefill_int8_bf16_query_past_fp16_range_is_reported():
    """The pass runs in fp16, so a bf16 query element of magnitude 2^16 or more
    cannot be held: it is clamped to 65504 and PA_DEV_RANGE is set; every
    other (row, head) output is what it was."""
    wl, q, cu, ctx = _prefill8_case(153, [40, 70], [0, 30], 32, 8, 128, torch.bfloat16)
    cache = Cache(wl)
    out = _prefill8(wl, cache, q, cu, ctx)
    assert pa.pa_device_status() == 0
    q2 = q.clone()
    q2[45, 3, 7] = 1.0e5                                  # sequence 1, its row 5, head 3
    out2 = _prefill8(wl, cache, q2, cu, ctx)
    assert pa.pa_device_status() & pa.PA_DEV_RANGE
    assert torch.isfinite(out2.float()).all()
    same = torch.ones(out.shape[:2], dtype=torch.bool)
    same[45, 3] = False
    assert torch.equal(out2[same.to(DEV)], out[same.to(DEV)])


def test_prefill_int8_matches_the_float_pass_on_its_dequantised_pools():
    """Consistency check, not parity evidence: on a cache whose x_hat is exactly
    representable in fp16 (power-of-two scales, 8-bit codes), the INT8 prompt
    pass with fp16 activations and the fp16 prompt pass over the same values
    agree bit for bit."""
    wl, q, cu, ctx = _prefill8_case(151, [100, 37], [20, 60], 32, 8, 128, torch.float16)
    g = torch.Generator().manual_seed(152)
    e = torch.randint(-8, -2, wl.k_scales.shape, generator=g).to(torch.float32)
    wl.k_scales.copy_(torch.exp2(e))
    wl.v_scales.copy_(torch.exp2(e.flip(0)))
    cache = Cache(wl)
    out8 = _prefill8(wl, cache, q, cu, ctx)
    kf = (wl.k_scales[..., None].double() * wl.k_pool.double()).to(torch.float16).to(DEV)
    vf = (wl.v_scales[..., None].double() * wl.v_pool.double()).to(torch.float16).to(DEV)
    outf = torch.empty_like(out8)
    pa.pa_prefill_attention(outf, q.to(DEV), kf, vf, wl.block_tables.contiguous().to(DEV), cu.to(DEV),
                            ctx.to(DEV), wl.scale, max_q_len=100, max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    assert torch.equal(out8, outf)


def test_prefill_int8_mixed_mistral7b_prompts():
    """The four prompts (512..2048 tokens) of the mixed Mistral-7B-shaped step
    over an INT8 cache (the prompts' K and V quantised by the oracle's rule),
    every query row against the oracle."""
    wl = W.mixed_mistral7b()
    st = wl.step(0)
    k_np, v_np = oracle_append(wl, st)
    ctx = st.prefill_context_lens
    bt = wl.prefill_block_tables
    kc = np.zeros(k_np.shape, dtype=np.int8)
    vc = np.zeros(v_np.shape, dtype=np.int8)
    ks = np.zeros(k_np.shape[:3], dtype=np.float32)
    vs = np.zeros(v_np.shape[:3], dtype=np.float32)
    for s in range(len(ctx)):
        for b in range((int(ctx[s]) + 15) // 16):
            blk = int(bt[s, b])
            kc[blk], ks[blk] = oracle.quantize_rows_int8(k_np[blk])
            vc[blk], vs[blk] = oracle.quantize_rows_int8(v_np[blk])
    cache = type("C", (), {})()
    cache.kc, cache.vc = torch.from_numpy(kc).to(DEV), torch.from_numpy(vc).to(DEV)
    cache.ks, cache.vs = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    q = st.q_prefill
    out = torch.empty(q.shape, dtype=q.dtype, device=DEV)
    pa.pa_prefill_attention_int8(out, q.to(DEV), cache.kc, cache.vc, cache.ks, cache.vs, bt.contiguous().to(DEV),
                                 st.cu_q_lens.to(DEV), ctx.to(DEV), wl.scale,
                                 max_q_len=int((st.cu_q_lens[1:] - st.cu_q_lens[:-1]).max()),
                                 max_context_len=int(ctx.max()))
    torch.cuda.synchronize()
    ref = oracle.prefill_int8_ref(to_np(q), kc, vc, ks, vs, bt.numpy(), st.cu_q_lens.numpy(), ctx.numpy(), wl.scale)
    assert_close_to_ref(out, ref, wl.dtype, "int8 mixed prefill")
    assert pa.pa_device_status() == 0
