"""Pins of the INT8 KV-cache oracle against things other than itself.

The quantiser is checked against hand-worked rows of the absmax rule of "LLM
Inference Server", *Required Mathematical Concepts* (s = max|x| / 127,
x_q = round(x / s)), against exact rational arithmetic in pure Python (with
the float32 decision allowed to differ only at exact ties), and against the
rule's invariants (range, the largest element maps to +-127, the
reconstruction error is at most s / 2, power-of-two scaling commutes).  The
INT8 decode is checked against the pinned float oracle on pools whose values
are exactly representable as code x scale, against a pure-Python walk of the
code and scale pools, and against the error bound that V quantisation
implies.  The INT8 verification pass is checked against the decode oracle at
q_len = 1, the pinned float prompt pass on exactly representable pools, a
torch float64 masked softmax over rows walked out of the pools, and the one-key
case of a fresh context.  The INT8 prompt pass is checked against the pinned
float prompt pass on exactly representable pools and against the INT8
verification pass (one sequence's whole prompt as its q_len rows).  The last
group plants plausible mistakes and checks that the pins catch them.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import kv_int8 as q8
from _util import to_np

BS = 16


def _bf16_rows(seed, n, d, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn((n, d), generator=g) * scale).to(torch.bfloat16)
    return to_np(x), x.to(torch.float64).numpy()


def _exact_round_half_even(fr: Fraction) -> int:
    fl = math.floor(fr)
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


# ---------------------------------------------------------------------------
# the quantiser
# ---------------------------------------------------------------------------

def test_hand_worked_rows():
    """Rows whose scale is exact (max|x| = 127 or 254) so every step of the rule
    can be done by hand, ties included (half to even)."""
    x = np.array([[127.0, -63.5, 2.5, 0.5, -0.5, 1.5, 0.0, 126.5],
                  [-254.0, 1.0, 3.0, -1.0, 5.0, -5.0, 0.0, 0.0],
                  [0.0] * 8], dtype=np.float32)
    codes, s = q8.quantize_rows_int8(x)
    assert s.dtype == np.float32 and codes.dtype == np.int8
    assert s.tolist() == [1.0, 2.0, 0.0]
    assert codes[0].tolist() == [127, -64, 2, 0, 0, 2, 0, 126]
    assert codes[1].tolist() == [-127, 0, 2, 0, 2, -2, 0, 0]
    assert codes[2].tolist() == [0] * 8


def test_against_exact_rationals_tiny():
    """Pure Python with Fractions: code = round_half_even(127 x / max|x|).  The
    float32 decision may differ from the exact one only where 127 x / max|x|
    sits within 1e-4 of a half-integer, and then only by one step."""
    bits, vals = _bf16_rows(6, 40, 12)
    codes, s = q8.quantize_rows_int8(bits)
    for r in range(vals.shape[0]):
        amax = max(Fraction(abs(float(v))) for v in vals[r])
        for e in range(vals.shape[1]):
            t = Fraction(float(vals[r, e])) * 127 / amax
            want = _exact_round_half_even(t)
            near_tie = abs(t - math.floor(t) - Fraction(1, 2)) < Fraction(1, 10000)
            got = int(codes[r, e])
            assert got == want or (near_tie and abs(got - want) == 1), (r, e, got, want)


@pytest.mark.parametrize("src", ["bf16", "fp16", "fp32"])
def test_rule_invariants(src):
    g = torch.Generator().manual_seed(7)
    x = torch.randn((500, 128), generator=g) * torch.exp(torch.randn((500, 1), generator=g) * 3)
    x = x.to({"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[src])
    xv = x.to(torch.float64).numpy()
    codes, s = q8.quantize_rows_int8(to_np(x))
    c = codes.astype(np.int64)
    assert c.min() >= -127 and c.max() <= 127
    amax = np.max(np.abs(xv), axis=1)
    # the scale is max|x| / 127 rounded once to float32
    assert np.all(np.abs(s.astype(np.float64) - amax / 127) <= amax / 127 * 2.0 ** -24)
    # the largest element maps to +-127 with its sign
    arg = np.argmax(np.abs(xv), axis=1)
    assert np.all(c[np.arange(500), arg] == 127 * np.sign(xv[np.arange(500), arg]))
    # round to nearest: the reconstruction error is at most half a step
    err = np.abs(xv - s.astype(np.float64)[:, None] * c)
    assert np.all(err <= s.astype(np.float64)[:, None] * (0.5 + 1e-5))
    # codes never have the opposite sign of the value
    assert np.all(c * np.sign(xv) >= 0)


def test_power_of_two_scaling_commutes():
    bits, _ = _bf16_rows(8, 64, 64)
    x = q8._as_f32(bits)
    c0, s0 = q8.quantize_rows_int8(x)
    for k in (-20, -3, 1, 7, 30):
        c1, s1 = q8.quantize_rows_int8((x * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** k)).astype(np.float32))


def test_exact_codes_round_trip():
    """Values that already are code x 2^e with max|code| = 127 come back
    unchanged, and dequantise to themselves exactly."""
    rng = np.random.default_rng(9)
    codes = rng.integers(-127, 128, size=(30, 64)).astype(np.int8)
    codes[np.arange(30), rng.integers(0, 64, 30)] = rng.choice([-127, 127], 30)
    s = (2.0 ** rng.integers(-8, 4, 30)).astype(np.float32)
    x = (s[:, None] * codes.astype(np.float32)).astype(np.float32)
    c1, s1 = q8.quantize_rows_int8(x)
    assert np.array_equal(c1, codes) and np.array_equal(s1, s)
    assert np.array_equal(q8.dequantize_rows_int8(c1, s1), x.astype(np.float64))


def test_zero_row_and_single_nonzero():
    x = np.zeros((2, 16), dtype=np.float32)
    x[1, 5] = -3.0
    c, s = q8.quantize_rows_int8(x)
    assert s[0] == 0 and not c[0].any()
    assert s[1] == np.float32(3.0) / np.float32(127) and c[1, 5] == -127 and np.count_nonzero(c[1]) == 1


def test_tiny_rows_keep_the_full_code_range():
    """No floor on the row maximum: a row whose largest magnitude is far below
    1e-8 still maps it to +-127 (s = max / 127 in float32), and minus half of
    it to -64 (the float32 quotient is -63.5, which rounds to the even -64)."""
    x = np.zeros((1, 8), dtype=np.float32)
    x[0, 0] = np.float32(2.0 ** -40)
    x[0, 3] = np.float32(-(2.0 ** -41))
    c, s = q8.quantize_rows_int8(x)
    assert s[0] == np.float32(2.0 ** -40) / np.float32(127)
    assert c[0, 0] == 127 and c[0, 3] == -64 and np.count_nonzero(c[0]) == 2


# ---------------------------------------------------------------------------
# append: quantise-on-write through the slot mapping
# ---------------------------------------------------------------------------

def test_append_int8_writes_only_its_slots():
    rng = np.random.default_rng(10)
    nb, h, d, T = 7, 3, 32, 20
    kc = np.full((nb, h, BS, d), 77, dtype=np.int8)
    vc = np.full((nb, h, BS, d), -55, dtype=np.int8)
    ks = np.full((nb, h, BS), 123.0, dtype=np.float32)
    vs = np.full((nb, h, BS), 321.0, dtype=np.float32)
    slots = rng.permutation(nb * BS)[:T].astype(np.int64)
    slots[3] = -1
    kn_bits, kn = _bf16_rows(11, T * h, d)
    vn_bits, vn = _bf16_rows(12, T * h, d)
    kn_bits, vn_bits = kn_bits.reshape(T, h, d), vn_bits.reshape(T, h, d)
    kn, vn = kn.reshape(T, h, d), vn.reshape(T, h, d)
    okc, ovc, oks, ovs = oracle.append_int8_ref(kc, vc, ks, vs, slots, kn_bits, vn_bits)
    written = np.zeros((nb, BS), dtype=bool)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = divmod(int(sl), BS)
        written[b, o] = True
        for hh in range(h):
            for new, codes, sc in ((kn, okc, oks), (vn, ovc, ovs)):
                rec = sc[b, hh, o].astype(np.float64) * codes[b, hh, o].astype(np.float64)
                amax = np.max(np.abs(new[t, hh]))
                assert sc[b, hh, o] == np.float32(amax) / np.float32(127)
                assert np.all(np.abs(rec - new[t, hh]) <= sc[b, hh, o] * (0.5 + 1e-5))
    # everything else is untouched, byte for byte
    keep = ~np.broadcast_to(written[:, None, :], (nb, h, BS))
    for before, after in ((kc, okc), (vc, ovc), (ks, oks), (vs, ovs)):
        assert np.array_equal(before[keep], after[keep])
    assert int(written.sum()) == T - 1


# ---------------------------------------------------------------------------
# decode over the dequantised cache
# ---------------------------------------------------------------------------

def _int8_pools(seed, nb, h, d, pow2_scales=False):
    rng = np.random.default_rng(seed)
    kc = rng.integers(-127, 128, size=(nb, h, BS, d)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(nb, h, BS, d)).astype(np.int8)
    if pow2_scales:
        ks = (2.0 ** rng.integers(-9, -4, size=(nb, h, BS))).astype(np.float32)
        vs = (2.0 ** rng.integers(-9, -4, size=(nb, h, BS))).astype(np.float32)
    else:
        ks = rng.uniform(0.005, 0.05, size=(nb, h, BS)).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, size=(nb, h, BS)).astype(np.float32)
    return kc, vc, ks, vs


def _tables(seed, nb, ctx):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(nb)
    mb = max((c + BS - 1) // BS for c in ctx)
    bt = np.zeros((len(ctx), mb), dtype=np.int32)
    pos = 0
    for s, c in enumerate(ctx):
        n = (c + BS - 1) // BS
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    return bt


def test_decode_int8_equals_float_oracle_on_exact_pools():
    """x_hat = s * x_q exactly, so the INT8 decode must equal the pinned float
    decode of the pools that hold x_hat (bit for bit in float64); per-row
    power-of-two scales make any mix-up of the scale indexing visible."""
    nb, h, hq, d = 24, 2, 8, 16
    kc, vc, ks, vs = _int8_pools(20, nb, h, d, pow2_scales=True)
    ctx = [1, 17, 40, 95]
    bt = _tables(21, nb, ctx)
    g = torch.Generator().manual_seed(22)
    q = torch.randn((len(ctx), hq, d), generator=g).numpy()
    kf = ks[..., None].astype(np.float64) * kc.astype(np.float64)
    vf = vs[..., None].astype(np.float64) * vc.astype(np.float64)
    ref = oracle.decode_ref(q, kf, vf, bt, np.array(ctx), 0.25)
    got = oracle.decode_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.25)
    assert np.array_equal(got, ref)


def test_decode_int8_brute_force_from_pools():
    """Pure-Python loops reading codes and scales straight from the pools
    (block table walk, dequantise, softmax), no gather helper."""
    nb, h, hq, d = 10, 2, 4, 6
    kc, vc, ks, vs = _int8_pools(23, nb, h, d)
    ctx = [5, 33]
    bt = _tables(24, nb, ctx)
    g = torch.Generator().manual_seed(25)
    q = torch.randn((2, hq, d), generator=g).numpy()
    got = oracle.decode_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.4)
    G = hq // h
    for s, c in enumerate(ctx):
        for hh in range(hq):
            kv = hh // G
            xs, vrows = [], []
            for p in range(c):
                b, o = int(bt[s][p // BS]), p % BS
                krow = [float(ks[b, kv, o]) * int(kc[b, kv, o, e]) for e in range(d)]
                vrows.append([float(vs[b, kv, o]) * int(vc[b, kv, o, e]) for e in range(d)])
                xs.append(0.4 * sum(float(q[s, hh, e]) * krow[e] for e in range(d)))
            m = max(xs)
            w = [math.exp(x - m) for x in xs]
            z = sum(w)
            for e in range(d):
                want = sum(w[i] * vrows[i][e] for i in range(c)) / z
                assert abs(got[s, hh, e] - want) < 1e-12


def test_v_quantisation_error_is_bounded():
    """With K exact and only V quantised, the output is a convex combination of
    the V rows, so it moves by at most max_i s_v,i / 2 from the float result."""
    nb, h, hq, d = 20, 2, 8, 32
    rng = np.random.default_rng(26)
    kc, _, ks, _ = _int8_pools(27, nb, h, d, pow2_scales=True)
    kf = ks[..., None].astype(np.float64) * kc.astype(np.float64)
    vbits = to_np(torch.randn((nb, h, BS, d), generator=torch.Generator().manual_seed(28)).to(torch.bfloat16))
    vf = oracle.as_f64(vbits)
    vc, vs = q8.quantize_rows_int8(vbits)
    ctx = [16, 50, 120]
    bt = _tables(29, nb, ctx)
    q = rng.standard_normal((3, hq, d))
    ref = oracle.decode_ref(q, kf, vf, bt, np.array(ctx), 0.2)
    got = oracle.decode_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.2)
    bound = float(np.max(vs)) * (0.5 + 1e-5)
    assert np.max(np.abs(got - ref)) <= bound
    assert np.max(np.abs(got - ref)) > 0


# ---------------------------------------------------------------------------
# verification pass (q_len query tokens per sequence, causal)
# ---------------------------------------------------------------------------

def test_verify_int8_with_one_query_is_decode():
    """q_len = 1: the only query sits at position c - 1 and sees the whole
    context, which is the decode oracle's computation."""
    nb, h, hq, d = 16, 2, 8, 16
    kc, vc, ks, vs = _int8_pools(40, nb, h, d)
    ctx = [1, 30, 64, 0]
    bt = _tables(41, nb, ctx)
    q = torch.randn((4, hq, d), generator=torch.Generator().manual_seed(42)).numpy()
    want = oracle.decode_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.3)
    got = oracle.verify_int8_ref(q[:, None], kc, vc, ks, vs, bt, np.array(ctx), 0.3)
    assert np.array_equal(got[:, 0], want)


def test_verify_int8_equals_float_prefill_on_exact_pools():
    """On pools that hold x_hat = s * x_q exactly, the verification pass is the
    pinned float prompt pass over a cached prefix with q_len new rows per
    sequence (bit for bit in float64), including a context shorter than q_len."""
    nb, h, hq, d, ql = 24, 2, 8, 16, 5
    kc, vc, ks, vs = _int8_pools(43, nb, h, d, pow2_scales=True)
    ctx = [5, 17, 3, 90]
    bt = _tables(44, nb, ctx)
    q = torch.randn((len(ctx), ql, hq, d), generator=torch.Generator().manual_seed(45)).numpy()
    kf = ks[..., None].astype(np.float64) * kc.astype(np.float64)
    vf = vs[..., None].astype(np.float64) * vc.astype(np.float64)
    cu = np.arange(len(ctx) + 1, dtype=np.int64) * ql
    want = oracle.prefill_ref(q.reshape(-1, hq, d), kf, vf, bt, cu, np.array(ctx), 0.25)
    got = oracle.verify_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.25)
    assert np.array_equal(got.reshape(-1, hq, d), want)


def test_verify_int8_against_masked_softmax_from_pools():
    """Each sequence's K_hat and V_hat built by walking the block table and the
    code and scale pools in plain Python; all q_len x H_q scores at once in
    torch float64 with a causal mask (query i may see key j iff
    j <= c - q_len + i); fully masked rows are zero."""
    nb, h, hq, d, ql = 12, 2, 4, 8, 4
    kc, vc, ks, vs = _int8_pools(46, nb, h, d)
    ctx = [4, 2, 37, 16]
    bt = _tables(47, nb, ctx)
    q = torch.randn((len(ctx), ql, hq, d), generator=torch.Generator().manual_seed(48), dtype=torch.float64)
    got = oracle.verify_int8_ref(q.numpy(), kc, vc, ks, vs, bt, np.array(ctx), 0.35)
    G = hq // h
    for s, c in enumerate(ctx):
        kh = torch.zeros((c, h, d), dtype=torch.float64)
        vh = torch.zeros((c, h, d), dtype=torch.float64)
        for p in range(c):
            b, o = int(bt[s][p // BS]), p % BS
            for g in range(h):
                for e in range(d):
                    kh[p, g, e] = float(ks[b, g, o]) * int(kc[b, g, o, e])
                    vh[p, g, e] = float(vs[b, g, o]) * int(vc[b, g, o, e])
        allowed = torch.tensor([[j <= c - ql + i for j in range(c)] for i in range(ql)], dtype=torch.bool)
        for hh in range(hq):
            x = 0.35 * q[s, :, hh, :] @ kh[:, hh // G, :].T                 # [q_len][c]
            x = x.masked_fill(~allowed, float("-inf"))
            w = torch.softmax(x, dim=-1).nan_to_num(0.0)                      # all-masked rows -> 0
            want = (w @ vh[:, hh // G, :]).numpy()
            assert np.max(np.abs(got[s, :, hh, :] - want)) < 1e-12


def test_prefill_int8_equals_float_prefill_on_exact_pools():
    """On pools that hold x_hat = s * x_q exactly, the INT8 prompt pass is the
    pinned float prompt pass (bit for bit in float64), with ragged prompts,
    cached prefixes and an empty prompt."""
    nb, h, hq, d = 40, 2, 8, 16
    kc, vc, ks, vs = _int8_pools(60, nb, h, d, pow2_scales=True)
    qlens = [5, 0, 33, 17]
    ctx = [5, 9, 70, 40]
    bt = _tables(61, nb, ctx)
    cu = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int64)
    q = torch.randn((int(cu[-1]), hq, d), generator=torch.Generator().manual_seed(62)).numpy()
    kf = ks[..., None].astype(np.float64) * kc.astype(np.float64)
    vf = vs[..., None].astype(np.float64) * vc.astype(np.float64)
    want = oracle.prefill_ref(q, kf, vf, bt, cu, np.array(ctx), 0.3)
    got = oracle.prefill_int8_ref(q, kc, vc, ks, vs, bt, cu, np.array(ctx), 0.3)
    assert np.array_equal(got, want)
    # a subset of rows leaves the others zero and computes the same values
    sub = oracle.prefill_int8_ref(q, kc, vc, ks, vs, bt, cu, np.array(ctx), 0.3, rows=[0, 40])
    assert np.array_equal(sub[[0, 40]], want[[0, 40]]) and not sub[1:40].any()


def test_prefill_int8_is_the_verification_of_the_whole_prompt():
    """A sequence whose q_len rows are its last q_len positions: the prompt pass
    over those rows is the INT8 verification pass with that q_len (float64,
    to rounding order), on arbitrary codes and scales."""
    nb, h, hq, d = 20, 2, 4, 8
    kc, vc, ks, vs = _int8_pools(63, nb, h, d)
    ctx, ql = [37, 12], 12
    bt = _tables(64, nb, ctx)
    q = torch.randn((len(ctx), ql, hq, d), generator=torch.Generator().manual_seed(65)).numpy()
    want = oracle.verify_int8_ref(q, kc, vc, ks, vs, bt, np.array(ctx), 0.4)
    cu = np.arange(len(ctx) + 1, dtype=np.int64) * ql
    got = oracle.prefill_int8_ref(q.reshape(-1, hq, d), kc, vc, ks, vs, bt, cu, np.array(ctx), 0.4)
    assert np.max(np.abs(got.reshape(want.shape) - want)) < 1e-12


def test_verify_int8_first_query_of_a_fresh_context_sees_one_key():
    """c = q_len: query 0 sits at position 0, so its output is V_hat of slot 0
    of the first block, whatever q holds."""
    nb, h, hq, d, ql = 6, 2, 4, 8, 5
    kc, vc, ks, vs = _int8_pools(49, nb, h, d)
    bt = _tables(50, nb, [ql])
    q = torch.randn((1, ql, hq, d), generator=torch.Generator().manual_seed(51)).numpy() * 7.0
    got = oracle.verify_int8_ref(q, kc, vc, ks, vs, bt, np.array([ql]), 1.0)
    b = int(bt[0, 0])
    for hh in range(hq):
        g = hh // (hq // h)
        v0 = float(vs[b, g, 0]) * vc[b, g, 0].astype(np.float64)
        assert np.allclose(got[0, 0, hh], v0, rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

def _mutant_quantizer(kind):
    def quantize(x):
        x32 = q8._as_f32(x)
        if kind == "per_tensor":
            amax = np.full(x32.shape[:-1], np.max(np.abs(x32)), dtype=np.float32)
        else:
            amax = np.max(np.abs(x32), axis=-1)
        div = np.float32(128 if kind == "div128" else 127)
        s = (amax / div).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1))
        r = x32 / safe[..., None]
        if kind == "floor":
            c = np.floor(r)
        elif kind == "half_away":
            c = np.sign(r) * np.floor(np.abs(r) + 0.5)
        else:
            c = np.rint(r)
        c = np.where(s[..., None] > 0, c, 0)
        return np.clip(c, -127, 127).astype(np.int8), s
    return quantize


@pytest.mark.parametrize("kind", ["div128", "floor", "half_away", "per_tensor"])
def test_planted_quantiser_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(q8, "quantize_rows_int8", _mutant_quantizer(kind))
    failed = 0
    for pin in (test_hand_worked_rows, test_against_exact_rationals_tiny,
                lambda: test_rule_invariants("bf16")):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0


def test_planted_scale_transpose_is_caught(monkeypatch):
    """Reading the scale pool as [block][16][H_kv] instead of [block][H_kv][16]."""
    def gather(codes, scales, block_table, context_len):
        c = oracle.gather_contiguous(codes, block_table, context_len)
        nb, h, bs = scales.shape
        wrong = scales.reshape(nb, bs, h).transpose(0, 2, 1)
        s = oracle.gather_contiguous(np.ascontiguousarray(wrong)[..., None], block_table, context_len)
        return s * c
    monkeypatch.setattr(q8, "gather_dequantized", gather)
    with pytest.raises(AssertionError):
        test_decode_int8_equals_float_oracle_on_exact_pools()


@pytest.mark.parametrize("shift", [-1, 1])
def test_planted_causal_offset_is_caught(shift, monkeypatch):
    """A query that sees one key too few or one too many."""
    real = q8.attend

    def attend(q_row, k, v, scale, n_keys, return_lse=False):
        n = min(max(n_keys + shift, 0), k.shape[0])
        return real(q_row, k, v, scale, n, return_lse)
    monkeypatch.setattr(q8, "attend", attend)
    with pytest.raises(AssertionError):
        test_verify_int8_against_masked_softmax_from_pools()
