"""The rounding test of the INT8 append, replayed in float32 on the host.

The append ("LLM Inference Server", Optional Bonus Extensions: INT8
KV-Cache Quantization; Required Mathematical Concepts: s = max|x| / 127,
x_q = round(x / s)) decides each code without a division: t = x * (1/s)
with the correctly rounded reciprocal, t + 1.5 * 2^23 holds the nearest
integer n of t in its low bits, e = t - n is the rounding error, and the
row falls back to the IEEE division when !(|e| < 1/2 - 2^-12) (Ziv's
strategy: t is within 2^-16 of x / s, so away from a tie both round alike).

These tests replay exactly those float32 steps with NumPy (every operation
rounds to nearest even, as the kernel's explicit-rounding intrinsics do) on
rows built to hit the edges: ties, scales down to the subnormal range,
infinities and NaNs.  They pin the argument, not the kernel: wherever the
one-comparison test passes, the low byte of the sum is the code of
round-to-nearest-even(fl(x / s)); and it flags exactly the elements that the
earlier two-comparison form (t finite and below 256, |e| more than 2^-12
from 1/2) flagged.  The GPU tests compare the kernel's codes with the
oracle's bit for bit.
"""
import numpy as np

F = np.float32
MAGIC = F(12582912.0)   # 1.5 * 2^23


def _replay(x: np.ndarray):
    with np.errstate(all="ignore"):
        amax = np.max(np.abs(np.where(np.isnan(x), F(0), x)), axis=1)   # fmaxf ignores NaN
        s = (amax / F(127)).astype(F)
        r = np.where(s > 0, (F(1) / s).astype(F), F(0)).astype(F)
        t = (x * r[:, None]).astype(F)
        m = (t + MAGIC).astype(F)
        e = (t - (m - MAGIC)).astype(F)
        near_one = ~(np.abs(e) < F(0.5) - F(2.0 ** -12))
        near_two = ~(np.abs(t) < F(256)) | ~(np.abs(np.abs(e) - F(0.5)) > F(2.0 ** -12))
        low = (m.view(np.int32) & 0xFF).astype(np.int64)
        fast = np.where(low > 127, low - 256, low)
        q = (x / np.where(s > 0, s, F(1))[:, None]).astype(F)
        exact = np.clip(np.rint(q), -127, 127)
    return s, near_one, near_two, fast, exact


def _rows(rng) -> list:
    out = []
    for scale in (1e-3, 1.0, 3e4, 1e30, 1e-36, 1e-38, 1e-40, 1e-43):
        out.append((rng.standard_normal((1500, 128)) * scale).astype(F))
    sp = rng.standard_normal((700, 128)).astype(F)
    sp[::7, 3] = np.inf
    sp[1::7, 5] = -np.inf
    sp[2::7, 9] = np.nan
    sp[3::7] = 0
    sp[4::7, :] = F(1e-45)
    out.append(sp)
    for s0 in (F(0.37), F(1e-39), F(3.0e30)):
        ties = ((rng.integers(-127, 127, (700, 128)) + F(0.5)) * s0).astype(F)
        ties[:, 0] = F(127) * s0   # the row's maximum fixes s = s0 (up to rounding)
        out.append(ties)
    return out


def test_fast_code_equals_the_rounded_quotient_where_the_test_passes():
    rng = np.random.default_rng(11)
    checked = 0
    for x in _rows(rng):
        s, near, _, fast, exact = _replay(x)
        ok = near | (s[:, None] == 0) | (fast == exact)
        assert bool(ok.all())
        checked += int((~near & (s[:, None] > 0)).sum())
    assert checked > 1_000_000


def test_one_comparison_flags_what_the_two_comparison_form_flags():
    rng = np.random.default_rng(12)
    for x in _rows(rng):
        _, near_one, near_two, _, _ = _replay(x)
        assert np.array_equal(near_one, near_two)


def test_rows_of_ties_are_flagged_and_specials_fall_back():
    rng = np.random.default_rng(13)
    s0 = F(0.37)
    ties = ((rng.integers(-120, 120, (64, 128)) + F(0.5)) * s0).astype(F)
    ties[:, 0] = F(127) * s0
    _, near, _, _, _ = _replay(ties)
    assert near.any(axis=1).all()   # every row holds quotients at (or next to) a half-integer
    x = np.zeros((3, 128), F)
    x[0, 1] = np.nan
    x[1, 2] = np.inf
    x[2, 3] = F(1e-45)   # the scale underflows to zero: every code is 0
    s, near, _, fast, _ = _replay(x)
    assert near[0, 1] and near[1, 2]
    assert s[2] == 0 and not near[2].any() and (fast[2] == 0).all()
