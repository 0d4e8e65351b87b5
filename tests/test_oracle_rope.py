"""Pins of the RoPE oracle against things other than itself.

The rotary embedding (Llama form: entries j and j + D/2 rotated together by
p * theta^(-2j/D)) is checked against library trigonometry at the frequencies
whose values are known in closed form (j = 0 turns one radian per position;
with theta = 10000 and j = D/4 the frequency is 1/100), against the image of a
unit vector (which fixes both the pairing and the sign), and against the
invariants of a rotation: position 0 is the identity, pair norms are kept,
and scores depend on positions only through their difference.  Planted
mistakes (interleaved pairs, the opposite sign, a wrong frequency exponent)
must fail them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import rope as R

D = 128


def test_position_zero_is_the_identity():
    cache = R.rope_cache_ref(4, D, 10000.0)
    assert np.array_equal(cache[0, :, 0], np.ones(D // 2, np.float32))
    assert np.array_equal(cache[0, :, 1], np.zeros(D // 2, np.float32))
    x = np.random.default_rng(1).standard_normal((3, 2, D)).astype(np.float32)
    assert np.array_equal(R.rope_rotate_ref(x, np.zeros(3, np.int64), cache), x.astype(np.float64))


@pytest.mark.parametrize("theta", [10000.0, 500000.0])
def test_first_pair_turns_one_radian_per_position(theta):
    cache = R.rope_cache_ref(9000, D, theta)
    for p in (1, 2, 7, 100, 4095, 8191, 8999):
        assert cache[p, 0, 0] == np.float32(math.cos(p)) and cache[p, 0, 1] == np.float32(math.sin(p))


def test_quarter_frequency_is_one_hundredth_at_theta_1e4():
    cache = R.rope_cache_ref(301, D, 10000.0)
    for p, a in ((100, 1.0), (300, 3.0)):
        assert abs(float(cache[p, D // 4, 0]) - math.cos(a)) < 1e-7
        assert abs(float(cache[p, D // 4, 1]) - math.sin(a)) < 1e-7


def test_unit_vector_rotates_into_the_second_half():
    cache = R.rope_cache_ref(10, D, 10000.0)
    e0 = np.zeros((1, 1, D), np.float32)
    e0[0, 0, 0] = 1.0
    y = R.rope_rotate_ref(e0, np.array([3]), cache)[0, 0]
    assert y[0] == np.float64(np.float32(math.cos(3)))
    assert y[D // 2] == np.float64(np.float32(math.sin(3)))
    assert np.count_nonzero(y) == 2
    # and the second-half unit vector rotates back into the first half with a minus sign
    eh = np.zeros((1, 1, D), np.float32)
    eh[0, 0, D // 2] = 1.0
    z = R.rope_rotate_ref(eh, np.array([3]), cache)[0, 0]
    assert z[0] == -np.float64(np.float32(math.sin(3))) and z[D // 2] == np.float64(np.float32(math.cos(3)))


def test_pair_norms_are_kept():
    cache = R.rope_cache_ref(5000, D, 10000.0)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 4, D)).astype(np.float32)
    pos = rng.integers(0, 5000, 50)
    y = R.rope_rotate_ref(x, pos, cache)
    h = D // 2
    n0 = x[..., :h].astype(np.float64) ** 2 + x[..., h:].astype(np.float64) ** 2
    n1 = y[..., :h] ** 2 + y[..., h:] ** 2
    assert np.max(np.abs(n1 - n0) / np.maximum(n0, 1e-30)) < 1e-6   # cos^2 + sin^2 = 1 to float32 rounding


def test_scores_depend_on_the_position_difference_only():
    cache = R.rope_cache_ref(9000, D, 10000.0)
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    k = rng.standard_normal((1, 1, D)).astype(np.float32)
    def score(m, n):
        return float(np.sum(R.rope_rotate_ref(q, np.array([m]), cache) * R.rope_rotate_ref(k, np.array([n]), cache)))
    base = score(40, 13)
    for shift in (1, 100, 3000, 8000):
        assert abs(score(40 + shift, 13 + shift) - base) < 2e-4 * np.linalg.norm(q) * np.linalg.norm(k)
    assert abs(score(41, 13) - base) > 1e-3   # a different difference does change it


def test_append_rope_copies_v_exactly_and_skips_padding():
    rng = np.random.default_rng(4)
    nb, h, d, T = 5, 2, 16, 6
    v_pool = np.full((nb, h, 16, d), 9.0, np.float32)
    slots = np.array([3, 17, -1, 40, 77, 5], np.int64)
    pos = np.array([0, 5, 6, 7, 100, 2])
    k_new = rng.standard_normal((T, h, d)).astype(np.float32)
    v_new = rng.standard_normal((T, h, d)).astype(np.float32)
    cache = R.rope_cache_ref(128, d, 10000.0)
    k_rot, v_out = R.append_rope_ref(v_pool, slots, pos, k_new, v_new, cache)
    assert np.array_equal(k_rot[0], k_new[0].astype(np.float64))      # position 0
    for t, sl in enumerate(slots):
        if sl >= 0:
            assert np.array_equal(v_out[sl // 16, :, sl % 16], v_new[t])
    assert np.count_nonzero(v_out != 9.0) == 5 * h * d


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

def _mutant_cache(kind):
    def cache(max_positions, head_dim, theta):
        j = np.arange(head_dim // 2, dtype=np.float64)
        expo = -j / head_dim if kind == "exponent" else -2.0 * j / head_dim
        ang = np.arange(max_positions, dtype=np.float64)[:, None] * np.power(theta, expo)[None, :]
        out = np.empty((max_positions, head_dim // 2, 2), np.float32)
        out[..., 0] = np.cos(ang)
        out[..., 1] = -np.sin(ang) if kind == "sign" else np.sin(ang)
        return out
    return cache


def _interleaved_rotate(x, positions, cache):
    x64 = x.astype(np.float64)
    c = cache[positions, :, 0].astype(np.float64)[:, None, :]
    s = cache[positions, :, 1].astype(np.float64)[:, None, :]
    ev, od = x64[..., 0::2], x64[..., 1::2]
    out = np.empty_like(x64)
    out[..., 0::2] = ev * c - od * s
    out[..., 1::2] = od * c + ev * s
    return out


@pytest.mark.parametrize("kind", ["exponent", "sign"])
def test_planted_cache_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(R, "rope_cache_ref", _mutant_cache(kind))
    caught = 0
    for pin in (test_quarter_frequency_is_one_hundredth_at_theta_1e4, test_unit_vector_rotates_into_the_second_half):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught > 0


def test_planted_interleaved_pairs_are_caught(monkeypatch):
    monkeypatch.setattr(R, "rope_rotate_ref", _interleaved_rotate)
    with pytest.raises(AssertionError):
        test_unit_vector_rotates_into_the_second_half()
