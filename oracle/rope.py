"""CPU oracle for rotary position embedding fused into the KV append -- TEST
INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  The CUDA path never calls it and shares no code
with it.

The pages name RoPE only as one of the steps a fused attention path should
take in ("Mini inference engine (KV cache + sampling + quantization)", Story /
portfolio: fuse qkv_proj + RoPE + attention) and do not define it; the
reading used here is the rotary embedding of the Llama family the pages build
on, in its half-split form: for head dimension D and position p, entry j and
entry j + D/2 of a row (j < D/2) are rotated together by the angle
p * theta^(-2j/D):

    x'[j]       = x[j] cos(a) - x[j + D/2] sin(a)
    x'[j + D/2] = x[j + D/2] cos(a) + x[j] sin(a)

* ``rope_cache_ref`` -- the table of (cos, sin) per (position, j): angles and
  trigonometry in float64, stored as float32 (the table's precision).
* ``rope_rotate_ref`` -- rows [T][H][D] rotated at their positions with a given
  table, in float64 (the table's float32 values widened exactly); the result
  stays float64.
* ``append_rope_ref`` -- the KV append with K rotated on the way into the pool
  (V is copied): returns the float64 rotated K rows and the exact V pool.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import BLOCK_SIZE, as_f64


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2j/D) for j < D/2, float64."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * j / head_dim)


def rope_cache_ref(max_positions: int, head_dim: int, theta: float) -> np.ndarray:
    """float32 [max_positions][D/2][2]: (cos, sin) of p * theta^(-2j/D)."""
    ang = np.arange(max_positions, dtype=np.float64)[:, None] * rope_inv_freq(head_dim, theta)[None, :]
    out = np.empty((max_positions, head_dim // 2, 2), dtype=np.float32)
    out[..., 0] = np.cos(ang)
    out[..., 1] = np.sin(ang)
    return out


def rope_rotate_ref(x: np.ndarray, positions: np.ndarray, cache: np.ndarray) -> np.ndarray:
    """x: [T][H][D] (bf16 bits, fp16 or fp32), positions int [T] -> float64
    [T][H][D] with every row of token t rotated at positions[t]."""
    x64 = as_f64(x)
    half = x64.shape[-1] // 2
    c = cache[positions, :, 0].astype(np.float64)[:, None, :]   # [T][1][D/2]
    s = cache[positions, :, 1].astype(np.float64)[:, None, :]
    lo, hi = x64[..., :half], x64[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def append_rope_ref(v_pool: np.ndarray, slot_mapping: np.ndarray, positions: np.ndarray,
                    k_new: np.ndarray, v_new: np.ndarray, cache: np.ndarray, block_size: int = BLOCK_SIZE):
    """(rotated K rows float64 [T][H][D], V pool after the append).  Token t
    goes to slot slot_mapping[t] (negative: skipped); its K row is the one
    rotate_ref gives at positions[t], its V row is copied bit for bit."""
    k_rot = rope_rotate_ref(k_new, positions, cache)
    v_out = v_pool.copy()
    for t in range(slot_mapping.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        v_out[blk, :, off, :] = v_new[t]
    return k_rot, v_out
