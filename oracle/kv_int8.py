"""CPU oracle for the INT8 KV cache -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  The CUDA path never calls it and shares no code
with it.

What it computes ("LLM Inference Server", *INT8 KV-Cache Quantization*: the
cached K and V are quantised dynamically to int8 per token head; the rule is
the symmetric absmax one of *Required Mathematical Concepts*: s = max|x| / 127,
x_q = round(x / s), x_hat = s * x_q):

* ``quantize_rows_int8`` -- one scale per row of D values, where a row is one
  token of one KV head.  The scale and the division are taken in float32 (the
  stored scale is float32), and round() is round-half-to-even (what the
  page's own PyTorch rounding does).  A row of zeros has s = 0 and codes 0.
* ``dequantize_rows_int8`` -- s * x_q, exact in float64.
* ``append_int8_ref`` -- the per-step in-place KV write of the float oracle,
  with each new (token, head) row quantised on the way into the pool.
* ``decode_int8_ref`` -- decode attention over the dequantised cache: the
  float oracle's softmax(scale * q K_hat^T) V_hat, in float64.
* ``verify_int8_ref`` -- the verification pass of speculative decoding over
  the same cache ("LLM Inference Server", *Batched Scheduling & Speculative
  Decoding*: the target model checks the K drafted tokens in one pass, q_len =
  K + 1 query tokens per sequence): query i of a sequence with context c sits
  at position c - q_len + i and attends the dequantised keys 0..that position.
* ``prefill_int8_ref`` -- the prompt pass over the same cache ("LLM Inference
  Server", Stage 1: all prompt tokens at once under the causal mask): the float
  oracle's prompt pass with each sequence's K and V dequantised.

Layout: codes ``int8 [num_blocks][H_kv][16][D]`` (the float pool's layout),
scales ``float32 [num_blocks][H_kv][16]`` (one per token slot and head).
"""
from __future__ import annotations

import numpy as np

from .paged_attention import BLOCK_SIZE, as_f64, attend, gather_contiguous

QMAX = 127


def _as_f32(x: np.ndarray) -> np.ndarray:
    """Stored element values as float32, exactly (bf16 arrives as raw uint16
    bits; fp16 and fp32 widen exactly)."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.asarray(x, dtype=np.float32)


def quantize_rows_int8(x: np.ndarray):
    """x: [..., D] values to store.  Returns (codes int8 [..., D], scales
    float32 [...]) with, per row, s = max|x| / 127 and codes = round(x / s)
    (half to even), both in float32; zero rows give s = 0 and zero codes.
    The codes never leave [-127, 127]; the clip only guards the float32
    rounding of the largest element."""
    x32 = _as_f32(x)
    amax = np.max(np.abs(x32), axis=-1)
    s = (amax / np.float32(QMAX)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1))
    r = (x32 / safe[..., None]).astype(np.float32)
    codes = np.where(s[..., None] > 0, np.rint(r), np.float32(0))
    codes = np.clip(codes, -QMAX, QMAX).astype(np.int8)
    return codes, s


def dequantize_rows_int8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """x_hat = s * x_q in float64 (exact: a float32 times a small integer)."""
    return scales.astype(np.float64)[..., None] * codes.astype(np.float64)


def append_int8_ref(k_codes: np.ndarray, v_codes: np.ndarray, k_scales: np.ndarray,
                    v_scales: np.ndarray, slot_mapping: np.ndarray, k_new: np.ndarray,
                    v_new: np.ndarray, block_size: int = BLOCK_SIZE):
    """Copies of the four pools with token t's rows (all KV heads) quantised
    and written at slot ``slot_mapping[t]`` (block slot // 16, offset
    slot % 16); negative slots are skipped.  k_new, v_new: [T][H_kv][D]."""
    kc, vc = k_codes.copy(), v_codes.copy()
    ks, vs = k_scales.copy(), v_scales.copy()
    qk, sk = quantize_rows_int8(k_new)
    qv, sv = quantize_rows_int8(v_new)
    for t in range(slot_mapping.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        kc[blk, :, off, :] = qk[t]
        vc[blk, :, off, :] = qv[t]
        ks[blk, :, off] = sk[t]
        vs[blk, :, off] = sv[t]
    return kc, vc, ks, vs


def gather_dequantized(codes: np.ndarray, scales: np.ndarray, block_table: np.ndarray,
                       context_len: int) -> np.ndarray:
    """The sequence's first ``context_len`` positions, dequantised:
    float64 [context_len][H_kv][D]."""
    c = gather_contiguous(codes, block_table, context_len)
    s = gather_contiguous(scales[..., None], block_table, context_len)   # [c][H_kv][1]
    return s * c


def decode_int8_ref(q: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray, k_scales: np.ndarray,
                    v_scales: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
                    scale: float, seqs=None) -> np.ndarray:
    """q: [S][H_q][D] (bf16 bits, fp16 or fp32).  Returns float64 [S][H_q][D]
    (rows not in ``seqs`` stay zero when a subset is asked for)."""
    q64 = as_f64(q)
    S, h_q, d = q64.shape
    out = np.zeros((S, h_q, d), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        c = int(context_lens[s])
        k = gather_dequantized(k_codes, k_scales, block_tables[s], c)
        v = gather_dequantized(v_codes, v_scales, block_tables[s], c)
        out[s] = attend(q64[s], k, v, scale, c)
    return out


def verify_int8_ref(q: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray, k_scales: np.ndarray,
                    v_scales: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
                    scale: float, seqs=None) -> np.ndarray:
    """q: [S][q_len][H_q][D] (bf16 bits, fp16 or fp32), the last accepted token
    and the drafted ones of each sequence, all already in the cache.  Returns
    float64 [S][q_len][H_q][D]; a query whose position is negative (context
    shorter than q_len) sees no key and gives a zero row.  Rows of sequences
    not in ``seqs`` stay zero when a subset is asked for."""
    q64 = as_f64(q)
    S, q_len, h_q, d = q64.shape
    out = np.zeros((S, q_len, h_q, d), dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        c = int(context_lens[s])
        k = gather_dequantized(k_codes, k_scales, block_tables[s], c)
        v = gather_dequantized(v_codes, v_scales, block_tables[s], c)
        for i in range(q_len):
            pos = c - q_len + i
            out[s, i] = attend(q64[s, i], k, v, scale, max(pos + 1, 0))
    return out


def prefill_int8_ref(q: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray, k_scales: np.ndarray,
                     v_scales: np.ndarray, block_tables: np.ndarray, cu_q_lens: np.ndarray,
                     context_lens: np.ndarray, scale: float, rows=None) -> np.ndarray:
    """q: [sum_s q_len_s][H_q][D] (bf16 bits, fp16 or fp32); sequence s owns
    rows cu_q_lens[s] .. cu_q_lens[s+1]-1, its prompt already in the cache.
    Query i of sequence s sits at position p = context_lens[s] - q_len_s + i
    and attends the dequantised keys 0..p.  Returns float64 [sum q_len][H_q][D];
    ``rows`` optionally restricts the computation to a set of global rows
    (the others stay zero)."""
    q64 = as_f64(q)
    total, h_q, d = q64.shape
    out = np.zeros((total, h_q, d), dtype=np.float64)
    want = None if rows is None else set(int(r) for r in rows)
    for s in range(len(context_lens)):
        lo, hi = int(cu_q_lens[s]), int(cu_q_lens[s + 1])
        n = hi - lo
        c = int(context_lens[s])
        if n == 0 or (want is not None and not any(lo <= r < hi for r in want)):
            continue
        k = gather_dequantized(k_codes, k_scales, block_tables[s], c)
        v = gather_dequantized(v_codes, v_scales, block_tables[s], c)
        for i in range(n):
            if want is not None and (lo + i) not in want:
                continue
            out[lo + i] = attend(q64[lo + i], k, v, scale, max(c - n + i + 1, 0))
    return out
