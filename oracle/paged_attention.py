"""CPU oracle for paged KV-cache decode attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  The product path (the CUDA library and its Python
binding) never calls it and shares no code with it: no kernels, no headers, no
helpers, no constants.  It is plain, slow and meant to be checked by eye.

What it computes is the plain definition of the operations, in float64:

* ``append_ref`` -- the in-place KV write of each step ("Mini inference
  engine (KV cache + sampling + quantization)", step 2 *KV cache*: append on
  each step; "LLM Inference Server", Stage 1: new K/V slices written in place
  into pre-allocated buffers), routed through a slot mapping into the pool of
  16-token blocks ("Mini inference engine", step 2 stretch goal; "LLM
  Inference Server", *Paged KV-Cache Block Allocator*).  A pure indexed copy.
* ``gather_contiguous`` -- a sequence's blocks, read through its block table
  ("LLM Inference Server From Scratch", *How it works*, 3 Block Manager:
  block table, paged KV slots), laid end to end: the contiguous per-request
  cache of "Mini inference engine" step 2 / the ``LayerKVCache`` buffer of
  "LLM Inference Server", *Reference Architecture & Verification Code*.
* ``decode_ref`` -- one query token per sequence attending to all of its
  cached keys: softmax(scale * q K^T) V, with grouped-query heads (q head h
  reads KV head floor(h / G)) ("LLM Inference Server From Scratch", *How it
  works*, 4 Attention Kernel: causal mask, GQA; "LLM Inference Server",
  Stage 1: decode passes only the new token, shape (B, 1)).
* ``prefill_ref`` -- the prompt pass (q_len = prompt length, "LLM Inference
  Server", Stage 1) with the causal mask: query i of a sequence of context
  c and q_len n sits at position c - n + i and sees keys 0 .. c - n + i.
* ``kv_cache_bytes`` -- the footprint formula of "LLM Inference Server",
  *Required Mathematical Concepts*: 2 * n_layers * n_kv_heads * d_head *
  seq_len * bytes_per_elem.

Readings where the pages are silent (each is listed with the design notes):
pool layout [num_blocks][H_kv][16][D]; slot = block * 16 + offset with a
negative slot skipped; context lengths count the token appended in this step;
a zero-length context yields a zero output row.

bf16 inputs are accepted as raw ``uint16`` bit patterns and widened exactly
(bits << 16 is the float32 value); every other float dtype is widened with
``astype``.  Outputs stay float64 and are never rounded.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZE = 16


# ---------------------------------------------------------------------------
# exact widening of the stored element types
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the top half of an IEEE float32, so shifting the 16 stored
    bits left by 16 gives the float32 with exactly that value."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# memory footprint ("LLM Inference Server", Required Mathematical Concepts)
# ---------------------------------------------------------------------------

def kv_cache_bytes(n_layers: int, n_kv_heads: int, d_head: int, seq_len: int,
                   bytes_per_elem: int) -> int:
    """K and V (the factor 2) for every layer, KV head, head dimension and
    cached position."""
    return 2 * n_layers * n_kv_heads * d_head * seq_len * bytes_per_elem


# ---------------------------------------------------------------------------
# append: the per-step in-place KV write, through the slot mapping
# ---------------------------------------------------------------------------

def append_ref(k_pool: np.ndarray, v_pool: np.ndarray, slot_mapping: np.ndarray,
               k_new: np.ndarray, v_new: np.ndarray, block_size: int = BLOCK_SIZE):
    """Return copies of the pools with token t's K/V rows (all KV heads)
    written at slot ``slot_mapping[t]``: block ``slot // block_size``,
    offset ``slot % block_size``.  Negative slots are skipped.  The element
    type is whatever the arrays hold (raw bits for bf16), so the copy is
    exact by construction."""
    k_out = k_pool.copy()
    v_out = v_pool.copy()
    for t in range(slot_mapping.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        k_out[blk, :, off, :] = k_new[t]
        v_out[blk, :, off, :] = v_new[t]
    return k_out, v_out


# ---------------------------------------------------------------------------
# block-table gather into the contiguous per-request cache
# ---------------------------------------------------------------------------

def gather_contiguous(pool: np.ndarray, block_table: np.ndarray, context_len: int,
                      block_size: int = BLOCK_SIZE) -> np.ndarray:
    """Logical block j of the sequence is physical block ``block_table[j]``;
    token p lives in logical block p // 16 at offset p % 16.  Returns the
    first ``context_len`` positions as a float64 ``[context_len][H_kv][D]``
    array."""
    n_blocks = (context_len + block_size - 1) // block_size
    h_kv, d = pool.shape[1], pool.shape[3]
    out = np.empty((context_len, h_kv, d), dtype=np.float64)
    for j in range(n_blocks):
        phys = int(block_table[j])
        lo = j * block_size
        hi = min(context_len, lo + block_size)
        # pool[phys] is [H_kv][16][D]; positions lo..hi-1 are offsets 0..hi-lo-1
        out[lo:hi] = as_f64(pool[phys][:, : hi - lo, :]).transpose(1, 0, 2)
    return out


# ---------------------------------------------------------------------------
# attention over a contiguous cache
# ---------------------------------------------------------------------------

def attend(q_row: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
           n_keys: int, return_lse: bool = False):
    """One query row (all H_q heads) against the first ``n_keys`` cached
    positions.  q_row: [H_q][D]; k, v: [>= n_keys][H_kv][D].

    For q head h the KV head is g = h // (H_q / H_kv).  Scores
    x_i = scale * <q_h, k_i>, weights p = exp(x - max x) / sum exp(x - max x),
    output = sum_i p_i v_i.  With ``return_lse`` also returns the natural-log
    log-sum-exp of the scores per head (used only by tests of the split /
    merge algebra).  ``n_keys == 0`` gives a zero row (and lse = -inf)."""
    h_q, d = q_row.shape
    h_kv = k.shape[1]
    group = h_q // h_kv
    out = np.zeros((h_q, d), dtype=np.float64)
    lse = np.full((h_q,), -np.inf, dtype=np.float64)
    if n_keys == 0:
        return (out, lse) if return_lse else out
    for h in range(h_q):
        g = h // group
        kh = k[:n_keys, g, :]
        vh = v[:n_keys, g, :]
        x = scale * (kh @ q_row[h])
        m = np.max(x)
        w = np.exp(x - m)
        z = np.sum(w)
        out[h] = (w / z) @ vh
        lse[h] = m + np.log(z)
    return (out, lse) if return_lse else out


# ---------------------------------------------------------------------------
# decode: one new query token per sequence over its paged cache
# ---------------------------------------------------------------------------

def decode_ref(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
               block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
               seqs=None, return_lse: bool = False):
    """q: [S][H_q][D]; pools [N_blk][H_kv][16][D]; block_tables int [S][max_blocks];
    context_lens int [S].  Returns float64 [S][H_q][D] (rows not listed in
    ``seqs`` are left zero when a subset is asked for)."""
    q64 = as_f64(q)
    S, h_q, d = q64.shape
    out = np.zeros((S, h_q, d), dtype=np.float64)
    lse = np.full((S, h_q), -np.inf, dtype=np.float64)
    for s in (range(S) if seqs is None else seqs):
        c = int(context_lens[s])
        k = gather_contiguous(k_pool, block_tables[s], c)
        v = gather_contiguous(v_pool, block_tables[s], c)
        out[s], lse[s] = attend(q64[s], k, v, scale, c, return_lse=True)
    return (out, lse) if return_lse else out


# ---------------------------------------------------------------------------
# prefill: the causal prompt pass over the same pool
# ---------------------------------------------------------------------------

def prefill_ref(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                block_tables: np.ndarray, cu_q_lens: np.ndarray,
                context_lens: np.ndarray, scale: float, rows=None) -> np.ndarray:
    """q: [sum_s q_len_s][H_q][D], sequence s owns rows cu_q_lens[s] ..
    cu_q_lens[s+1]-1.  Query i of sequence s sits at absolute position
    p = context_lens[s] - q_len_s + i and attends keys 0..p (causal mask).
    ``rows`` optionally restricts the computation to a set of global row
    indices (other rows stay zero)."""
    q64 = as_f64(q)
    total, h_q, d = q64.shape
    out = np.zeros((total, h_q, d), dtype=np.float64)
    want = None if rows is None else set(int(r) for r in rows)
    for s in range(len(context_lens)):
        lo, hi = int(cu_q_lens[s]), int(cu_q_lens[s + 1])
        n = hi - lo
        c = int(context_lens[s])
        if n == 0:
            continue
        if want is not None and not any(lo <= r < hi for r in want):
            continue
        k = gather_contiguous(k_pool, block_tables[s], c)
        v = gather_contiguous(v_pool, block_tables[s], c)
        for i in range(n):
            if want is not None and (lo + i) not in want:
                continue
            pos = c - n + i
            # a query before the first cached position sees no key: zero row
            out[lo + i] = attend(q64[lo + i], k, v, scale, max(pos + 1, 0))
    return out
