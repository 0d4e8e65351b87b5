"""Pins of the float64 CPU oracle against things other than itself.

Each test compares the oracle with an independent statement of the result:
torch's own scaled-dot-product attention (float64, CPU), pure-Python brute
force, closed forms (constant V, one-token context, uniform weights, a
hand-worked two-token example), invariants of attention over a set (block and
token permutations), the paged == contiguous identity and the full-sequence
recomputation check of "LLM Inference Server", Stage 1 (cached decoding must
match full recomputation to 1e-5), the KV footprint formula of its *Required
Mathematical Concepts*, and the algebra of merging split softmaxes.  The last
group plants plausible mistakes in copies of the oracle and checks that the
pins catch them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import paged_attention as pa_ref
from paged_kv_decode_27_gb300 import workloads as W
from _util import to_np, to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent statements used by the pins
# ---------------------------------------------------------------------------

def sdpa_rows(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal_offset=None):
    """torch.nn.functional.scaled_dot_product_attention in float64 on the CPU.
    q_rows [n][H_q][D]; k, v [c][H_kv][D]; KV heads repeated G times so that q
    head h reads KV head h // G.  With ``causal_offset`` = c - n, row i sees
    keys 0 .. c - n + i; otherwise every row sees every key."""
    n, hq, d = q_rows.shape
    c, hkv, _ = k.shape
    g = hq // hkv
    qt = torch.from_numpy(q_rows).permute(1, 0, 2).unsqueeze(0)           # [1,H_q,n,D]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
    mask = None
    if causal_offset is not None:
        i = torch.arange(n).unsqueeze(1)
        j = torch.arange(c).unsqueeze(0)
        mask = j <= (i + causal_offset)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.squeeze(0).permute(1, 0, 2).numpy()


def brute_decode_one(q_row, k, v, scale, n_keys):
    """Pure-Python loops, math.exp, no vectorisation."""
    hq, d = len(q_row), len(q_row[0])
    hkv = len(k[0])
    g = hq // hkv
    out = [[0.0] * d for _ in range(hq)]
    for h in range(hq):
        kh = h // g
        xs = []
        for i in range(n_keys):
            dot = 0.0
            for e in range(d):
                dot += float(q_row[h][e]) * float(k[i][kh][e])
            xs.append(scale * dot)
        m = max(xs)
        ws = [math.exp(x - m) for x in xs]
        z = sum(ws)
        for e in range(d):
            acc = 0.0
            for i in range(n_keys):
                acc += ws[i] * float(v[i][kh][e])
            out[h][e] = acc / z
    return out


def _wl_np(wl: W.Workload, t: int = 0):
    st = wl.step(t)
    return st, to_np(wl.k_pool), to_np(wl.v_pool), wl.decode_block_tables.numpy(), st.context_lens.numpy()


# ---------------------------------------------------------------------------
# widening and footprint
# ---------------------------------------------------------------------------

def test_bf16_widening_matches_torch():
    g = torch.Generator().manual_seed(7)
    x = (torch.randn(4096, generator=g) * 100).to(torch.bfloat16)
    special = torch.tensor([0.0, -0.0, 1.0, -2.0, float("inf"), -float("inf"), 1e-40, 3.0e38],
                           dtype=torch.float32).to(torch.bfloat16)
    x = torch.cat([x, special])
    got = oracle.bf16_bits_to_f64(to_np(x))
    want = to_f64(x)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))
    assert oracle.bf16_bits_to_f64(np.array([0x3F80, 0xC000], dtype=np.uint16)).tolist() == [1.0, -2.0]


def test_kv_cache_bytes_golden():
    rows = 0
    with open(os.path.join(GOLDEN, "kv_cache_bytes.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split()
            nl, hkv, d, L, e, want = (int(p) for p in parts[:6])
            assert oracle.kv_cache_bytes(nl, hkv, d, L, e) == want, line
            rows += 1
    assert rows >= 5


@pytest.mark.parametrize("factory", [W.tiny_fp32, W.prefix_shared_8k])
def test_pool_bytes_per_token_match_formula(factory):
    wl = factory()
    per_tok = (wl.k_pool.numel() + wl.v_pool.numel()) * wl.elem_bytes // (wl.num_blocks * 16)
    assert per_tok == oracle.kv_cache_bytes(1, wl.num_kv_heads, wl.head_dim, 1, wl.elem_bytes)


# ---------------------------------------------------------------------------
# append: a pure indexed copy
# ---------------------------------------------------------------------------

def _canary_pool(n_blk, hkv, d, dtype, fill_bits):
    t = torch.empty((n_blk, hkv, 16, d), dtype=dtype)
    t.view({2: torch.int16, 4: torch.int32}[t.element_size()]).fill_(fill_bits)
    return t


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_append_ref_against_index_put(dtype):
    """Library scatter (index_put over a [slot][H_kv][D] view) as the
    independent statement; canary bytes outside written slots untouched."""
    g = torch.Generator().manual_seed(3)
    n_blk, hkv, d, T = 7, 3, 8, 20
    canary = 0x7FC1 if dtype == torch.bfloat16 else 0x7FC00001  # NaN payloads
    kp = _canary_pool(n_blk, hkv, d, dtype, canary)
    vp = _canary_pool(n_blk, hkv, d, dtype, canary)
    slots = torch.randperm(n_blk * 16, generator=g)[:T].to(torch.int64)
    slots[3] = -1
    slots[11] = -5
    k_new = torch.randn((T, hkv, d), generator=g).to(dtype)
    v_new = torch.randn((T, hkv, d), generator=g).to(dtype)
    k_out, v_out = oracle.append_ref(to_np(kp), to_np(vp), slots.numpy(), to_np(k_new), to_np(v_new))

    for pool, new, got in ((kp, k_new, k_out), (vp, v_new, v_out)):
        want = pool.clone()
        flat = want.permute(0, 2, 1, 3).reshape(n_blk * 16, hkv, d).clone()
        keep = slots >= 0
        flat.index_put_((slots[keep],), new[keep])
        want = flat.reshape(n_blk, 16, hkv, d).permute(0, 2, 1, 3).contiguous()
        assert np.array_equal(got.view(np.uint8), to_np(want).view(np.uint8))
    # untouched slots still hold the canary bit pattern
    written = set(int(s) for s in slots if s >= 0)
    kb = k_out.view(np.uint16 if dtype == torch.bfloat16 else np.uint32)
    for slot in range(n_blk * 16):
        if slot not in written:
            assert (kb[slot // 16, :, slot % 16, :] == canary).all()


def test_append_then_gather_reads_new_token_at_last_position():
    """The off-by-one pitfall of "Mini inference engine" (prompt length vs
    write index): after appending a sequence's new token at position c-1, the
    gathered cache's last row is that token."""
    wl = W.tiny_fp32()
    st = wl.step(0)
    kp, vp = oracle.append_ref(to_np(wl.k_pool), to_np(wl.v_pool), st.slot_mapping.numpy(),
                               to_np(st.k_new), to_np(st.v_new))
    bt = wl.decode_block_tables.numpy()
    for s, c in enumerate(st.context_lens.tolist()):
        k = oracle.gather_contiguous(kp, bt[s], c)
        v = oracle.gather_contiguous(vp, bt[s], c)
        assert np.array_equal(k[c - 1], to_f64(st.k_new[s]))
        assert np.array_equal(v[c - 1], to_f64(st.v_new[s]))


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def test_decode_matches_torch_sdpa_tiny():
    wl = W.tiny_fp32()
    st, kp, vp, bt, ctx = _wl_np(wl)
    kp, vp = oracle.append_ref(kp, vp, st.slot_mapping.numpy(), to_np(st.k_new), to_np(st.v_new))
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    for s in range(len(ctx)):
        k = oracle.gather_contiguous(kp, bt[s], int(ctx[s]))
        v = oracle.gather_contiguous(vp, bt[s], int(ctx[s]))
        want = sdpa_rows(to_f64(st.q[s:s + 1]), k, v, wl.scale)[0]
        assert np.max(np.abs(out[s] - want)) < 1e-13


@pytest.mark.parametrize("seed,hq,hkv,d", [(1, 2, 1, 4), (2, 6, 3, 8), (3, 4, 4, 5), (4, 8, 2, 3)])
def test_decode_matches_brute_force(seed, hq, hkv, d):
    wl = W.small_random(seed, num_seqs=3, max_ctx=40, hq=hq, hkv=hkv, d=d, dtype=torch.float32)
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    for s in range(len(ctx)):
        k = oracle.gather_contiguous(kp, bt[s], int(ctx[s])).tolist()
        v = oracle.gather_contiguous(vp, bt[s], int(ctx[s])).tolist()
        want = np.array(brute_decode_one(to_f64(st.q[s]).tolist(), k, v, wl.scale, int(ctx[s])))
        assert np.max(np.abs(out[s] - want)) < 1e-12


def test_brute_force_on_tiny_workload_directly_from_pool():
    """Brute force that walks the pool itself (block id, offset) rather than
    the oracle's gather."""
    wl = W.tiny_fp32()
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    for s in range(2):
        c = int(ctx[s])
        k = [[kp[bt[s][p // 16], h, p % 16].tolist() for h in range(2)] for p in range(c)]
        v = [[vp[bt[s][p // 16], h, p % 16].tolist() for h in range(2)] for p in range(c)]
        want = np.array(brute_decode_one(st.q[s].tolist(), k, v, wl.scale, c))
        assert np.max(np.abs(out[s] - want)) < 1e-12


def test_hand_worked_two_token_example():
    """scale = 1, q = (1, 0), k0 = (0, 0), k1 = (ln 3, 0): scores 0 and ln 3,
    weights 1/4 and 3/4, so out = v0/4 + 3 v1/4."""
    q = np.array([[[1.0, 0.0]]])
    k = np.zeros((1, 1, 16, 2))
    v = np.zeros((1, 1, 16, 2))
    k[0, 0, 1, 0] = math.log(3.0)
    v[0, 0, 0] = [4.0, -8.0]
    v[0, 0, 1] = [8.0, 4.0]
    out = oracle.decode_ref(q, k, v, np.array([[0]]), np.array([2]), 1.0)
    assert np.allclose(out[0, 0], [0.25 * 4 + 0.75 * 8, 0.25 * -8 + 0.75 * 4], atol=1e-15, rtol=0)


def test_constant_v_gives_v():
    wl = W.small_random(5, num_seqs=3, max_ctx=70, hq=8, hkv=2, d=16, dtype=torch.float32)
    st, kp, vp, bt, ctx = _wl_np(wl)
    vc = np.empty_like(vp)
    vc[:] = np.linspace(-3, 3, vp.shape[-1], dtype=np.float32)
    out = oracle.decode_ref(to_np(st.q), kp, vc, bt, ctx, wl.scale)
    assert np.max(np.abs(out - vc[0, 0, 0].astype(np.float64))) < 1e-14


def test_single_token_context_is_exactly_its_v():
    wl = W.small_random(6, num_seqs=4, max_ctx=1, hq=4, hkv=2, d=8, dtype=torch.float32,
                        ctx=[1, 1, 1, 1])
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    for s in range(4):
        for h in range(4):
            assert np.array_equal(out[s, h], vp[bt[s][0], h // 2, 0].astype(np.float64))


def test_zero_scale_gives_mean_of_v():
    wl = W.small_random(7, num_seqs=3, max_ctx=50, hq=4, hkv=1, d=8, dtype=torch.float32)
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, 0.0)
    for s in range(3):
        v = oracle.gather_contiguous(vp, bt[s], int(ctx[s]))
        assert np.max(np.abs(out[s] - np.mean(v[:, 0, :], axis=0))) < 1e-14


def test_zero_context_gives_zero_row():
    wl = W.small_random(8, num_seqs=3, max_ctx=20, hq=4, hkv=2, d=8, dtype=torch.float32,
                        ctx=[5, 0, 17])
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    assert np.array_equal(out[1], np.zeros_like(out[1]))
    assert np.abs(out[0]).sum() > 0 and np.abs(out[2]).sum() > 0


def test_paged_equals_contiguous_bit_exact():
    """The same tokens laid out with an identity block table give the
    identical float64 result: the gather is exact."""
    wl = W.small_random(9, num_seqs=3, max_ctx=90, hq=4, hkv=2, d=16, dtype=torch.bfloat16)
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    for s in range(3):
        nb = (int(ctx[s]) + 15) // 16
        kc = kp[bt[s][:nb]]
        vc = vp[bt[s][:nb]]
        ident = np.arange(nb)[None, :]
        o2 = oracle.decode_ref(to_np(st.q[s:s + 1]), kc, vc, ident, ctx[s:s + 1], wl.scale)
        assert np.array_equal(out[s], o2[0])


def test_physical_block_shuffle_is_bit_exact():
    wl = W.small_random(10, num_seqs=4, max_ctx=120, hq=8, hkv=2, d=8, dtype=torch.float32)
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    rng = np.random.default_rng(0)
    perm = rng.permutation(kp.shape[0])           # new position of old block b is perm[b]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    out2 = oracle.decode_ref(to_np(st.q), kp2, vp2, perm[bt], ctx, wl.scale)
    assert np.array_equal(out, out2)


def test_token_permutation_invariance():
    """Attention without position encoding is a function of the set of
    (k, v) pairs: permuting positions (K and V together) keeps the output."""
    wl = W.small_random(11, num_seqs=1, max_ctx=1, hq=4, hkv=2, d=16, dtype=torch.float32, ctx=[77])
    st, kp, vp, bt, ctx = _wl_np(wl)
    k = oracle.gather_contiguous(kp, bt[0], 77)
    v = oracle.gather_contiguous(vp, bt[0], 77)
    q = to_f64(st.q[0])
    a = oracle.attend(q, k, v, wl.scale, 77)
    p = np.random.default_rng(1).permutation(77)
    b = oracle.attend(q, k[p], v[p], wl.scale, 77)
    assert np.max(np.abs(a - b)) < 1e-13


def test_full_recompute_last_row_equals_decode():
    """"LLM Inference Server", Stage 1 acceptance: cached decoding matches
    full-sequence recomputation to 1e-5.  With no model, the recomputation is
    causal attention of all c positions over the full cache (torch SDPA); its
    last row must equal the decode output for the same query."""
    wl = W.small_random(12, num_seqs=3, max_ctx=150, hq=8, hkv=2, d=32, dtype=torch.bfloat16)
    st, kp, vp, bt, ctx = _wl_np(wl)
    out = oracle.decode_ref(to_np(st.q), kp, vp, bt, ctx, wl.scale)
    g = torch.Generator().manual_seed(99)
    for s in range(3):
        c = int(ctx[s])
        k = oracle.gather_contiguous(kp, bt[s], c)
        v = oracle.gather_contiguous(vp, bt[s], c)
        q_all = torch.randn((c, 8, 32), generator=g, dtype=torch.float64).numpy()
        q_all[-1] = to_f64(st.q[s])
        full = sdpa_rows(q_all, k, v, wl.scale, causal_offset=0)
        assert np.max(np.abs(full[-1] - out[s])) < 1e-5
        assert np.max(np.abs(full[-1] - out[s])) < 1e-12


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def _prefill_case(seed, prompt_lens, prior, hq=4, hkv=2, d=16, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    ctx = [p + n for p, n in zip(prior, prompt_lens)]
    wl = W.small_random(seed, num_seqs=len(ctx), max_ctx=max(ctx), hq=hq, hkv=hkv, d=d,
                        dtype=dtype, ctx=ctx)
    total = sum(prompt_lens)
    q = torch.randn((total, hq, d), generator=g).to(dtype)
    cu = np.concatenate([[0], np.cumsum(prompt_lens)]).astype(np.int32)
    return wl, q, cu, np.array(ctx, dtype=np.int32)


def test_prefill_matches_sdpa_causal():
    wl, q, cu, ctx = _prefill_case(13, [33, 1, 64, 17], [0, 0, 0, 0])
    kp, vp, bt = to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy()
    out = oracle.prefill_ref(to_np(q), kp, vp, bt, cu, ctx, wl.scale)
    for s in range(4):
        lo, hi = cu[s], cu[s + 1]
        k = oracle.gather_contiguous(kp, bt[s], int(ctx[s]))
        v = oracle.gather_contiguous(vp, bt[s], int(ctx[s]))
        want = sdpa_rows(to_f64(q[lo:hi]), k, v, wl.scale, causal_offset=int(ctx[s]) - (hi - lo))
        assert np.max(np.abs(out[lo:hi] - want)) < 1e-13


def test_prefill_with_cached_prefix_matches_sdpa():
    """Queries placed after an already-cached prefix (c - q_len > 0)."""
    wl, q, cu, ctx = _prefill_case(14, [5, 20, 16], [40, 3, 16])
    kp, vp, bt = to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy()
    out = oracle.prefill_ref(to_np(q), kp, vp, bt, cu, ctx, wl.scale)
    for s in range(3):
        lo, hi = cu[s], cu[s + 1]
        k = oracle.gather_contiguous(kp, bt[s], int(ctx[s]))
        v = oracle.gather_contiguous(vp, bt[s], int(ctx[s]))
        want = sdpa_rows(to_f64(q[lo:hi]), k, v, wl.scale, causal_offset=int(ctx[s]) - (hi - lo))
        assert np.max(np.abs(out[lo:hi] - want)) < 1e-13


def test_prefill_row_equals_decode_at_that_position():
    """Prefill/decode split of "LLM Inference Server", Stage 1: row i of the
    prompt pass equals a decode of that query with context position + 1."""
    wl, q, cu, ctx = _prefill_case(15, [40], [0])
    kp, vp, bt = to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy()
    pre = oracle.prefill_ref(to_np(q), kp, vp, bt, cu, ctx, wl.scale)
    for i in (0, 15, 16, 39):
        dec = oracle.decode_ref(to_np(q[i:i + 1]), kp, vp, bt[:1], np.array([i + 1]), wl.scale)
        assert np.array_equal(pre[i], dec[0])


def test_prefill_query_before_the_context_is_zero():
    """q_len larger than the context: the leading queries sit at negative
    positions, see no key and give zero rows (the zero-context reading); the
    others are ordinary causal rows."""
    wl = W.small_random(19, num_seqs=1, max_ctx=1, hq=4, hkv=2, d=8, dtype=torch.float32, ctx=[3])
    q = np.random.default_rng(3).standard_normal((5, 4, 8))
    out = oracle.prefill_ref(q, to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy(),
                             np.array([0, 5]), np.array([3]), 0.5)
    assert not out[:2].any()
    k = oracle.gather_contiguous(to_np(wl.k_pool), wl.block_tables[0].numpy(), 3)
    v = oracle.gather_contiguous(to_np(wl.v_pool), wl.block_tables[0].numpy(), 3)
    for i in range(2, 5):
        ref = sdpa_rows(q[i:i + 1], k[:i - 1], v[:i - 1], 0.5)
        assert np.max(np.abs(out[i] - ref[0])) < 1e-12


def test_prefill_brute_force_tiny():
    wl, q, cu, ctx = _prefill_case(16, [3, 5], [2, 0], hq=2, hkv=1, d=3)
    kp, vp, bt = to_np(wl.k_pool), to_np(wl.v_pool), wl.block_tables.numpy()
    out = oracle.prefill_ref(to_np(q), kp, vp, bt, cu, ctx, wl.scale)
    for s in range(2):
        lo, hi = int(cu[s]), int(cu[s + 1])
        c = int(ctx[s])
        k = [[kp[bt[s][p // 16], 0, p % 16].tolist()] for p in range(c)]
        v = [[vp[bt[s][p // 16], 0, p % 16].tolist()] for p in range(c)]
        for i in range(hi - lo):
            want = brute_decode_one(q[lo + i].tolist(), k, v, wl.scale, c - (hi - lo) + i + 1)
            assert np.max(np.abs(out[lo + i] - np.array(want))) < 1e-12


# ---------------------------------------------------------------------------
# split-K algebra: merging partial softmaxes by log-sum-exp is exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("parts", [1, 2, 3, 7, 40])
def test_lse_merge_of_splits_equals_whole(parts):
    wl = W.small_random(17, num_seqs=1, max_ctx=1, hq=4, hkv=2, d=16, dtype=torch.float32, ctx=[97])
    st, kp, vp, bt, ctx = _wl_np(wl)
    k = oracle.gather_contiguous(kp, bt[0], 97)
    v = oracle.gather_contiguous(vp, bt[0], 97)
    q = to_f64(st.q[0])
    whole, whole_lse = oracle.attend(q, k, v, wl.scale, 97, return_lse=True)
    edges = np.linspace(0, 97, parts + 1).round().astype(int)
    outs, lses = [], []
    for a, b in zip(edges[:-1], edges[1:]):
        o, l = oracle.attend(q, k[a:b], v[a:b], wl.scale, b - a, return_lse=True)
        outs.append(o)
        lses.append(l)
    lses = np.stack(lses)                       # [P][H_q]
    M = np.max(lses, axis=0)
    w = np.exp(lses - M)                        # empty parts have lse -inf -> weight 0
    merged = np.einsum("ph,phd->hd", w, np.stack(outs)) / w.sum(axis=0)[:, None]
    assert np.max(np.abs(merged - whole)) < 1e-13
    assert np.max(np.abs(M + np.log(w.sum(axis=0)) - whole_lse)) < 1e-12


# ---------------------------------------------------------------------------
# planted mistakes: copies of the oracle with one plausible bug each must fail
# ---------------------------------------------------------------------------

def _mutant_attend(kind):
    def attend(q_row, k, v, scale, n_keys, return_lse=False):
        h_q, d = q_row.shape
        h_kv = k.shape[1]
        group = h_q // h_kv
        out = np.zeros((h_q, d))
        lse = np.full((h_q,), -np.inf)
        if n_keys == 0:
            return (out, lse) if return_lse else out
        for h in range(h_q):
            g = h % h_kv if kind == "gqa_modulo" else h // group
            n = n_keys - 1 if kind == "drop_last_key" else n_keys
            kh, vh = k[:n, g, :], v[:n, g, :]
            x = (kh @ q_row[h]) * (1.0 if kind == "no_scale" else scale)
            m = np.max(x)
            w = np.exp(x - m)
            out[h] = (w / (1.0 if kind == "no_normalise" else w.sum())) @ vh
            lse[h] = m + np.log(w.sum())
        return (out, lse) if return_lse else out
    return attend


def _mutant_gather(kind):
    def gather(pool, block_table, context_len, block_size=16):
        nb = (context_len + block_size - 1) // block_size
        h_kv, d = pool.shape[1], pool.shape[3]
        out = np.empty((context_len, h_kv, d))
        for j in range(nb):
            phys = int(block_table[nb - 1 - j]) if kind == "reversed_table" else int(block_table[j])
            lo = j * block_size
            hi = min(context_len, lo + block_size)
            src = pa_ref.as_f64(pool[phys])
            if kind == "head_offset_swapped":
                # reads [offset][head] as if the block were token-major
                src = src.reshape(16, h_kv, d).transpose(1, 0, 2)
            out[lo:hi] = src[:, : hi - lo, :].transpose(1, 0, 2)
        return out
    return gather


@pytest.mark.parametrize("kind", ["gqa_modulo", "drop_last_key", "no_scale", "no_normalise"])
def test_planted_attend_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(pa_ref, "attend", _mutant_attend(kind))
    with pytest.raises(AssertionError):
        test_decode_matches_torch_sdpa_tiny()


@pytest.mark.parametrize("kind", ["reversed_table", "head_offset_swapped"])
def test_planted_gather_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(pa_ref, "gather_contiguous", _mutant_gather(kind))
    # the brute force walks the pool itself, so it sees through the gather
    with pytest.raises(AssertionError):
        test_brute_force_on_tiny_workload_directly_from_pool()
