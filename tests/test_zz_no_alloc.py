"""pa_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (a serving loop that may not grow its memory pool, an
embedder that only hands over tensors it already owns, a C host without a
device allocator).  The entry point takes no workspace; its split-K partials
live in the library's built-in 32 MiB per-device array.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it.  It must pass on its own in a
fresh process as well as after the rest of the suite."""
from __future__ import annotations

import ctypes

import pytest
import torch

from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _util import tolerance


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_27_gb300 import build
    build.build()
    return pa.load_library()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(lib):
    """Two consecutive calls (different shapes, both split-K so the built-in
    array is really used, the second after the first left its partials there)
    agree with pa_decode_attention given a caller workspace.  Both run the
    same kernel with the same partition and merge order, so the outputs must
    be bit-identical (which is also within the bf16 parity bar)."""
    dev = "cuda"
    cases = [W.small_random(90, 8, 3000, 32, 8, 128, torch.bfloat16),
             W.small_random(91, 5, 1500, 16, 4, 64, torch.bfloat16)]
    atol, rtol = tolerance(torch.bfloat16)
    for wl in cases:
        st = wl.step(0)
        kp, vp = wl.k_pool.to(dev), wl.v_pool.to(dev)
        pa.pa_append_kv(kp, vp, st.slot_mapping.to(dev), st.k_new.to(dev), st.v_new.to(dev))
        q, bt, ctx = st.q.to(dev), wl.decode_block_tables.contiguous().to(dev), st.context_lens.to(dev)
        mc = int(st.context_lens.max())
        assert pa.pa_decode_workspace_size(wl.num_decode_seqs, wl.num_q_heads, mc, kp) > 0
        ref = torch.empty_like(q)
        pa.pa_decode_attention(ref, q, kp, vp, bt, ctx, wl.scale, max_context_len=mc)
        out = torch.full_like(q, float("nan"))
        pa.pa_decode_attention_noalloc(out, q, kp, vp, bt, ctx, wl.scale, max_context_len=mc)
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs()
        assert bool((err <= atol + rtol * ref.float().abs()).all()), f"max err {err.max().item():.3e}"
        assert torch.equal(out, ref)
    assert pa.pa_device_status() == 0


def test_noalloc_rejects_shapes_beyond_the_array(lib):
    """64 sequences x 32 heads at 64k tokens (1024-token partitions, 64 splits)
    need about 67 MB of partials (64 x 32 x 64 rows of 128 fp32 values):
    refused on the host with a clear message, before any device work.  out and
    q are NULL, so even a call that got past the size check would be refused
    as a null-pointer error and never launch."""
    desc = pa.pa_pool_desc(4096 * 8, 8, 16, 128, pa.PA_BF16)
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode_workspace_size.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(pa.pa_pool_desc)]
    assert lib.pa_decode_workspace_size(64, 32, 65536, 0, ctypes.byref(desc)) > pa.PA_NOALLOC_SCRATCH_BYTES
    fn = lib.pa_decode_attention_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_float] + [ctypes.c_int] * 5 + \
        [ctypes.POINTER(pa.pa_pool_desc), ctypes.c_void_p]
    rc = fn(None, None, None, None, None, None, 0.08, 64, 32, 4096, 65536, 0, ctypes.byref(desc), None)
    assert rc == pa.PA_ERR_INVALID
    msg = pa.pa_last_error()
    assert "scratch" in msg and str(pa.PA_NOALLOC_SCRATCH_BYTES) in msg
