"""The C-ABI library on the CPU host: it loads, exports every symbol that
include/pa.h declares, and rejects bad arguments on the host before touching
any GPU (no compute calls here)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from paged_kv_decode_27_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_27_gb300 import build
    build.build()
    return B.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for want in ("pa_append_kv", "pa_decode_attention", "pa_prefill_attention", "pa_decode_workspace_size",
                 "pa_last_error", "pa_device_status", "pa_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(lib):
    assert lib.pa_version() == 1


def _desc(nb=64, hkv=8, bs=16, d=128, dt=B.PA_BF16):
    return B.pa_pool_desc(nb, hkv, bs, d, dt)


FAKE = 0x10000000   # 16-byte aligned, never dereferenced: every call below fails validation first


def _decode(lib, desc, out=FAKE, q=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, cl=FAKE, scale=0.125, S=4, hq=32, mb=8,
            maxc=100, part=0, ws=None, wsb=0):
    return lib.pa_decode_attention(ctypes.c_void_p(out), ctypes.c_void_p(q), ctypes.c_void_p(kp),
                                   ctypes.c_void_p(vp), ctypes.c_void_p(bt), ctypes.c_void_p(cl), scale, S, hq,
                                   mb, maxc, part, ctypes.byref(desc), ctypes.c_void_p(ws), wsb, None)


def test_decode_rejects_bad_arguments_on_the_host(lib):
    d = _desc()
    assert _decode(lib, d, out=0) == B.PA_ERR_INVALID
    assert "null" in B.pa_last_error()
    assert _decode(lib, _desc(bs=32)) == B.PA_ERR_INVALID
    assert _decode(lib, _desc(d=96)) == B.PA_ERR_UNSUPPORTED
    assert _decode(lib, _desc(dt=7)) == B.PA_ERR_UNSUPPORTED
    assert _decode(lib, d, hq=12) == B.PA_ERR_INVALID              # 12 % 8 != 0
    assert _decode(lib, d, hq=8 * 16) == B.PA_ERR_UNSUPPORTED       # group of 16
    assert _decode(lib, d, q=FAKE + 8) == B.PA_ERR_INVALID          # misaligned
    assert _decode(lib, d, maxc=8 * 16 + 1) == B.PA_ERR_INVALID     # exceeds block table
    assert _decode(lib, d, part=17) == B.PA_ERR_INVALID
    assert _decode(lib, d, part=4096) == B.PA_ERR_INVALID
    assert _decode(lib, d, scale=float("nan")) == B.PA_ERR_INVALID
    assert _decode(lib, d, S=-1) == B.PA_ERR_INVALID
    # a split-K shape without workspace, then with a too-small one
    assert _decode(lib, d, maxc=128, part=16) == B.PA_ERR_INVALID
    assert "workspace" in B.pa_last_error()
    assert _decode(lib, d, maxc=128, part=16, ws=FAKE, wsb=16) == B.PA_ERR_INVALID
    assert _decode(lib, _desc(nb=1 << 25)) == B.PA_ERR_UNSUPPORTED  # rows overflow int32


def test_zero_sequences_is_a_no_op(lib):
    assert _decode(lib, _desc(), S=0) == B.PA_OK


def test_append_rejects_bad_arguments_on_the_host(lib):
    d = _desc()
    f = ctypes.c_void_p(FAKE)
    call = lambda kp=f, slots=f, T=4, desc=d: lib.pa_append_kv(kp, f, slots, f, f, T, ctypes.byref(desc), None)
    assert call(kp=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
    assert call(kp=ctypes.c_void_p(FAKE + 4)) == B.PA_ERR_INVALID
    assert call(slots=ctypes.c_void_p(FAKE + 4)) == B.PA_ERR_INVALID
    assert call(T=-1) == B.PA_ERR_INVALID
    assert call(desc=_desc(d=80)) == B.PA_ERR_UNSUPPORTED
    assert call(T=0) == B.PA_OK


def test_prefill_rejects_bad_arguments_on_the_host(lib):
    f = ctypes.c_void_p(FAKE)
    call = lambda desc, maxq=64, maxc=64, out=f: lib.pa_prefill_attention(
        out, f, f, f, f, f, f, 0.1, 2, 32, 4, maxq, maxc, ctypes.byref(desc), None)
    assert call(_desc(dt=B.PA_F32)) == B.PA_ERR_UNSUPPORTED
    assert call(_desc(), maxq=65) == B.PA_ERR_INVALID
    assert call(_desc(), maxc=65) == B.PA_ERR_INVALID
    assert call(_desc(), out=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
    # the run-time schedule counts (query tile, sequence, head) items in
    # int32: 65535 sequences x 64 heads x 512 tiles of 128 rows is refused
    big = lib.pa_prefill_attention(f, f, f, f, f, f, f, 0.1, 65535, 64, 4096, 65536, 65536,
                                   ctypes.byref(_desc()), None)
    assert big == B.PA_ERR_UNSUPPORTED
    assert "query tiles" in B.pa_last_error()


def test_int8_prefill_validates_on_the_host(lib):
    """The INT8 prompt pass: the pool must be INT8 with a bf16/fp16 act_dtype,
    the workspace present and large enough.  The workspace is the fp16 K and V
    copies of num_seqs x ceil(max_context_len / 16) blocks (each 256-byte
    aligned) and their int32 block table, whatever the activations' type:
    bf16 queries are converted and the output stored by the pass itself."""
    f = ctypes.c_void_p(FAKE)
    i8 = _desc(dt=B.PA_I8)
    al = lambda n: ((n + 255) // 256) * 256
    pool = 2 * 4 * 8 * 16 * 128 * 2                      # 2 seqs x 4 blocks x 8 heads x 16 x 128 x 2 bytes
    size = lib.pa_prefill_int8_workspace_size(2, 64, ctypes.byref(i8))
    assert size == 2 * al(pool) + 2 * 4 * 4
    assert lib.pa_prefill_int8_workspace_size(2, 50, ctypes.byref(i8)) == size    # 50 tokens: 4 blocks too
    assert lib.pa_prefill_int8_workspace_size(0, 64, ctypes.byref(i8)) == 0
    assert lib.pa_prefill_int8_workspace_size(2, 64, ctypes.byref(_desc(dt=B.PA_BF16))) == 0
    assert lib.pa_prefill_int8_workspace_size(-1, 64, ctypes.byref(i8)) == 0
    f16 = size
    call = lambda desc, act=B.PA_BF16, ws=f, wsb=size, maxq=64, maxc=64, S=2: lib.pa_prefill_attention_int8(
        f, f, f, f, f, f, f, f, f, 0.1, S, 32, 4, maxq, maxc, act, ctypes.byref(desc), ws, wsb, None)
    assert call(_desc(dt=B.PA_BF16)) == B.PA_ERR_INVALID          # float pool
    assert call(i8, act=B.PA_F32) == B.PA_ERR_INVALID
    assert call(i8, ws=ctypes.c_void_p(0)) == B.PA_ERR_INVALID    # no workspace
    assert call(i8, wsb=size - 1) == B.PA_ERR_INVALID              # too small
    assert call(i8, act=B.PA_F16, wsb=f16 - 1) == B.PA_ERR_INVALID
    assert call(i8, maxq=65) == B.PA_ERR_INVALID
    assert call(i8, S=0) == B.PA_OK                                # nothing to do
    # the float prompt pass refuses the INT8 pool
    assert lib.pa_prefill_attention(f, f, f, f, f, f, f, 0.1, 2, 32, 4, 64, 64, ctypes.byref(i8), None) == \
        B.PA_ERR_INVALID


def test_workspace_size_and_partition(lib):
    d = _desc(d=128)
    # batch 64, 8 KV heads, contexts to 8224: 1024-token partitions, 9 splits
    assert lib.pa_decode_partition_size(64, 8224, 0, ctypes.byref(d)) == 1024
    n = lib.pa_decode_workspace_size(64, 32, 8224, 0, ctypes.byref(d))
    rows = 64 * 32 * 9
    o_end = 256 * 1024 + rows * 128 * 4          # counters, then partial outputs
    assert n == ((o_end + 255) // 256) * 256 + rows * 4
    # a batch that fits one resident wave (456 units) takes the smallest
    # partition that still fits: 8 x 8 pairs of <= 2063 tokens -> 512 (320 units)
    assert lib.pa_decode_partition_size(8, 2063, 0, ctypes.byref(_desc(d=64))) == 512
    # 8 x 8 pairs of 8192 tokens: 2048 (256 units; 1024 would need 512)
    assert lib.pa_decode_partition_size(8, 8192, 0, ctypes.byref(d)) == 2048
    # tiny batches stop at 256 tokens
    assert lib.pa_decode_partition_size(2, 40, 0, ctypes.byref(_desc(hkv=2, d=64))) == 256
    # one partition covers everything: no workspace
    assert lib.pa_decode_workspace_size(4, 32, 512, 512, ctypes.byref(d)) == 0
    assert lib.pa_decode_partition_size(4, 512, 256, ctypes.byref(d)) == 256


def test_partition_choice_follows_the_sm_count(lib):
    """The automatic partition is sized to one resident wave of 3 CTAs per SM
    of the device it is asked for, not to a fixed SM count."""
    lib.pa_decode_partition_size_on.restype = ctypes.c_int
    lib.pa_decode_partition_size_on.argtypes = [ctypes.c_int] * 3 + [ctypes.POINTER(B.pa_pool_desc), ctypes.c_int]
    d = _desc(d=128)
    on = lambda S, maxc, sms, part=0, desc=d: lib.pa_decode_partition_size_on(S, maxc, part, ctypes.byref(desc), sms)
    # 8 x 8 pairs of 8192 tokens: 64 pairs x 4 partitions of 2048 = 256 units.
    # 152 SMs (456 slots): 2048 (1024 would need 512 units)
    assert on(8, 8192, 152) == 2048
    # 176 SMs (528 slots): 1024 fits; 352 SMs (1056): 512 fits (1024 units)
    assert on(8, 8192, 176) == 1024 and on(8, 8192, 352) == 512
    # 64 SMs (192 slots): not even 2048-token partitions fit one wave -> 1024, several waves
    assert on(8, 8192, 64) == 1024
    # every choice stays in [256, 2048]
    for sms in (1, 8, 76, 132, 152, 160, 1000, 100000):
        p = on(3, 3000, sms)
        assert 256 <= p <= 2048 and p % 16 == 0
    # a forced partition is returned as is; a bad SM count is refused
    assert on(8, 8192, 64, part=128) == 128
    assert on(8, 8192, 0) == 0 and lib.pa_last_error()


def test_no_gpu_means_cuda_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _decode(lib, _desc(), maxc=100, mb=8, part=512) == B.PA_ERR_CUDA


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        B.load_library(str(tmp_path / "nope.so"))


def _decode8(lib, desc, act=B.PA_BF16, ks=FAKE, out=FAKE, maxc=100, part=512, S=4):
    f = ctypes.c_void_p(FAKE)
    return lib.pa_decode_attention_int8(ctypes.c_void_p(out), f, f, f, ctypes.c_void_p(ks), f, f, f, 0.125, S, 32,
                                        8, maxc, part, act, ctypes.byref(desc), None, 0, None)


def test_int8_cache_entry_points_validate_on_the_host(lib):
    i8 = _desc(dt=B.PA_I8)
    # the float calls refuse an INT8 pool, the INT8 calls refuse a float pool
    assert _decode(lib, i8) == B.PA_ERR_INVALID and "int8" in B.pa_last_error()
    assert _decode8(lib, _desc(dt=B.PA_BF16)) == B.PA_ERR_INVALID
    assert _decode8(lib, i8, act=B.PA_F32) == B.PA_ERR_INVALID
    assert _decode8(lib, i8, act=B.PA_I8) == B.PA_ERR_INVALID
    assert _decode8(lib, i8, ks=0) == B.PA_ERR_INVALID
    assert _decode8(lib, i8, ks=FAKE + 4) == B.PA_ERR_INVALID        # scales misaligned
    assert _decode8(lib, _desc(d=96, dt=B.PA_I8)) == B.PA_ERR_UNSUPPORTED
    assert _decode8(lib, i8, S=0) == B.PA_OK
    f = ctypes.c_void_p(FAKE)
    app = lambda desc=i8, act=B.PA_BF16, T=4, ks=f: lib.pa_append_kv_int8(f, f, ks, f, f, f, f, T, act,
                                                                          ctypes.byref(desc), None)
    assert app(desc=_desc()) == B.PA_ERR_INVALID
    assert app(act=B.PA_F32) == B.PA_ERR_INVALID
    assert app(ks=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
    assert app(T=-1) == B.PA_ERR_INVALID
    assert app(T=0) == B.PA_OK
    fl = ctypes.c_void_p(FAKE)
    assert lib.pa_append_kv(fl, fl, fl, fl, fl, 4, ctypes.byref(i8), None) == B.PA_ERR_INVALID
    # the workspace of an INT8 cache has the float formula (partials are fp32)
    assert lib.pa_decode_workspace_size(64, 32, 8224, 0, ctypes.byref(_desc(d=128, dt=B.PA_I8))) == \
        lib.pa_decode_workspace_size(64, 32, 8224, 0, ctypes.byref(_desc(d=128)))


def _verify8(lib, desc, act=B.PA_BF16, ql=5, hq=32, maxc=100, part=512, S=4):
    f = ctypes.c_void_p(FAKE)
    return lib.pa_verify_attention_int8(f, f, f, f, f, f, f, f, 0.125, S, ql, hq, 8, maxc, part, act,
                                        ctypes.byref(desc), None, 0, None)


def test_int8_verify_validates_on_the_host(lib):
    i8 = _desc(dt=B.PA_I8)
    assert _verify8(lib, _desc(dt=B.PA_BF16)) == B.PA_ERR_INVALID      # float pool
    assert _verify8(lib, i8, act=B.PA_F32) == B.PA_ERR_INVALID
    assert _verify8(lib, i8, ql=0) == B.PA_ERR_INVALID
    assert _verify8(lib, i8, ql=9) == B.PA_ERR_UNSUPPORTED              # G = 4: 36 columns
    assert _verify8(lib, i8, ql=5, S=0) == B.PA_OK
    # the float verify call refuses the INT8 pool
    f = ctypes.c_void_p(FAKE)
    assert lib.pa_verify_attention(f, f, f, f, f, f, 0.125, 4, 5, 32, 8, 100, 512, ctypes.byref(i8), None, 0,
                                   None) == B.PA_ERR_INVALID
    # INT8 verification splits by partitions: its workspace is the decode
    # workspace of S x q_len rows at the same partition size
    d8 = _desc(d=128, dt=B.PA_I8)
    for S, ql, maxc, part in ((64, 5, 8224, 512), (3, 2, 4000, 256), (8, 8, 100, 16)):
        assert lib.pa_verify_workspace_size(S, ql, 32, maxc, part, ctypes.byref(d8)) == \
            lib.pa_decode_workspace_size(S * ql, 32, maxc, part, ctypes.byref(d8))
    # The automatic partition of a wide INT8 verification pass (G x q_len > 8
    # query columns: 2 CTAs per SM) fills one wave of 2 x 152 CTAs when it can
    # (1 sequence x 8 KV heads x 33 partitions of 256 tokens = 264) and
    # otherwise takes 2048-token partitions (the batch of 64: 2560 units).
    auto = lambda S, ql, maxc: lib.pa_verify_workspace_size(S, ql, 32, maxc, 0, ctypes.byref(d8))
    assert auto(64, 5, 8224) == lib.pa_decode_workspace_size(64 * 5, 32, 8224, 2048, ctypes.byref(d8))
    assert auto(1, 5, 8192) == lib.pa_decode_workspace_size(5, 32, 8192, 256, ctypes.byref(d8))
    # two query columns per KV head (one 8-column tile) keep the decode rule
    assert lib.pa_verify_workspace_size(64, 2, 8, 8224, 0, ctypes.byref(d8)) == \
        lib.pa_decode_workspace_size(64 * 2, 8, 8224, 1024, ctypes.byref(d8))


def test_int8_without_gpu_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _decode8(lib, _desc(dt=B.PA_I8)) == B.PA_ERR_CUDA


def test_verify_validates_on_the_host(lib):
    f = ctypes.c_void_p(FAKE)
    call = lambda desc=_desc(), ql=5, hq=32, part=512: lib.pa_verify_attention(
        f, f, f, f, f, f, 0.1, 4, ql, hq, 8, 100, part, ctypes.byref(desc), None, 0, None)
    assert call(ql=0) == B.PA_ERR_INVALID
    assert call(desc=_desc(dt=B.PA_F32)) == B.PA_ERR_UNSUPPORTED
    assert call(desc=_desc(dt=B.PA_I8)) == B.PA_ERR_INVALID
    assert call(hq=64, ql=5) == B.PA_ERR_UNSUPPORTED        # G 8 x 5 = 40 columns
    # the verify workspace holds q_len rows per sequence; q_len 1 is the decode workspace
    d = _desc()
    assert lib.pa_verify_workspace_size(64, 1, 32, 8224, 0, ctypes.byref(d)) == \
        lib.pa_decode_workspace_size(64, 32, 8224, 0, ctypes.byref(d))
    # head dim 128, q_len > 1: the tensor-core kernel keeps one partial per stream-K
    # segment; with 1024-token partitions a CTA's range costs at least 8 tiles, so a
    # context of 8224 tokens (65 tiles, plus its start-up cost) meets at most
    # ceil(65 / 8) + 2 = 11 ranges
    rows = 64 * 5 * 32 * 11
    assert lib.pa_verify_workspace_size(64, 5, 32, 8224, 0, ctypes.byref(d)) == \
        ((256 * 1024 + rows * 128 * 4 + 255) // 256) * 256 + rows * 4
    # head dim 64 stays on the mma.sync kernel: one partial per 1024-token partition
    d64 = _desc(d=64)
    rows = 64 * 5 * 32 * 9
    assert lib.pa_verify_workspace_size(64, 5, 32, 8224, 0, ctypes.byref(d64)) == \
        ((256 * 1024 + rows * 64 * 4 + 255) // 256) * 256 + rows * 4


def test_rope_entry_points_validate_on_the_host(lib):
    f = ctypes.c_void_p(FAKE)
    assert lib.pa_rope_cache(f, 10, 96, ctypes.c_double(1e4), None) == B.PA_ERR_UNSUPPORTED
    assert lib.pa_rope_cache(f, 10, 128, ctypes.c_double(0.0), None) == B.PA_ERR_INVALID
    assert lib.pa_rope_cache(ctypes.c_void_p(FAKE + 4), 10, 128, ctypes.c_double(1e4), None) == B.PA_ERR_INVALID
    assert lib.pa_rope_cache(f, 0, 128, ctypes.c_double(1e4), None) == B.PA_OK
    d = _desc()
    app = lambda pos=f, T=4, desc=d: lib.pa_append_kv_rope(f, f, f, pos, f, f, T, f, 100, ctypes.byref(desc), None)
    assert app(pos=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
    assert app(pos=ctypes.c_void_p(FAKE + 2)) == B.PA_ERR_INVALID
    assert app(desc=_desc(dt=B.PA_I8)) == B.PA_ERR_INVALID
    assert app(T=0) == B.PA_OK
    assert lib.pa_apply_rope(f, f, 4, 8, 128, B.PA_I8, f, 100, None) == B.PA_ERR_UNSUPPORTED
    assert lib.pa_apply_rope(ctypes.c_void_p(FAKE + 8), f, 4, 8, 128, B.PA_BF16, f, 100, None) == B.PA_ERR_INVALID


def test_decode_step_validates_on_the_host(lib):
    f = ctypes.c_void_p(FAKE)
    call = lambda kn=f, d=_desc(): lib.pa_decode_step(f, f, f, f, kn, f, f, f, 0.1, 4, 32, 8, 100, 512,
                                                      ctypes.byref(d), None, 0, None)
    assert call(kn=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
    assert call(kn=ctypes.c_void_p(FAKE + 8)) == B.PA_ERR_INVALID
    assert call(d=_desc(dt=B.PA_I8)) == B.PA_ERR_INVALID


def test_copy_blocks_validate_on_the_host(lib):
    f = ctypes.c_void_p(FAKE)
    cp = lambda desc, n=2, pairs=f: lib.pa_copy_blocks(f, f, pairs, n, ctypes.byref(desc), None)
    cp8 = lambda desc, n=2, pairs=f, ks=f: lib.pa_copy_blocks_int8(f, f, ks, f, pairs, n, ctypes.byref(desc), None)
    assert cp(_desc(dt=B.PA_I8)) == B.PA_ERR_INVALID            # an INT8 cache has its own call
    assert cp8(_desc(dt=B.PA_BF16)) == B.PA_ERR_INVALID         # and it takes INT8 pools only
    assert cp8(_desc(dt=B.PA_I8), n=-1) == B.PA_ERR_INVALID
    assert cp8(_desc(dt=B.PA_I8), n=0) == B.PA_OK                # nothing to copy
    assert cp8(_desc(dt=B.PA_I8), ks=ctypes.c_void_p(FAKE + 4)) == B.PA_ERR_INVALID   # scales not 16-byte aligned
    assert cp8(_desc(dt=B.PA_I8), pairs=ctypes.c_void_p(FAKE + 4)) == B.PA_ERR_INVALID
    assert cp8(_desc(dt=B.PA_I8), ks=ctypes.c_void_p(0)) == B.PA_ERR_INVALID
