"""Python binding of libpa (``include/pa.h``): argument marshalling only.

Each function has the name of the C entry point it calls and takes torch
tensors already on the GPU.  It checks shapes, dtypes and contiguity, passes
raw device pointers and the current CUDA stream, and raises ``PaError`` on a
non-OK status.  Every step of the computation runs in the CUDA library; there
is no fallback: if ``lib/libpa.so`` has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libpa.so")

PA_F32, PA_BF16, PA_F16, PA_I8 = 0, 1, 2, 3
PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE = 0, -1, -2, -3, -4
PA_ERR_NO_BLOCKS = -5
PA_DEV_BAD_SLOT, PA_DEV_BAD_BLOCK_ID, PA_DEV_BAD_CONTEXT, PA_DEV_WAIT_TIMEOUT = 1, 2, 4, 8
PA_DEV_BAD_POSITION = 16
PA_DEV_RANGE = 32
BLOCK_SIZE = 16

_DTYPES = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16, torch.int8: PA_I8}


class PaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpa error {code}: {msg}")
        self.code = code


class pa_pool_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("block_size", ctypes.c_int), ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int)]


class pa_bm_stats(ctypes.Structure):
    _fields_ = [("hit_blocks", ctypes.c_int64), ("miss_blocks", ctypes.c_int64), ("cow_copies", ctypes.c_int64),
                ("evictions", ctypes.c_int64), ("free_blocks", ctypes.c_int32),
                ("cached_free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpa.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    pdesc = ctypes.POINTER(pa_pool_desc)
    L.pa_version.restype = i32
    L.pa_version.argtypes = []
    L.pa_last_error.restype = ctypes.c_char_p
    L.pa_last_error.argtypes = []
    L.pa_append_kv.restype = i32
    L.pa_append_kv.argtypes = [vp, vp, vp, vp, vp, i32, pdesc, vp]
    L.pa_decode_workspace_size.restype = sz
    L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, pdesc]
    L.pa_decode_partition_size.restype = i32
    L.pa_decode_partition_size.argtypes = [i32, i32, i32, pdesc]
    L.pa_decode_partition_size_on.restype = i32
    L.pa_decode_partition_size_on.argtypes = [i32, i32, i32, pdesc, i32]
    L.pa_decode_attention.restype = i32
    L.pa_decode_attention.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, pdesc,
                                      vp, sz, vp]
    L.pa_decode_step.restype = i32
    L.pa_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, pdesc, vp, sz, vp]
    L.pa_prefill_attention.restype = i32
    L.pa_prefill_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32,
                                       pdesc, vp]
    L.pa_device_status.restype = i32
    L.pa_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
    L.pa_verify_workspace_size.restype = sz
    L.pa_verify_workspace_size.argtypes = [i32, i32, i32, i32, i32, pdesc]
    L.pa_verify_attention.restype = i32
    L.pa_verify_attention.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, i32, pdesc, vp, sz,
                                      vp]
    L.pa_rope_cache.restype = i32
    L.pa_rope_cache.argtypes = [vp, i32, i32, ctypes.c_double, vp]
    L.pa_append_kv_rope.restype = i32
    L.pa_append_kv_rope.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, pdesc, vp]
    L.pa_apply_rope.restype = i32
    L.pa_apply_rope.argtypes = [vp, vp, i32, i32, i32, i32, vp, i32, vp]
    L.pa_bm_create.restype = vp
    L.pa_bm_create.argtypes = [i32, i32, i32]
    L.pa_bm_destroy.restype = None
    L.pa_bm_destroy.argtypes = [vp]
    L.pa_bm_add_sequence.restype = i32
    L.pa_bm_add_sequence.argtypes = [vp, i32, vp, i32, vp]
    L.pa_bm_append.restype = i32
    L.pa_bm_append.argtypes = [vp, i32, vp, i32, vp, vp, i32, ctypes.POINTER(ctypes.c_int)]
    L.pa_bm_append_step.restype = i32
    L.pa_bm_append_step.argtypes = [vp, vp, vp, i32, vp, vp, i32, ctypes.POINTER(ctypes.c_int)]
    L.pa_bm_fork.restype = i32
    L.pa_bm_fork.argtypes = [vp, i32, i32]
    L.pa_bm_free_sequence.restype = i32
    L.pa_bm_free_sequence.argtypes = [vp, i32]
    L.pa_bm_block_tables.restype = i32
    L.pa_bm_block_tables.argtypes = [vp, vp, i32, vp, i32, vp]
    L.pa_bm_get_stats.restype = i32
    L.pa_bm_get_stats.argtypes = [vp, ctypes.POINTER(pa_bm_stats)]
    L.pa_copy_blocks.restype = i32
    L.pa_copy_blocks.argtypes = [vp, vp, vp, i32, pdesc, vp]
    L.pa_copy_blocks_int8.restype = i32
    L.pa_copy_blocks_int8.argtypes = [vp, vp, vp, vp, vp, i32, pdesc, vp]
    L.pa_append_kv_int8.restype = i32
    L.pa_append_kv_int8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, pdesc, vp]
    L.pa_decode_attention_int8.restype = i32
    L.pa_decode_attention_int8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, i32,
                                           pdesc, vp, sz, vp]
    L.pa_verify_attention_int8.restype = i32
    L.pa_verify_attention_int8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, i32,
                                           i32, pdesc, vp, sz, vp]
    L.pa_prefill_int8_workspace_size.restype = sz
    L.pa_prefill_int8_workspace_size.argtypes = [i32, i32, pdesc]
    L.pa_prefill_attention_int8.restype = i32
    L.pa_prefill_attention_int8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, i32,
                                            pdesc, vp, sz, vp]
    _lib = L
    return L


def pa_last_error() -> str:
    return load_library().pa_last_error().decode()


def _check(rc: int):
    if rc != PA_OK:
        raise PaError(rc, pa_last_error())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def pool_desc(k_pool: torch.Tensor) -> pa_pool_desc:
    """Geometry of a pool tensor laid out [num_blocks][H_kv][16][D]."""
    if k_pool.dim() != 4 or k_pool.shape[2] != BLOCK_SIZE:
        raise ValueError(f"pool must be [num_blocks][H_kv][16][D], got {tuple(k_pool.shape)}")
    if k_pool.dtype not in _DTYPES:
        raise ValueError(f"unsupported pool dtype {k_pool.dtype}")
    n, h, b, d = k_pool.shape
    return pa_pool_desc(int(n), int(h), int(b), int(d), _DTYPES[k_pool.dtype])


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(name: str, t: torch.Tensor):
    _need(t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")


def _pools(k_pool, v_pool):
    _cuda_contig("k_pool", k_pool)
    _cuda_contig("v_pool", v_pool)
    _need(k_pool.shape == v_pool.shape and k_pool.dtype == v_pool.dtype,
          "k_pool and v_pool must have the same shape and dtype")
    return pool_desc(k_pool)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def pa_append_kv(k_pool: torch.Tensor, v_pool: torch.Tensor, slot_mapping: torch.Tensor,
                 k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
    """Write k_new/v_new [T][H_kv][D] into the pools at slot_mapping (int64 [T])."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("slot_mapping", slot_mapping), ("k_new", k_new), ("v_new", v_new)):
        _cuda_contig(n, t)
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.dim() == 1, "slot_mapping must be int64 [T]")
    T = slot_mapping.shape[0]
    shape = (T, k_pool.shape[1], k_pool.shape[3])
    _need(tuple(k_new.shape) == shape and tuple(v_new.shape) == shape, f"k_new/v_new must be {shape}")
    _need(k_new.dtype == k_pool.dtype and v_new.dtype == k_pool.dtype, "k_new/v_new dtype must match the pool")
    L = load_library()
    _check(L.pa_append_kv(_ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping), _ptr(k_new), _ptr(v_new),
                          int(T), ctypes.byref(desc), _stream(stream)))


def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, max_context_len: int,
                             k_pool: torch.Tensor, partition_size: int = 0) -> int:
    L = load_library()
    desc = pool_desc(k_pool)
    n = L.pa_decode_workspace_size(int(num_seqs), int(num_q_heads), int(max_context_len),
                                   int(partition_size), ctypes.byref(desc))
    msg = pa_last_error()
    if msg:
        raise PaError(PA_ERR_INVALID, msg)
    return int(n)


def pa_decode_partition_size(num_seqs: int, max_context_len: int, k_pool: torch.Tensor,
                             partition_size: int = 0) -> int:
    L = load_library()
    desc = pool_desc(k_pool)
    return int(L.pa_decode_partition_size(int(num_seqs), int(max_context_len), int(partition_size),
                                          ctypes.byref(desc)))


def pa_decode_partition_size_on(num_seqs: int, max_context_len: int, k_pool: torch.Tensor, sm_count: int,
                                partition_size: int = 0) -> int:
    """The automatic partition choice for a device of ``sm_count`` SMs."""
    L = load_library()
    desc = pool_desc(k_pool)
    n = int(L.pa_decode_partition_size_on(int(num_seqs), int(max_context_len), int(partition_size),
                                          ctypes.byref(desc), int(sm_count)))
    if n == 0:
        raise PaError(PA_ERR_INVALID, pa_last_error())
    return n


def pa_decode_attention(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                        max_context_len: int, partition_size: int = 0,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out, q: [S][H_q][D]; block_tables int32 [S][max_blocks]; context_lens int32 [S].
    ``workspace`` (uint8 CUDA tensor, zero-filled before its first use) is
    allocated here, zero-filled, when not given."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_pool.shape[3], "q must be [S][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype == k_pool.dtype, "out/q shape or dtype mismatch")
    S, hq = int(q.shape[0]), int(q.shape[1])
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    if workspace is None:   # the library checks the size of a workspace it is given
        need = pa_decode_workspace_size(S, hq, max_context_len, k_pool, partition_size)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_decode_attention(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 _ptr(context_lens), float(scale), S, hq, int(block_tables.shape[1]),
                                 int(max_context_len), int(partition_size), ctypes.byref(desc),
                                 _ptr(workspace), int(ws_bytes), _stream(stream)))


def pa_verify_workspace_size(num_seqs: int, q_len: int, num_q_heads: int, max_context_len: int,
                             k_pool: torch.Tensor, partition_size: int = 0) -> int:
    L = load_library()
    desc = pool_desc(k_pool)
    n = L.pa_verify_workspace_size(int(num_seqs), int(q_len), int(num_q_heads), int(max_context_len),
                                   int(partition_size), ctypes.byref(desc))
    msg = pa_last_error()
    if msg:
        raise PaError(PA_ERR_INVALID, msg)
    return int(n)


def pa_verify_attention(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                        max_context_len: int, partition_size: int = 0,
                        workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out, q: [S][q_len][H_q][D]: the last q_len positions of each sequence
    (already appended), each attending causally to the cache."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 4 and q.shape[3] == k_pool.shape[3], "q must be [S][q_len][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype == k_pool.dtype, "out/q shape or dtype mismatch")
    S, ql, hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    if workspace is None:
        need = pa_verify_workspace_size(S, ql, hq, max_context_len, k_pool, partition_size)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_verify_attention(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                 _ptr(context_lens), float(scale), S, ql, hq, int(block_tables.shape[1]),
                                 int(max_context_len), int(partition_size), ctypes.byref(desc), _ptr(workspace),
                                 int(ws_bytes), _stream(stream)))


def pa_decode_step(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                   k_new: torch.Tensor, v_new: torch.Tensor, block_tables: torch.Tensor,
                   context_lens: torch.Tensor, scale: float, max_context_len: int, partition_size: int = 0,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append each sequence's new token (k_new / v_new [S][H_kv][D], at
    position context_lens[s] - 1) and decode, in one launch."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("out", out), ("q", q), ("k_new", k_new), ("v_new", v_new), ("block_tables", block_tables),
                 ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_pool.shape[3], "q must be [S][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype == k_pool.dtype, "out/q shape or dtype mismatch")
    S, hq = int(q.shape[0]), int(q.shape[1])
    shape = (S, k_pool.shape[1], k_pool.shape[3])
    _need(tuple(k_new.shape) == shape and tuple(v_new.shape) == shape, f"k_new/v_new must be {shape}")
    _need(k_new.dtype == v_new.dtype == k_pool.dtype, "k_new/v_new dtype must match the pool")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    if workspace is None:
        need = pa_decode_workspace_size(S, hq, max_context_len, k_pool, partition_size)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_decode_step(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_new), _ptr(v_new),
                            _ptr(block_tables), _ptr(context_lens), float(scale), S, hq, int(block_tables.shape[1]),
                            int(max_context_len), int(partition_size), ctypes.byref(desc), _ptr(workspace),
                            int(ws_bytes), _stream(stream)))


def pa_prefill_attention(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                         block_tables: torch.Tensor, cu_q_lens: torch.Tensor, context_lens: torch.Tensor,
                         scale: float, max_q_len: int, max_context_len: int, stream=None) -> None:
    """out, q: [sum q_len][H_q][D]; cu_q_lens int32 [S+1]; context_lens int32 [S]."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("cu_q_lens", cu_q_lens),
                 ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_pool.shape[3], "q must be [sum q_len][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype == k_pool.dtype, "out/q shape or dtype mismatch")
    S = int(context_lens.shape[0])
    _need(cu_q_lens.dtype == torch.int32 and tuple(cu_q_lens.shape) == (S + 1,), "cu_q_lens must be int32 [S+1]")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    L = load_library()
    _check(L.pa_prefill_attention(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                  _ptr(cu_q_lens), _ptr(context_lens), float(scale), S, int(q.shape[1]),
                                  int(block_tables.shape[1]), int(max_q_len), int(max_context_len),
                                  ctypes.byref(desc), _stream(stream)))


def pa_device_status(stream=None) -> int:
    """Read and clear the device status word (PA_DEV_* bits); 0 when clean."""
    L = load_library()
    st = ctypes.c_int(0)
    rc = L.pa_device_status(ctypes.byref(st), _stream(stream))
    if rc not in (PA_OK, PA_ERR_DEVICE):
        raise PaError(rc, pa_last_error())
    return int(st.value)


PA_NOALLOC_SCRATCH_BYTES = 32 << 20


def pa_decode_attention_noalloc(out: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                max_context_len: int, partition_size: int = 0, stream=None) -> None:
    """pa_decode_attention for callers that cannot allocate device memory: no
    workspace argument, and nothing is allocated here or in the library; the
    split-K partials use the library's built-in 32 MiB per-device array.
    Shapes needing more scratch raise PaError; calls overlapping on the GPU
    share that array and must be serialised."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_pool.shape[3], "q must be [S][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype == k_pool.dtype, "out/q shape or dtype mismatch")
    S, hq = int(q.shape[0]), int(q.shape[1])
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    fn = L.pa_decode_attention_noalloc
    if fn.argtypes is None:
        vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.restype = i32
        fn.argtypes = [vp, vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, i32, ctypes.POINTER(pa_pool_desc), vp]
    _check(fn(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables), _ptr(context_lens),
              float(scale), S, hq, int(block_tables.shape[1]), int(max_context_len), int(partition_size),
              ctypes.byref(desc), _stream(stream)))


# ---------------------------------------------------------------------------
# INT8 KV cache: int8 code pools [N_blk][H_kv][16][D] + float32 scales [N_blk][H_kv][16]
# ---------------------------------------------------------------------------

def _int8_cache(k_codes, v_codes, k_scales, v_scales):
    desc = _pools(k_codes, v_codes)
    _need(k_codes.dtype == torch.int8, "INT8 cache code pools must be torch.int8")
    for n, t in (("k_scales", k_scales), ("v_scales", v_scales)):
        _cuda_contig(n, t)
        _need(t.dtype == torch.float32 and tuple(t.shape) == tuple(k_codes.shape[:3]),
              f"{n} must be float32 {tuple(k_codes.shape[:3])}")
    return desc


def _act(t: torch.Tensor) -> int:
    _need(t.dtype in (torch.bfloat16, torch.float16), "INT8 cache activations must be bf16 or fp16")
    return _DTYPES[t.dtype]


def pa_append_kv_int8(k_codes: torch.Tensor, v_codes: torch.Tensor, k_scales: torch.Tensor,
                      v_scales: torch.Tensor, slot_mapping: torch.Tensor, k_new: torch.Tensor,
                      v_new: torch.Tensor, stream=None) -> None:
    """Quantise k_new/v_new [T][H_kv][D] (bf16/fp16) per (token, head) row into
    the INT8 cache at slot_mapping (int64 [T])."""
    desc = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    for n, t in (("slot_mapping", slot_mapping), ("k_new", k_new), ("v_new", v_new)):
        _cuda_contig(n, t)
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.dim() == 1, "slot_mapping must be int64 [T]")
    T = slot_mapping.shape[0]
    shape = (T, k_codes.shape[1], k_codes.shape[3])
    _need(tuple(k_new.shape) == shape and tuple(v_new.shape) == shape, f"k_new/v_new must be {shape}")
    _need(k_new.dtype == v_new.dtype, "k_new and v_new must share a dtype")
    L = load_library()
    _check(L.pa_append_kv_int8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), _ptr(slot_mapping),
                               _ptr(k_new), _ptr(v_new), int(T), _act(k_new), ctypes.byref(desc),
                               _stream(stream)))


def pa_decode_attention_int8(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                             k_scales: torch.Tensor, v_scales: torch.Tensor, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, scale: float, max_context_len: int,
                             partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                             stream=None) -> None:
    """pa_decode_attention over an INT8 cache; out, q: [S][H_q][D] bf16/fp16.
    ``workspace`` as in pa_decode_attention (sized with the int8 code pool)."""
    desc = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_codes.shape[3], "q must be [S][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype, "out/q shape or dtype mismatch")
    S, hq = int(q.shape[0]), int(q.shape[1])
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    if workspace is None:
        need = pa_decode_workspace_size(S, hq, max_context_len, k_codes, partition_size)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_decode_attention_int8(_ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                                      _ptr(v_scales), _ptr(block_tables), _ptr(context_lens), float(scale), S, hq,
                                      int(block_tables.shape[1]), int(max_context_len), int(partition_size),
                                      _act(q), ctypes.byref(desc), _ptr(workspace), int(ws_bytes),
                                      _stream(stream)))



def pa_verify_attention_int8(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                             k_scales: torch.Tensor, v_scales: torch.Tensor, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, scale: float, max_context_len: int,
                             partition_size: int = 0, workspace: Optional[torch.Tensor] = None,
                             stream=None) -> None:
    """pa_verify_attention over an INT8 cache; out, q: [S][q_len][H_q][D]
    bf16/fp16, the last q_len positions of each sequence (already appended),
    each attending causally to the cache.  ``workspace`` as in
    pa_verify_attention (sized with the int8 code pool)."""
    desc = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 4 and q.shape[3] == k_codes.shape[3], "q must be [S][q_len][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype, "out/q shape or dtype mismatch")
    S, ql, hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    _need(context_lens.dtype == torch.int32 and tuple(context_lens.shape) == (S,), "context_lens must be int32 [S]")
    L = load_library()
    if workspace is None:
        need = pa_verify_workspace_size(S, ql, hq, max_context_len, k_codes, partition_size)
        if need > 0:
            workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_verify_attention_int8(_ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                                      _ptr(v_scales), _ptr(block_tables), _ptr(context_lens), float(scale), S, ql,
                                      hq, int(block_tables.shape[1]), int(max_context_len), int(partition_size),
                                      _act(q), ctypes.byref(desc), _ptr(workspace), int(ws_bytes),
                                      _stream(stream)))

def pa_prefill_int8_workspace_size(num_seqs: int, max_context_len: int, k_codes: torch.Tensor) -> int:
    """Bytes of workspace pa_prefill_attention_int8 needs (k_codes: the int8
    pool)."""
    L = load_library()
    desc = pool_desc(k_codes)
    n = L.pa_prefill_int8_workspace_size(int(num_seqs), int(max_context_len), ctypes.byref(desc))
    msg = pa_last_error()
    if msg:
        raise PaError(PA_ERR_INVALID, msg)
    return int(n)


def pa_prefill_attention_int8(out: torch.Tensor, q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor,
                              k_scales: torch.Tensor, v_scales: torch.Tensor, block_tables: torch.Tensor,
                              cu_q_lens: torch.Tensor, context_lens: torch.Tensor, scale: float, max_q_len: int,
                              max_context_len: int, workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """pa_prefill_attention over an INT8 cache; out, q: [sum q_len][H_q][D]
    bf16/fp16.  ``workspace``: a device uint8 tensor of at least
    pa_prefill_int8_workspace_size() bytes (allocated here when omitted)."""
    desc = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    for n, t in (("out", out), ("q", q), ("block_tables", block_tables), ("cu_q_lens", cu_q_lens),
                 ("context_lens", context_lens)):
        _cuda_contig(n, t)
    _need(q.dim() == 3 and q.shape[2] == k_codes.shape[3], "q must be [sum q_len][H_q][D]")
    _need(out.shape == q.shape and out.dtype == q.dtype, "out/q shape or dtype mismatch")
    S = int(context_lens.shape[0])
    _need(cu_q_lens.dtype == torch.int32 and tuple(cu_q_lens.shape) == (S + 1,), "cu_q_lens must be int32 [S+1]")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2 and block_tables.shape[0] == S,
          "block_tables must be int32 [S][max_blocks]")
    L = load_library()
    if workspace is None:
        need = pa_prefill_int8_workspace_size(S, max_context_len, k_codes)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.pa_prefill_attention_int8(_ptr(out), _ptr(q), _ptr(k_codes), _ptr(v_codes), _ptr(k_scales),
                                       _ptr(v_scales), _ptr(block_tables), _ptr(cu_q_lens), _ptr(context_lens),
                                       float(scale), S, int(q.shape[1]), int(block_tables.shape[1]), int(max_q_len),
                                       int(max_context_len), _act(q), ctypes.byref(desc), _ptr(workspace),
                                       int(ws_bytes), _stream(stream)))


# ---------------------------------------------------------------------------
# rotary position embedding (half-split, Llama form)
# ---------------------------------------------------------------------------

def pa_rope_cache(cos_sin: torch.Tensor, theta: float, stream=None) -> None:
    """Fill cos_sin, float32 CUDA [max_positions][D/2][2], with (cos, sin) of
    p * theta^(-2j/D)."""
    _cuda_contig("cos_sin", cos_sin)
    _need(cos_sin.dtype == torch.float32 and cos_sin.dim() == 3 and cos_sin.shape[2] == 2,
          "cos_sin must be float32 [max_positions][D/2][2]")
    L = load_library()
    _check(L.pa_rope_cache(_ptr(cos_sin), int(cos_sin.shape[0]), int(2 * cos_sin.shape[1]), float(theta),
                           _stream(stream)))


def pa_append_kv_rope(k_pool: torch.Tensor, v_pool: torch.Tensor, slot_mapping: torch.Tensor,
                      positions: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cos_sin: torch.Tensor,
                      stream=None) -> None:
    """pa_append_kv with K rotated at positions (int32 [T]) on the way in."""
    desc = _pools(k_pool, v_pool)
    for n, t in (("slot_mapping", slot_mapping), ("positions", positions), ("k_new", k_new), ("v_new", v_new),
                 ("cos_sin", cos_sin)):
        _cuda_contig(n, t)
    T = slot_mapping.shape[0]
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.dim() == 1, "slot_mapping must be int64 [T]")
    _need(positions.dtype == torch.int32 and tuple(positions.shape) == (T,), "positions must be int32 [T]")
    shape = (T, k_pool.shape[1], k_pool.shape[3])
    _need(tuple(k_new.shape) == shape and tuple(v_new.shape) == shape, f"k_new/v_new must be {shape}")
    _need(k_new.dtype == k_pool.dtype and v_new.dtype == k_pool.dtype, "k_new/v_new dtype must match the pool")
    _need(cos_sin.dtype == torch.float32 and cos_sin.dim() == 3 and cos_sin.shape[1] * 2 == k_pool.shape[3],
          "cos_sin must be float32 [max_positions][D/2][2]")
    L = load_library()
    _check(L.pa_append_kv_rope(_ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping), _ptr(positions), _ptr(k_new),
                               _ptr(v_new), int(T), _ptr(cos_sin), int(cos_sin.shape[0]), ctypes.byref(desc),
                               _stream(stream)))


def pa_apply_rope(x: torch.Tensor, positions: torch.Tensor, cos_sin: torch.Tensor, stream=None) -> None:
    """Rotate x [T][H][D] in place at positions (int32 [T])."""
    for n, t in (("x", x), ("positions", positions), ("cos_sin", cos_sin)):
        _cuda_contig(n, t)
    _need(x.dim() == 3 and x.dtype in _DTYPES and x.dtype != torch.int8, "x must be [T][H][D] fp32/bf16/fp16")
    _need(positions.dtype == torch.int32 and tuple(positions.shape) == (x.shape[0],), "positions must be int32 [T]")
    _need(cos_sin.dtype == torch.float32 and cos_sin.dim() == 3 and cos_sin.shape[1] * 2 == x.shape[2],
          "cos_sin must be float32 [max_positions][D/2][2]")
    L = load_library()
    _check(L.pa_apply_rope(_ptr(x), _ptr(positions), int(x.shape[0]), int(x.shape[1]), int(x.shape[2]),
                           _DTYPES[x.dtype], _ptr(cos_sin), int(cos_sin.shape[0]), _stream(stream)))


# ---------------------------------------------------------------------------
# block manager with a prefix cache (host side)
# ---------------------------------------------------------------------------

def _i32(xs) -> "np.ndarray":
    import numpy as np
    return np.ascontiguousarray(np.asarray(xs, dtype=np.int32))


def pa_bm_create(num_blocks: int, max_blocks_per_seq: int, max_seqs: int) -> ctypes.c_void_p:
    h = load_library().pa_bm_create(int(num_blocks), int(max_blocks_per_seq), int(max_seqs))
    if not h:
        raise PaError(PA_ERR_INVALID, pa_last_error())
    return ctypes.c_void_p(h)


def pa_bm_destroy(bm) -> None:
    load_library().pa_bm_destroy(bm)


def pa_bm_add_sequence(bm, seq: int, prompt):
    """-> (number of prompt tokens found in the prefix cache, int64 slots of every prompt position)."""
    import numpy as np
    p = _i32(prompt)
    slots = np.zeros(max(1, p.size), dtype=np.int64)
    rc = load_library().pa_bm_add_sequence(bm, int(seq), p.ctypes.data, int(p.size), slots.ctypes.data)
    if rc < 0:
        raise PaError(rc, pa_last_error())
    return rc, slots[:p.size]


def pa_bm_append(bm, seq: int, tokens):
    """-> (int64 slots of the new tokens, list of copy-on-write pairs (src, dst))."""
    import numpy as np
    t = _i32(tokens)
    slots = np.zeros(max(1, t.size), dtype=np.int64)
    copies = np.zeros(2, dtype=np.int32)
    n = ctypes.c_int(0)
    _check(load_library().pa_bm_append(bm, int(seq), t.ctypes.data, int(t.size), slots.ctypes.data,
                                       copies.ctypes.data, 1, ctypes.byref(n)))
    return slots[:t.size], [(int(copies[2 * i]), int(copies[2 * i + 1])) for i in range(n.value)]


def pa_bm_append_step(bm, seq_ids, tokens, slots_out=None):
    """One token per listed sequence.  -> (int64 slots, copy-on-write pairs).
    ``slots_out`` (int64 array or pinned CPU tensor of len(seq_ids)) receives
    the slots in place when given."""
    import numpy as np
    ids, toks = _i32(seq_ids), _i32(tokens)
    _need(ids.size == toks.size, "one token per sequence")
    if slots_out is None:
        slots_out = np.zeros(max(1, ids.size), dtype=np.int64)
    ptr = slots_out.data_ptr() if hasattr(slots_out, "data_ptr") else slots_out.ctypes.data
    copies = np.zeros(2 * max(1, ids.size), dtype=np.int32)
    n = ctypes.c_int(0)
    _check(load_library().pa_bm_append_step(bm, ids.ctypes.data, toks.ctypes.data, int(ids.size), ptr,
                                            copies.ctypes.data, max(1, ids.size), ctypes.byref(n)))
    return slots_out, [(int(copies[2 * i]), int(copies[2 * i + 1])) for i in range(n.value)]


def pa_bm_block_tables_into(bm, seq_ids, tables_out, ctx_out) -> None:
    """pa_bm_block_tables writing into given int32 host buffers (e.g. pinned
    tensors [n][max_blocks] and [n])."""
    ids = _i32(seq_ids)
    _check(load_library().pa_bm_block_tables(bm, ids.ctypes.data, int(ids.size), tables_out.data_ptr(),
                                             int(tables_out.shape[1]), ctx_out.data_ptr()))


def pa_bm_fork(bm, parent: int, child: int) -> None:
    _check(load_library().pa_bm_fork(bm, int(parent), int(child)))


def pa_bm_free_sequence(bm, seq: int) -> None:
    _check(load_library().pa_bm_free_sequence(bm, int(seq)))


def pa_bm_block_tables(bm, seq_ids, max_blocks: int):
    """-> (int32 [n][max_blocks] tables, int32 [n] context lengths), host numpy."""
    import numpy as np
    ids = _i32(seq_ids)
    tables = np.zeros((max(1, ids.size), max_blocks), dtype=np.int32)
    ctx = np.zeros(max(1, ids.size), dtype=np.int32)
    _check(load_library().pa_bm_block_tables(bm, ids.ctypes.data, int(ids.size), tables.ctypes.data,
                                             int(max_blocks), ctx.ctypes.data))
    return tables[:ids.size], ctx[:ids.size]


def pa_bm_get_stats(bm) -> dict:
    st = pa_bm_stats()
    _check(load_library().pa_bm_get_stats(bm, ctypes.byref(st)))
    return {name: int(getattr(st, name)) for name, _ in pa_bm_stats._fields_}


def pa_copy_blocks(k_pool: torch.Tensor, v_pool: torch.Tensor, pairs: torch.Tensor, stream=None) -> None:
    """Copy whole blocks for copy-on-write; pairs: int32 CUDA [n][2] (src, dst)."""
    desc = _pools(k_pool, v_pool)
    _cuda_contig("pairs", pairs)
    _need(pairs.dtype == torch.int32 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs must be int32 [n][2]")
    _check(load_library().pa_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(pairs), int(pairs.shape[0]),
                                         ctypes.byref(desc), _stream(stream)))



def pa_copy_blocks_int8(k_codes: torch.Tensor, v_codes: torch.Tensor, k_scales: torch.Tensor,
                        v_scales: torch.Tensor, pairs: torch.Tensor, stream=None) -> None:
    """Copy-on-write over an INT8 cache: code blocks and their scale rows;
    pairs: int32 CUDA [n][2] (src, dst)."""
    desc = _pools(k_codes, v_codes)
    for n, t in (("k_scales", k_scales), ("v_scales", v_scales), ("pairs", pairs)):
        _cuda_contig(n, t)
    _need(k_scales.dtype == v_scales.dtype == torch.float32 and k_scales.shape == v_scales.shape ==
          k_codes.shape[:3], "scales must be float32 [num_blocks][H_kv][16]")
    _need(pairs.dtype == torch.int32 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs must be int32 [n][2]")
    _check(load_library().pa_copy_blocks_int8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales),
                                              _ptr(pairs), int(pairs.shape[0]), ctypes.byref(desc),
                                              _stream(stream)))