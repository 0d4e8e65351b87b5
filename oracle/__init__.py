"""Float64 CPU oracle for paged decode attention.

Test infrastructure: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use it.  The CUDA path never imports it.
Every function is pinned by the ``-m "not gpu"`` tests in ``tests/test_oracle.py``
``tests/test_oracle_int8.py``, ``tests/test_oracle_rope.py`` and
``tests/test_oracle_block_manager.py``.
"""
from .paged_attention import (  # noqa: F401
    BLOCK_SIZE,
    append_ref,
    as_f64,
    attend,
    bf16_bits_to_f64,
    decode_ref,
    gather_contiguous,
    kv_cache_bytes,
    prefill_ref,
)
from .kv_int8 import (  # noqa: F401,E402
    append_int8_ref,
    decode_int8_ref,
    dequantize_rows_int8,
    gather_dequantized,
    prefill_int8_ref,
    quantize_rows_int8,
    verify_int8_ref,
)
from .rope import append_rope_ref, rope_cache_ref, rope_inv_freq, rope_rotate_ref  # noqa: F401,E402
from .block_manager import BlockManagerRef, NoBlocks, block_key, fnv1a64  # noqa: F401,E402
