"""Seeded synthetic workloads for paged decode attention.

This module only *builds inputs*: the KV block pool, block tables, context
lengths, slot mappings and the per-step q / new-K / new-V tensors.  It holds
none of the attention arithmetic and imports neither the CUDA library nor the
test oracle, so the tests, the benchmark and the oracle can all draw the same
inputs from it.

The shapes follow the model families named on the pages ("LLM Inference Server
From Scratch", *What you build*: Llama 2/3 or Mistral weights in fp16/bf16;
"Mini inference engine", step 1: Llama-3.2-1B) with their head geometry, the
16-token paged blocks of "Mini inference engine" (step 2, stretch) and
"LLM Inference Server" (*Paged KV-Cache Block Allocator*), and the prefill /
decode split of "LLM Inference Server", Stage 1.

Conventions (the plain reading where the pages leave a step open):
  * pool layout ``[num_blocks][H_kv][16][D]`` for both K and V;
  * ``slot = block_id * 16 + offset`` (int64), a negative slot means "skip";
  * ``context_lens`` are the lengths *after* the step's append, so the new
    token of a decode step sits at position ``context_len - 1``;
  * unused block-table entries are padded with 0 (a valid id, never read);
  * everything is drawn on the CPU with ``torch.Generator`` seeded
    ``1000 + config_id``; step ``t`` draws its q / k_new / v_new from a
    generator seeded ``(1000 + config_id) * 100 + t``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

BLOCK_SIZE = 16


def _dtype(name: str) -> torch.dtype:
    return {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[name]


@dataclass
class StepInputs:
    """What one decode (or mixed) step feeds the hot path."""

    slot_mapping: torch.Tensor      # int64 [T]
    k_new: torch.Tensor             # [T][H_kv][D]
    v_new: torch.Tensor             # [T][H_kv][D]
    q: torch.Tensor                 # decode queries [S_dec][H_q][D]
    context_lens: torch.Tensor      # int32 [S_dec], after the append
    # mixed continuous-batching step only (causal prompt pass):
    q_prefill: Optional[torch.Tensor] = None      # [sum q_len][H_q][D]
    cu_q_lens: Optional[torch.Tensor] = None      # int32 [S_pre + 1]
    prefill_context_lens: Optional[torch.Tensor] = None  # int32 [S_pre]


@dataclass
class Workload:
    name: str
    config_id: int
    dtype: torch.dtype
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    steps: int
    k_pool: torch.Tensor            # [N_blk][H_kv][16][D]
    v_pool: torch.Tensor
    block_tables: torch.Tensor      # int32 [S_all][max_blocks]
    ctx0: torch.Tensor              # int32 [S_dec]: decode context lens at step 0
    decode_rows: slice              # rows of block_tables used by decode
    prefill_rows: Optional[slice] = None
    prompt_lens: Optional[List[int]] = None
    factor: float = 1.0
    description: str = ""
    extra: dict = field(default_factory=dict)
    # INT8 cache only: k_pool / v_pool then hold int8 codes and these the
    # float32 scale of every (block, head, slot) row
    k_scales: Optional[torch.Tensor] = None   # float32 [N_blk][H_kv][16]
    v_scales: Optional[torch.Tensor] = None

    # ---- derived geometry -------------------------------------------------
    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def elem_bytes(self) -> int:
        """Bytes of one q / out / new K/V element (the activation dtype)."""
        return torch.tensor([], dtype=self.dtype).element_size()

    @property
    def kv_int8(self) -> bool:
        return self.k_pool.dtype == torch.int8

    @property
    def kv_row_bytes(self) -> int:
        """Pool bytes of one (token, KV head) row: D elements, plus the float32
        scale of an INT8 cache."""
        if self.kv_int8:
            return self.head_dim + 4
        return self.head_dim * self.elem_bytes

    @property
    def decode_block_tables(self) -> torch.Tensor:
        return self.block_tables[self.decode_rows]

    @property
    def prefill_block_tables(self) -> Optional[torch.Tensor]:
        if self.prefill_rows is None:
            return None
        return self.block_tables[self.prefill_rows]

    @property
    def num_decode_seqs(self) -> int:
        return int(self.ctx0.numel())

    def context_lens(self, t: int) -> torch.Tensor:
        return (self.ctx0 + t).to(torch.int32)

    def max_context_len(self, t: int = 0) -> int:
        return int(self.ctx0.max().item()) + t if self.ctx0.numel() else 0

    # ---- per-step draws ---------------------------------------------------
    def step(self, t: int) -> StepInputs:
        """Inputs of step ``t`` (0-based); deterministic in (config, t)."""
        if not 0 <= t < self.steps:
            raise ValueError(f"step {t} outside [0, {self.steps})")
        g = torch.Generator().manual_seed((1000 + self.config_id) * 100 + t)
        hq, hkv, d = self.num_q_heads, self.num_kv_heads, self.head_dim
        ctx = self.context_lens(t)
        bt = self.decode_block_tables
        s_dec = ctx.numel()
        # decode: the new token of sequence s sits at position ctx[s] - 1
        pos = (ctx.to(torch.int64) - 1)
        dec_slots = bt[torch.arange(s_dec), (pos.clamp(min=0) // BLOCK_SIZE)].to(torch.int64) \
            * BLOCK_SIZE + pos.clamp(min=0) % BLOCK_SIZE
        # an empty context appends nothing
        dec_slots = torch.where(ctx > 0, dec_slots, torch.full_like(dec_slots, -1))
        slots = [dec_slots]
        q_pre = cu = pre_ctx = None
        n_pre_tok = 0
        if self.prompt_lens:
            pbt = self.prefill_block_tables
            pre_slots = []
            for i, L in enumerate(self.prompt_lens):
                p = torch.arange(L, dtype=torch.int64)
                pre_slots.append(pbt[i, p // BLOCK_SIZE].to(torch.int64) * BLOCK_SIZE + p % BLOCK_SIZE)
            n_pre_tok = sum(self.prompt_lens)
            # prompt tokens first, then the decode tokens
            slots = pre_slots + slots
            cu = torch.tensor([0] + list(_cumsum(self.prompt_lens)), dtype=torch.int32)
            pre_ctx = torch.tensor(self.prompt_lens, dtype=torch.int32)
        slot_mapping = torch.cat(slots).contiguous()
        T = slot_mapping.numel()
        k_new = self._draw((T, hkv, d), g)
        v_new = self._draw((T, hkv, d), g)
        q = self._draw((s_dec, hq, d), g)
        if self.prompt_lens:
            q_pre = self._draw((n_pre_tok, hq, d), g)
        return StepInputs(slot_mapping=slot_mapping, k_new=k_new, v_new=v_new, q=q,
                          context_lens=ctx, q_prefill=q_pre, cu_q_lens=cu,
                          prefill_context_lens=pre_ctx)

    def verify_queries(self, t: int, q_len: int) -> torch.Tensor:
        """Queries of a speculative-decoding verification pass at step t:
        [S_dec][q_len][H_q][D], the last q_len cached positions of every
        sequence (seeded separately from the step's other draws)."""
        g = torch.Generator().manual_seed(((1000 + self.config_id) * 100 + t) * 16 + q_len)
        return self._draw((self.num_decode_seqs, q_len, self.num_q_heads, self.head_dim), g)

    def verify_bytes(self, t: int, q_len: int) -> int:
        """decode_bytes with q_len query rows (q and out) per sequence."""
        extra = 2 * (q_len - 1) * self.num_decode_seqs * self.num_q_heads * self.head_dim * self.elem_bytes
        return self.decode_bytes(t) + extra

    def _draw(self, shape, g) -> torch.Tensor:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if self.factor != 1.0:
            x.mul_(self.factor)
        return x.to(self.dtype).contiguous()

    # ---- byte accounting (algorithmic, for throughput reporting) ----------
    def decode_bytes(self, t: int = 0) -> int:
        """Bytes one decode-attention call must move at minimum: the valid K/V
        tokens, q and out, the block ids read and the context lengths."""
        ctx = self.context_lens(t).to(torch.int64)
        e = self.elem_bytes
        kv = int(ctx.sum()) * 2 * self.num_kv_heads * self.kv_row_bytes
        qo = 2 * self.num_decode_seqs * self.num_q_heads * self.head_dim * e
        ids = 4 * int(((ctx + BLOCK_SIZE - 1) // BLOCK_SIZE).sum()) + 4 * self.num_decode_seqs
        return kv + qo + ids

    def append_bytes(self, t: int = 0) -> int:
        """Read new K/V + slots, write the same K/V into the pool."""
        st_tokens = self.num_decode_seqs + (sum(self.prompt_lens) if self.prompt_lens else 0)
        row_in = self.num_kv_heads * self.head_dim * self.elem_bytes
        row_out = self.num_kv_heads * self.kv_row_bytes
        return 2 * st_tokens * (row_in + row_out) + 8 * st_tokens

    def prefill_flops(self) -> int:
        """4*D flops per (query, key, q-head) pair under the causal mask."""
        if not self.prompt_lens:
            return 0
        pairs = sum(L * (L + 1) // 2 for L in self.prompt_lens)
        return 4 * self.head_dim * self.num_q_heads * pairs


def _cumsum(xs):
    acc = 0
    for x in xs:
        acc += x
        yield acc


def _assign_blocks(need: List[int], pool_blocks: int, g: torch.Generator,
                   shared_prefix_blocks: int = 0) -> torch.Tensor:
    """Block tables drawn from a random permutation of the whole pool.

    Sequence s takes the next ``need[s]`` ids of the permutation; when
    ``shared_prefix_blocks`` > 0 the first ids are taken once and reused as
    the leading entries of every table (a shared system prompt)."""
    perm = torch.randperm(pool_blocks, generator=g).to(torch.int32)
    max_blocks = max(need) if need else 1
    bt = torch.zeros((len(need), max_blocks), dtype=torch.int32)
    cursor = 0
    shared = perm[:shared_prefix_blocks]
    cursor += shared_prefix_blocks
    for s, n in enumerate(need):
        bt[s, :shared_prefix_blocks] = shared
        priv = n - shared_prefix_blocks
        bt[s, shared_prefix_blocks:n] = perm[cursor:cursor + priv]
        cursor += priv
    if cursor > pool_blocks:
        raise ValueError("pool too small for the requested block tables")
    return bt


def _blocks_for(tokens: int) -> int:
    return (tokens + BLOCK_SIZE - 1) // BLOCK_SIZE


def _pool(n_blk, hkv, d, dtype, factor, g) -> torch.Tensor:
    x = torch.randn((n_blk, hkv, BLOCK_SIZE, d), generator=g, dtype=torch.float32)
    if factor != 1.0:
        x.mul_(factor)
    return x.to(dtype).contiguous()


def _pool_int8(n_blk, hkv, d, factor, g):
    """An INT8 cache drawn directly: codes uniform in [-127, 127], one float32
    scale per (block, head, slot) uniform in [2, 4] * factor / 127 (the range
    of max|x| / 127 for D values of N(0, factor^2))."""
    codes = torch.randint(-127, 128, (n_blk, hkv, BLOCK_SIZE, d), generator=g, dtype=torch.int16)
    scales = (torch.rand((n_blk, hkv, BLOCK_SIZE), generator=g) * 2.0 + 2.0) * (factor / 127.0)
    return codes.to(torch.int8).contiguous(), scales.to(torch.float32).contiguous()


def _kv_pools(n_blk, hkv, d, dtype, factor, g, kv: str):
    """(k_pool, v_pool, k_scales, v_scales) of a float or an INT8 cache."""
    if kv == "int8":
        kc, ks = _pool_int8(n_blk, hkv, d, factor, g)
        vc, vs = _pool_int8(n_blk, hkv, d, factor, g)
        return kc, vc, ks, vs
    return _pool(n_blk, hkv, d, dtype, factor, g), _pool(n_blk, hkv, d, dtype, factor, g), None, None


# --------------------------------------------------------------------------
# The five workloads.  Names say what each is; ids only pick the seed.
# --------------------------------------------------------------------------

def tiny_fp32() -> Workload:
    """2 sequences (contexts 17 and 40 after the append), h_q=4, h_kv=2, D=64,
    fp32, a 16-block pool handed out by a seeded permutation, scale 1/8."""
    cid = 1
    g = torch.Generator().manual_seed(1000 + cid)
    ctx = [17, 40]
    need = [_blocks_for(c) for c in ctx]
    bt = _assign_blocks(need, 16, g)
    k_pool = _pool(16, 2, 64, torch.float32, 1.0, g)
    v_pool = _pool(16, 2, 64, torch.float32, 1.0, g)
    return Workload(name="tiny_fp32", config_id=cid, dtype=torch.float32, num_q_heads=4,
                    num_kv_heads=2, head_dim=64, scale=1.0 / 8.0, steps=1,
                    k_pool=k_pool, v_pool=v_pool, block_tables=bt,
                    ctx0=torch.tensor(ctx, dtype=torch.int32), decode_rows=slice(0, 2),
                    description="tiny paged decode, fp32")


def _multi_step(cid: int, name: str, S: int, hq: int, hkv: int, d: int, steps: int,
                ctx0: torch.Tensor, factor: float, dtype=torch.bfloat16,
                description: str = "", kv: str = "float") -> Workload:
    g = torch.Generator().manual_seed(1000 + cid)
    g_ctx_consumed = ctx0  # drawn by the caller from the same generator
    need = [_blocks_for(int(c) + steps - 1) for c in g_ctx_consumed]
    pool_blocks = int(math.ceil(1.25 * sum(need)))
    bt = _assign_blocks(need, pool_blocks, g)
    k_pool, v_pool, k_scales, v_scales = _kv_pools(pool_blocks, hkv, d, dtype, factor, g, kv)
    return Workload(name=name, config_id=cid, dtype=dtype, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=d, scale=1.0 / math.sqrt(d), steps=steps, k_pool=k_pool,
                    v_pool=v_pool, block_tables=bt, ctx0=ctx0.to(torch.int32),
                    decode_rows=slice(0, S), factor=factor, description=description,
                    k_scales=k_scales, v_scales=v_scales)


def llama32_1b_decode(steps: int = 16, kv: str = "float") -> Workload:
    """Llama-3.2-1B-shaped decode, bf16: batch 8, h_q=32, h_kv=8, D=64,
    contexts uniform in [128, 2048], pool 1.25x the need, values N(0,1)*0.5.
    ``kv="int8"``: the same batch over an INT8 cache."""
    cid = 2
    gc = torch.Generator().manual_seed(1000 + cid + 500)
    ctx0 = torch.randint(128, 2048 + 1, (8,), generator=gc)
    name = "llama32_1b_decode" + ("_int8" if kv == "int8" else "")
    return _multi_step(cid, name, 8, 32, 8, 64, steps, ctx0, 0.5, kv=kv,
                       description="Llama-3.2-1B-shaped decode, bf16, batch 8" +
                       (", INT8 KV cache" if kv == "int8" else ""))


def llama3_8b_decode(steps: int = 32, batch: int = 64, kv: str = "float") -> Workload:
    """Llama-3-8B-shaped decode, bf16: batch 64, h_q=32, h_kv=8, D=128,
    contexts log-uniform in [512, 8192], randomly permuted pool (1.25x).
    ``kv="int8"``: the same batch (contexts, tables, per-step q and new K/V)
    over an INT8 cache."""
    cid = 3
    gc = torch.Generator().manual_seed(1000 + cid + 500)
    u = torch.rand((batch,), generator=gc, dtype=torch.float64)
    ctx0 = torch.floor(torch.exp(math.log(512) + u * (math.log(8192) - math.log(512))))
    ctx0 = ctx0.clamp(512, 8192).to(torch.int64)
    name = "llama3_8b_decode" + ("_int8" if kv == "int8" else "")
    return _multi_step(cid, name, batch, 32, 8, 128, steps, ctx0, 1.0, kv=kv,
                       description="Llama-3-8B-shaped decode, bf16, batch %d" % batch +
                       (", INT8 KV cache" if kv == "int8" else ""))


def llama3_8b_long(batch: int, steps: int = 32) -> Workload:
    """The Llama-3-8B head shape (h_q=32, h_kv=8, D=128, bf16) at the
    small-batch end of the decode range: ``batch`` sequences (1 or 4 in the
    tests and the benchmark) whose contexts reach 8192 on the last step
    (8192 - steps + 1 at step 0), blocks randomly permuted in a pool of 1.25x
    the need, values N(0, 1).  The batch is the speculative-decoding setting
    of "Mini inference engine", section 7 (batch 1)."""
    cid = 30 + batch
    ctx0 = torch.full((batch,), 8192 - steps + 1, dtype=torch.int64)
    return _multi_step(cid, "llama3_8b_long_b%d" % batch, batch, 32, 8, 128, steps, ctx0, 1.0,
                       description="Llama-3-8B-shaped long-context decode, bf16, batch %d, "
                                   "contexts up to 8192" % batch)


def prefix_shared_8k() -> Workload:
    """8 sequences of context 8192 whose first 13 blocks (208 tokens, a shared
    system prompt) are the same physical blocks; h_q=32, h_kv=8, D=128, bf16."""
    cid = 4
    g = torch.Generator().manual_seed(1000 + cid)
    S, ctx, shared = 8, 8192, 13
    need = [_blocks_for(ctx)] * S
    used = shared + S * (need[0] - shared)
    pool_blocks = int(math.ceil(1.25 * used))
    bt = _assign_blocks(need, pool_blocks, g, shared_prefix_blocks=shared)
    k_pool = _pool(pool_blocks, 8, 128, torch.bfloat16, 1.0, g)
    v_pool = _pool(pool_blocks, 8, 128, torch.bfloat16, 1.0, g)
    return Workload(name="prefix_shared_8k", config_id=cid, dtype=torch.bfloat16,
                    num_q_heads=32, num_kv_heads=8, head_dim=128, scale=1.0 / math.sqrt(128),
                    steps=1, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
                    ctx0=torch.full((S,), ctx, dtype=torch.int32), decode_rows=slice(0, S),
                    description="long-context prefix-shared decode, bf16",
                    extra={"shared_prefix_blocks": shared, "blocks_used": used})


def mixed_mistral7b(kv: str = "float") -> Workload:
    """One continuous-batching step, Mistral-7B-shaped (h_q=32, h_kv=8, D=128,
    bf16): 4 causal prompts of 512/1024/1536/2048 tokens written into the pool
    and 60 decode sequences with contexts uniform in [256, 4096].
    ``kv="int8"``: the same step over an INT8 cache."""
    cid = 5
    g = torch.Generator().manual_seed(1000 + cid)
    prompts = [512, 1024, 1536, 2048]
    ctx0 = torch.randint(256, 4096 + 1, (60,), generator=g)
    need = [_blocks_for(L) for L in prompts] + [_blocks_for(int(c)) for c in ctx0]
    pool_blocks = int(math.ceil(1.25 * sum(need)))
    bt = _assign_blocks(need, pool_blocks, g)
    k_pool, v_pool, k_scales, v_scales = _kv_pools(pool_blocks, 8, 128, torch.bfloat16, 1.0, g, kv)
    return Workload(name="mixed_mistral7b" + ("_int8" if kv == "int8" else ""), config_id=cid,
                    dtype=torch.bfloat16, num_q_heads=32, num_kv_heads=8, head_dim=128, scale=1.0 / math.sqrt(128),
                    steps=1, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
                    ctx0=ctx0.to(torch.int32), decode_rows=slice(4, 64),
                    prefill_rows=slice(0, 4), prompt_lens=prompts,
                    k_scales=k_scales, v_scales=v_scales,
                    description="mixed continuous-batching step (Mistral-7B-shaped), bf16" +
                                (", INT8 KV cache" if kv == "int8" else ""))


WORKLOADS = {
    "tiny_fp32": tiny_fp32,
    "llama32_1b_decode": llama32_1b_decode,
    "llama3_8b_decode": llama3_8b_decode,
    "prefix_shared_8k": prefix_shared_8k,
    "mixed_mistral7b": mixed_mistral7b,
    "mixed_mistral7b_int8": lambda: mixed_mistral7b(kv="int8"),
    "llama32_1b_decode_int8": lambda: llama32_1b_decode(kv="int8"),
    "llama3_8b_decode_int8": lambda: llama3_8b_decode(kv="int8"),
    "llama3_8b_verify": lambda: llama3_8b_verify(),
    "llama3_8b_verify_int8": lambda: llama3_8b_verify(kv="int8"),
    "llama3_8b_decode_rope": lambda: llama3_8b_decode_rope(),
    "llama3_8b_long_b1": lambda: llama3_8b_long(1),
    "llama3_8b_long_b4": lambda: llama3_8b_long(4),
}


def llama3_8b_decode_rope(steps: int = 32) -> Workload:
    """The batch-64 Llama-3-8B-shaped decode with rotary position embedding
    (theta 500000, Llama 3's base) applied to K on the append and to q before
    attention."""
    wl = llama3_8b_decode(steps=steps)
    wl.name = "llama3_8b_decode_rope"
    wl.description = "Llama-3-8B-shaped decode with RoPE (theta 5e5) fused into the append, bf16, batch 64"
    wl.extra["rope_theta"] = 500000.0
    return wl


def llama3_8b_verify(steps: int = 32, q_len: int = 5, kv: str = "float") -> Workload:
    """The batch-64 Llama-3-8B-shaped decode batch in a speculative-decoding
    verification pass: each sequence's last q_len = K + 1 = 5 positions (K = 4
    drafted tokens) are queries, causal over the cache.  ``kv="int8"``: the
    same batch over an INT8 cache."""
    wl = llama3_8b_decode(steps=steps, kv=kv)
    wl.name = "llama3_8b_verify" + ("_int8" if kv == "int8" else "")
    wl.description = ("Llama-3-8B-shaped verification of K=4 drafts (q_len 5), bf16, batch 64" +
                      (", INT8 KV cache" if kv == "int8" else ""))
    wl.extra["verify_q_len"] = q_len
    return wl


def small_random(seed: int, num_seqs: int, max_ctx: int, hq: int, hkv: int, d: int,
                 dtype: torch.dtype = torch.bfloat16, extra_blocks: int = 3,
                 ctx: Optional[List[int]] = None, kv: str = "float") -> Workload:
    """A small ad-hoc workload for edge-case tests (ragged contexts, small
    pools).  One step; contexts uniform in [1, max_ctx] unless given.
    ``kv="int8"`` draws an INT8 cache (q and new K/V stay ``dtype``)."""
    g = torch.Generator().manual_seed(seed)
    if ctx is None:
        ctx_t = torch.randint(1, max_ctx + 1, (num_seqs,), generator=g)
    else:
        ctx_t = torch.tensor(ctx, dtype=torch.int64)
    need = [max(1, _blocks_for(int(c))) for c in ctx_t]
    pool_blocks = sum(need) + extra_blocks
    bt = _assign_blocks(need, pool_blocks, g)
    k_pool, v_pool, k_scales, v_scales = _kv_pools(pool_blocks, hkv, d, dtype, 1.0, g, kv)
    return Workload(name="small_random_%d" % seed, config_id=10_000 + seed, dtype=dtype,
                    num_q_heads=hq, num_kv_heads=hkv, head_dim=d, scale=1.0 / math.sqrt(d),
                    steps=1, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
                    ctx0=ctx_t.to(torch.int32), decode_rows=slice(0, len(need)),
                    k_scales=k_scales, v_scales=v_scales)
