"""GPU-side helpers for the parity tests: run the C-ABI path on a workload and
produce the oracle's answer on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_decode_27_gb300 import binding as pa
from paged_kv_decode_27_gb300 import workloads as W
from _util import to_np

DEV = "cuda"


def run_append(wl: W.Workload, st: W.StepInputs, kp: torch.Tensor, vp: torch.Tensor):
    pa.pa_append_kv(kp, vp, st.slot_mapping.to(DEV), st.k_new.to(DEV), st.v_new.to(DEV))


def oracle_append(wl: W.Workload, st: W.StepInputs, k_np=None, v_np=None):
    k_np = to_np(wl.k_pool) if k_np is None else k_np
    v_np = to_np(wl.v_pool) if v_np is None else v_np
    return oracle.append_ref(k_np, v_np, st.slot_mapping.numpy(), to_np(st.k_new), to_np(st.v_new))


def run_decode(wl: W.Workload, st: W.StepInputs, kp, vp, partition_size: int = 0, max_ctx=None):
    bt = wl.decode_block_tables.contiguous()
    out = torch.empty(st.q.shape, dtype=st.q.dtype, device=DEV)
    mc = int(st.context_lens.max()) if max_ctx is None else max_ctx
    pa.pa_decode_attention(out, st.q.to(DEV), kp, vp, bt.to(DEV), st.context_lens.to(DEV), wl.scale,
                           max_context_len=mc, partition_size=partition_size)
    torch.cuda.synchronize()
    return out


def oracle_decode(wl: W.Workload, st: W.StepInputs, k_np, v_np, seqs=None):
    bt = wl.decode_block_tables.contiguous().numpy()
    return oracle.decode_ref(to_np(st.q), k_np, v_np, bt, st.context_lens.numpy(), wl.scale, seqs=seqs)


def device_status_clean():
    return pa.pa_device_status() == 0


def fill_unused_with_nan(wl: W.Workload, ctx: torch.Tensor, rows=None):
    """Overwrite every pool slot that no sequence's context covers with NaN,
    so any read past a context shows up in the output."""
    bt = wl.block_tables if rows is None else wl.block_tables[rows]
    used = set()
    for s in range(bt.shape[0]):
        c = int(ctx[s])
        for p in range(c):
            used.add(int(bt[s, p // 16]) * 16 + p % 16)
    n = wl.num_blocks * 16
    mask = torch.ones(n, dtype=torch.bool)
    if used:
        mask[torch.tensor(sorted(used))] = False
    for pool in (wl.k_pool, wl.v_pool):
        flat = pool.permute(0, 2, 1, 3).reshape(n, pool.shape[1], pool.shape[3])
        flat[mask] = float("nan")
        pool.copy_(flat.reshape(pool.shape[0], 16, pool.shape[1], pool.shape[3]).permute(0, 2, 1, 3))
