"""Run the fp64 oracle over many host cores.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by the tests and
the benchmark's CPU-baseline legs, never by the library.

Nothing here computes attention.  The work is cut into independent tasks --
one sequence, or one sequence and a subset of its query heads -- and each
task calls the unchanged ``oracle`` function (decode, prefill or their INT8
forms) on a slice of
the inputs; the tasks run on a thread pool (ctypes releases the interpreter
lock for the duration of each C call, so the threads run on separate cores).
Outputs are placed back where the single-threaded call would have put them,
so the result is the same array, bit for bit: every output row is computed by
the same C code on the same inputs.

The number of threads defaults to the host's cores, lowered when the
per-task gather buffers (the oracle widens each sequence's K and V to fp64)
would not fit in the available memory.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle


def host_cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def _available_bytes() -> Optional[int]:
    try:
        import psutil
        return int(psutil.virtual_memory().available)
    except Exception:  # noqa: BLE001 - psutil missing or unreadable: no memory bound
        return None


def pick_workers(task_bytes: int, workers: Optional[int] = None) -> int:
    """Threads to use: the requested count (default: every core), at most as
    many tasks' gather buffers as fit in half of the available memory."""
    n = host_cores() if workers is None else max(1, int(workers))
    avail = _available_bytes()
    if avail is not None and task_bytes > 0:
        n = max(1, min(n, int(avail // 2 // task_bytes)))
    return n


def _gather_bytes(ctx: int, hkv: int, d: int) -> int:
    return max(ctx, 1) * hkv * d * 8 * 2  # K and V widened to fp64


def _run(tasks, fn, workers: int) -> None:
    oracle.lib()  # build / load once, before any thread calls into it
    if workers <= 1 or len(tasks) <= 1:
        for t in tasks:
            fn(t)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for f in [ex.submit(fn, t) for t in tasks]:
            f.result()


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables,
           context_lens, scale: float, workers: Optional[int] = None,
           seqs: Optional[Sequence[int]] = None) -> np.ndarray:
    """Full [B, Hq, D] output of ``oracle.decode`` (rows of sequences not in
    ``seqs`` are left zero when ``seqs`` is given), one task per sequence."""
    b, hq, d = q.shape
    hkv = int(k_cache.shape[2])
    bt = torch.as_tensor(block_tables, dtype=torch.int32).contiguous()
    cl = torch.as_tensor(context_lens, dtype=torch.int32).contiguous()
    k_cache, v_cache = k_cache.contiguous(), v_cache.contiguous()
    out = np.zeros((b, hq, d), dtype=np.float64)
    todo: List[int] = list(range(b)) if seqs is None else [int(s) for s in seqs]
    biggest = max([int(cl[s]) for s in todo] + [1])

    def one(s: int) -> None:
        out[s] = oracle.decode(q[s:s + 1], k_cache, v_cache, bt[s:s + 1], cl[s:s + 1], scale)[0]

    _run(todo, one, pick_workers(_gather_bytes(biggest, hkv, d), workers))
    return out


def _prefill_tasks(call, q: torch.Tensor, hkv: int, block_tables, cu_seqlens_q, context_lens,
                   workers: Optional[int], head_groups: Optional[int]) -> np.ndarray:
    """Runs ``call(q_rows, bt_row, local_cu, cl_row, rows)`` -- one oracle
    prefill over a single sequence -- for every (sequence, group of query
    heads) task and assembles the full [T, Hq, D] output."""
    t, hq, d = q.shape
    bt = torch.as_tensor(block_tables, dtype=torch.int32).contiguous()
    cu = torch.as_tensor(cu_seqlens_q, dtype=torch.int32).tolist()
    cl = torch.as_tensor(context_lens, dtype=torch.int32).contiguous()
    b = len(cu) - 1
    out = np.zeros((t, hq, d), dtype=np.float64)
    n_workers = pick_workers(_gather_bytes(max([int(x) for x in cl.tolist()] + [1]), hkv, d),
                             workers)
    if head_groups is None:
        head_groups = 1
        while head_groups < hq and b * head_groups < n_workers:
            head_groups *= 2
    head_groups = max(1, min(int(head_groups), hq))
    per = -(-hq // head_groups)
    tasks = [(s, h0) for s in range(b) for h0 in range(0, hq, per) if cu[s + 1] > cu[s]]

    def one(task) -> None:
        s, h0 = task
        t0, t1 = cu[s], cu[s + 1]
        heads = list(range(h0, min(h0 + per, hq)))
        rows = [(r, h) for r in range(t1 - t0) for h in heads]
        local_cu = torch.tensor([0, t1 - t0], dtype=torch.int32)
        res = call(q[t0:t1], bt[s:s + 1], local_cu, cl[s:s + 1], rows)
        out[t0:t1, h0:h0 + len(heads)] = res.reshape(t1 - t0, len(heads), d)

    _run(tasks, one, n_workers)
    return out


def prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables,
            cu_seqlens_q, context_lens, scale: float, workers: Optional[int] = None,
            head_groups: Optional[int] = None) -> np.ndarray:
    """Full [T, Hq, D] output of ``oracle.prefill``, one task per (sequence,
    group of query heads); ``head_groups`` defaults to enough groups to give
    every thread a task."""
    k_cache, v_cache = k_cache.contiguous(), v_cache.contiguous()

    def call(qs, bt, cu, cl, rows):
        return oracle.prefill(qs, k_cache, v_cache, bt, cu, cl, scale, rows=rows)

    return _prefill_tasks(call, q, int(k_cache.shape[2]), block_tables, cu_seqlens_q,
                          context_lens, workers, head_groups)


def prefill_int8(q: torch.Tensor, k_codes, v_codes, k_scales, v_scales, block_tables,
                 cu_seqlens_q, context_lens, scale: float, workers: Optional[int] = None,
                 head_groups: Optional[int] = None) -> np.ndarray:
    """Full [T, Hq, D] output of ``oracle.prefill_int8``, split as ``prefill``."""
    k_codes, v_codes = k_codes.contiguous(), v_codes.contiguous()
    k_scales, v_scales = k_scales.contiguous(), v_scales.contiguous()

    def call(qs, bt, cu, cl, rows):
        return oracle.prefill_int8(qs, k_codes, v_codes, k_scales, v_scales, bt, cu, cl, scale,
                                   rows=rows)

    return _prefill_tasks(call, q, int(k_codes.shape[1]), block_tables, cu_seqlens_q,
                          context_lens, workers, head_groups)


def decode_int8(q: torch.Tensor, k_codes, v_codes, k_scales, v_scales, block_tables,
                context_lens, scale: float, workers: Optional[int] = None) -> np.ndarray:
    """Full [B, Hq, D] output of ``oracle.decode_int8``, one task per sequence."""
    b, hq, d = q.shape
    hkv = int(k_codes.shape[1])  # codes [NB, Hkv, 256, D]
    bt = torch.as_tensor(block_tables, dtype=torch.int32).contiguous()
    cl = torch.as_tensor(context_lens, dtype=torch.int32).contiguous()
    out = np.zeros((b, hq, d), dtype=np.float64)
    biggest = max([int(x) for x in cl.tolist()] + [1])

    def one(s: int) -> None:
        out[s] = oracle.decode_int8(q[s:s + 1], k_codes, v_codes, k_scales, v_scales,
                                    bt[s:s + 1], cl[s:s + 1], scale)[0]

    _run(list(range(b)), one, pick_workers(_gather_bytes(biggest, hkv, d), workers))
    return out
