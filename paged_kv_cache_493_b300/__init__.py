"""Python binding of libpkv: attention over a paged KV cache on B300.

The functions below carry the names of the C entry points declared in
``include/pkv.h`` and only marshal arguments: every step of the computation
runs in the library's CUDA kernels.  Tensors are torch CUDA tensors (torch
supplies device memory and streams); there is no CPU fallback, and a missing
or unloadable library raises ``PkvError``.

Layouts (see pkv.h): k_cache / v_cache bf16 [num_blocks, 256, Hkv, D];
block_tables int32 [B, max_blocks]; context_lens int32 [B]; decode q bf16
[B, Hq, D] (row stride free); prefill q bf16 [T, Hq, D] with cu_seqlens_q
int32 [B + 1]; store k / v bf16 [N, Hkv, D] with slot_mapping int32 [N].
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

BLOCK_SIZE = 256

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libpkv.so")

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
          4: "PKV_ERR_DEVICE_CHECK", 5: "PKV_ERR_TIMEOUT", 6: "PKV_ERR_NO_MEMORY"}
PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA = 0, 1, 2, 3
PKV_ERR_DEVICE_CHECK, PKV_ERR_TIMEOUT, PKV_ERR_NO_MEMORY = 4, 5, 6

# Every function the header declares, with its ctypes signature.
_P, _I32, _I64, _F, _D = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                          ctypes.c_double)
SIGNATURES = {
    "pkv_store_kvcache": ([_P, _P, _I64, _I64, _P, _I64, _P, _P, _I64, _I32, _I32, _P], _I32),
    "pkv_decode_attention": ([_P, _I64, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32, _F,
                              _P, _P], _I32),
    "pkv_prefill_attention": ([_P, _I64, _P, _P, _I64, _P, _I32, _P, _P, _I32, _I64, _I32, _I32,
                               _I32, _F, _P, _P], _I32),
    "pkv_decode_attention_noalloc": ([_P, _I64, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32,
                                      _I32, _F, _P, _P], _I32),
    "pkv_status_string": ([_I32], ctypes.c_char_p),
    "pkv_version": ([], ctypes.c_char_p),
    "pkv_get_device_error": ([_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)], _I32),
    "pkv_set_max_splits": ([_I32], _I32),
    "pkv_reserve_workspace": ([_I32, _I32, _I32, _I32], _I32),
    "pkv_set_wait_limit_ns": ([_I64], _I32),
    "pkv_profiler_enable": ([_I32], _I32),
    "pkv_profiler_reset": ([], _I32),
    "pkv_profiler_read": ([ctypes.c_char_p, ctypes.POINTER(_D), ctypes.POINTER(_I64)], _I32),
}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


_lib: Optional[ctypes.CDLL] = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpkv.so (built by ``_build.py``); raises PkvError if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise PkvError(PKV_ERR_CUDA, f"libpkv.so not built ({p}); run python -m "
                                     "paged_kv_cache_493_b300._build")
    lib = ctypes.CDLL(p)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise PkvError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise PkvError(PKV_ERR_INVALID_ARG, msg)


def _rows(t, name: str, heads: int, d: int) -> int:
    """Row stride (elements) of a [N, heads, d] bf16 view with contiguous rows."""
    import torch
    _need(t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 3, f"{name}: bf16 CUDA [N, H, D]")
    _need(t.shape[1] == heads and t.shape[2] == d, f"{name}: shape {tuple(t.shape)}")
    _need(t.stride(2) == 1 and t.stride(1) == d, f"{name}: heads and dims must be contiguous")
    return int(t.stride(0)) if t.shape[0] > 1 else heads * d


def _i32(t, name: str) -> None:
    import torch
    _need(t.is_cuda and t.dtype == torch.int32 and t.is_contiguous(), f"{name}: contiguous int32 CUDA")


def _cache(k_cache, v_cache):
    import torch
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t.is_cuda and t.dtype == torch.bfloat16 and t.dim() == 4 and t.is_contiguous()
              and t.shape[1] == BLOCK_SIZE, f"{n}: contiguous bf16 CUDA [NB, 256, Hkv, D]")
    _need(k_cache.shape == v_cache.shape, "k_cache and v_cache shapes differ")
    nb, _, hkv, d = k_cache.shape
    return int(nb), int(hkv), int(d)


def pkv_store_kvcache(k, v, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """Scatter rows of k / v [N, Hkv, D] into cache slots (slot -1 skips a row)."""
    nb, hkv, d = _cache(k_cache, v_cache)
    n = int(slot_mapping.numel())
    _i32(slot_mapping, "slot_mapping")
    ks = _rows(k, "k", hkv, d)
    vs = _rows(v, "v", hkv, d)
    _need(k.shape[0] == n and v.shape[0] == n, "k, v and slot_mapping disagree on N")
    _check(load_library().pkv_store_kvcache(_ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), n,
                                            _ptr(k_cache), _ptr(v_cache), nb, hkv, d,
                                            _stream(stream)), "pkv_store_kvcache")


def pkv_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float, out,
                         stream=None) -> None:
    """One query per sequence: q [B, Hq, D] -> out [B, Hq, D] (contiguous)."""
    nb, hkv, d = _cache(k_cache, v_cache)
    _need(q.dim() == 3, "q: [B, Hq, D]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    _i32(block_tables, "block_tables")
    _i32(context_lens, "context_lens")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b, "block_tables: [B, max_blocks]")
    _need(context_lens.numel() == b, "context_lens: [B]")
    _need(out.is_contiguous() and out.shape == q.shape and out.dtype == q.dtype and out.is_cuda,
          "out: contiguous, same shape/dtype as q")
    _check(load_library().pkv_decode_attention(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(context_lens), b, hq, hkv, d, float(scale), _ptr(out), _stream(stream)),
        "pkv_decode_attention")


def pkv_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                 out, stream=None) -> None:
    """pkv_decode_attention with its split-K scratch in the library's static
    16 MiB device array: the call allocates no device memory, for callers that
    cannot allocate (a KV pool that already holds the free memory, stream
    capture).  Raises PkvError(PKV_ERR_UNSUPPORTED) for a batch whose partials
    do not fit; overlapping calls on one device race on the shared array."""
    nb, hkv, d = _cache(k_cache, v_cache)
    _need(q.dim() == 3, "q: [B, Hq, D]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    _i32(block_tables, "block_tables")
    _i32(context_lens, "context_lens")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b, "block_tables: [B, max_blocks]")
    _need(context_lens.numel() == b, "context_lens: [B]")
    _need(out.is_contiguous() and out.shape == q.shape and out.dtype == q.dtype and out.is_cuda,
          "out: contiguous, same shape/dtype as q")
    _check(load_library().pkv_decode_attention_noalloc(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(context_lens), b, hq, hkv, d, float(scale), _ptr(out), _stream(stream)),
        "pkv_decode_attention_noalloc")


def pkv_prefill_attention(q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens,
                          scale: float, out, stream=None) -> None:
    """Chunked causal prefill: q [T, Hq, D] -> out [T, Hq, D] (contiguous)."""
    nb, hkv, d = _cache(k_cache, v_cache)
    _need(q.dim() == 3, "q: [T, Hq, D]")
    t, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    for x, n in ((block_tables, "block_tables"), (cu_seqlens_q, "cu_seqlens_q"),
                 (context_lens, "context_lens")):
        _i32(x, n)
    b = int(context_lens.numel())
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b, "block_tables: [B, max_blocks]")
    _need(cu_seqlens_q.numel() == b + 1, "cu_seqlens_q: [B + 1]")
    _need(out.is_contiguous() and out.shape == q.shape and out.dtype == q.dtype and out.is_cuda,
          "out: contiguous, same shape/dtype as q")
    _check(load_library().pkv_prefill_attention(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(cu_seqlens_q), _ptr(context_lens), b, t, hq, hkv, d, float(scale), _ptr(out),
        _stream(stream)), "pkv_prefill_attention")


def pkv_get_device_error(stream=None):
    """Synchronise the stream; return and clear (code, site) of the device error word."""
    code, info = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().pkv_get_device_error(_stream(stream), ctypes.byref(code),
                                               ctypes.byref(info)), "pkv_get_device_error")
    return int(code.value), int(info.value)


def pkv_set_max_splits(n: int) -> None:
    _check(load_library().pkv_set_max_splits(int(n)), "pkv_set_max_splits")


def pkv_reserve_workspace(num_seqs: int, num_q_heads: int, head_dim: int, max_blocks: int) -> None:
    _check(load_library().pkv_reserve_workspace(num_seqs, num_q_heads, head_dim, max_blocks),
           "pkv_reserve_workspace")


def pkv_set_wait_limit_ns(ns: int) -> None:
    _check(load_library().pkv_set_wait_limit_ns(int(ns)), "pkv_set_wait_limit_ns")


def pkv_version() -> str:
    return load_library().pkv_version().decode()


def pkv_status_string(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


def pkv_profiler_enable(on: bool) -> None:
    _check(load_library().pkv_profiler_enable(1 if on else 0), "pkv_profiler_enable")


def pkv_profiler_reset() -> None:
    _check(load_library().pkv_profiler_reset(), "pkv_profiler_reset")


def pkv_profiler_read(name: str):
    """(total milliseconds, launches) of kernel `name` since the last reset."""
    ms, n = ctypes.c_double(0), ctypes.c_int64(0)
    _check(load_library().pkv_profiler_read(name.encode(), ctypes.byref(ms), ctypes.byref(n)),
           "pkv_profiler_read")
    return float(ms.value), int(n.value)
