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
    "pkv_decode_attention_shared_prefix": ([_P, _I64, _P, _P, _I64, _P, _I32, _P, _I32, _I32,
                                            _I32, _I32, _F, _I32, _P, _P], _I32),
    "pkv_set_shared_prefix_units": ([_I32], _I32),
    "pkv_decode_attention_append": ([_P, _I64, _P, _P, _I64, _I64, _P, _P, _P, _I64, _P, _I32, _P,
                                     _I32, _I32, _I32, _I32, _F, _P, _P], _I32),
    "pkv_store_kvcache_int8": ([_P, _P, _I64, _I64, _P, _I64, _P, _P, _P, _P, _I64, _I32, _I32,
                                _P], _I32),
    "pkv_decode_attention_int8": ([_P, _I64, _P, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32,
                                   _I32, _I32, _F, _P, _P], _I32),
    "pkv_prefill_attention_int8": ([_P, _I64, _P, _P, _P, _P, _I64, _P, _I32, _P, _P, _I32, _I64,
                                    _I32, _I32, _I32, _F, _P, _P], _I32),
    "pkv_status_string": ([_I32], ctypes.c_char_p),
    "pkv_version": ([], ctypes.c_char_p),
    "pkv_get_device_error": ([_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)], _I32),
    "pkv_set_max_splits": ([_I32], _I32),
    "pkv_reserve_workspace": ([_I32, _I32, _I32, _I32], _I32),
    "pkv_set_wait_limit_ns": ([_I64], _I32),
    "pkv_profiler_enable": ([_I32], _I32),
    "pkv_profiler_reset": ([], _I32),
    "pkv_profiler_read": ([ctypes.c_char_p, ctypes.POINTER(_D), ctypes.POINTER(_I64)], _I32),
    "pkv_bm_create": ([_I32, ctypes.POINTER(_P)], _I32),
    "pkv_bm_destroy": ([_P], None),
    "pkv_bm_num_free_blocks": ([_P], _I32),
    "pkv_bm_ref_count": ([_P, _I32], _I32),
    "pkv_bm_allocate": ([_P, _I64, _P, _I32, ctypes.POINTER(_I32)], _I32),
    "pkv_bm_append": ([_P, _I64, _P, _I32, _P], _I32),
    "pkv_bm_append_decode": ([_P, _P, _I32, _P, _P], _I32),
    "pkv_bm_decode_step": ([_P, _P, _I32, _P, _I32, _P, _P, _P], _I32),
    "pkv_bm_free": ([_P, _I64], _I32),
    "pkv_bm_block_tables": ([_P, _P, _I32, _I32, _P, _P], _I32),
    "pkv_bm_slots": ([_P, _I64, _I32, _I32, _P], _I32),
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


def pkv_decode_attention_shared_prefix(q, k_cache, v_cache, block_tables, context_lens,
                                       scale: float, shared_blocks: int, out,
                                       stream=None) -> None:
    """Cascade decode: as pkv_decode_attention for a batch whose sequences all
    share their first ``shared_blocks`` table entries (and contexts at least
    that long); the shared blocks are read once for the whole batch."""
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
    _check(load_library().pkv_decode_attention_shared_prefix(
        _ptr(q), qs, _ptr(k_cache), _ptr(v_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(context_lens), b, hq, hkv, d, float(scale), int(shared_blocks), _ptr(out),
        _stream(stream)), "pkv_decode_attention_shared_prefix")


def pkv_decode_attention_append(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                                context_lens, scale: float, out, stream=None) -> None:
    """One decode step in one kernel: store row s of k_new / v_new [B, Hkv, D]
    (sequence s's new token, at position context_lens[s] - 1) at
    slot_mapping[s] (-1: not stored), then decode q [B, Hq, D] -> out."""
    nb, hkv, d = _cache(k_cache, v_cache)
    _need(q.dim() == 3, "q: [B, Hq, D]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    ks = _rows(k_new, "k_new", hkv, d)
    vs = _rows(v_new, "v_new", hkv, d)
    _need(k_new.shape[0] == b and v_new.shape[0] == b, "k_new, v_new: one row per sequence")
    for x, n in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                 (slot_mapping, "slot_mapping")):
        _i32(x, n)
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b, "block_tables: [B, max_blocks]")
    _need(context_lens.numel() == b and slot_mapping.numel() == b,
          "context_lens, slot_mapping: [B]")
    _need(out.is_contiguous() and out.shape == q.shape and out.dtype == q.dtype and out.is_cuda,
          "out: contiguous, same shape/dtype as q")
    _check(load_library().pkv_decode_attention_append(
        _ptr(q), qs, _ptr(k_new), _ptr(v_new), ks, vs, _ptr(slot_mapping), _ptr(k_cache),
        _ptr(v_cache), nb, _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), b,
        hq, hkv, d, float(scale), _ptr(out), _stream(stream)), "pkv_decode_attention_append")


def pkv_set_shared_prefix_units(n: int) -> None:
    _check(load_library().pkv_set_shared_prefix_units(int(n)), "pkv_set_shared_prefix_units")


def pkv_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                                 out, stream=None) -> None:
    """pkv_decode_attention with its split-K scratch in the library's static
    16 MiB device array: the call allocates no device memory, for callers that
    cannot allocate (a KV pool that already holds the free memory, a process
    whose memory all comes from one caching allocator).  Raises
    PkvError(PKV_ERR_UNSUPPORTED) for a batch whose partials do not fit;
    overlapping calls on one device race on the shared array.  Device-side
    check failures are read with pkv_get_device_error, as for every call."""
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


def _int8_cache(k_codes, v_codes, k_scales, v_scales):
    """INT8 cache: codes int8 [NB, Hkv, 256, D] and scales float32 [NB, Hkv, 256]
    (each block holds its KV heads one after another)."""
    import torch
    for t, n in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _need(t.is_cuda and t.dtype == torch.int8 and t.dim() == 4 and t.is_contiguous()
              and t.shape[2] == BLOCK_SIZE, f"{n}: contiguous int8 CUDA [NB, Hkv, 256, D]")
    for t, n in ((k_scales, "k_scales"), (v_scales, "v_scales")):
        _need(t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()
              and tuple(t.shape) == tuple(k_codes.shape[:3]), f"{n}: contiguous float32 CUDA [NB, Hkv, 256]")
    _need(k_codes.shape == v_codes.shape, "k_codes and v_codes shapes differ")
    nb, hkv, _, d = k_codes.shape
    return int(nb), int(hkv), int(d)


def pkv_store_kvcache_int8(k, v, slot_mapping, k_codes, v_codes, k_scales, v_scales,
                           stream=None) -> None:
    """Quantise rows k, v [N, Hkv, D] into the INT8 cache at slot_mapping (-1 skips)."""
    nb, hkv, d = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    ks, vs = _rows(k, "k", hkv, d), _rows(v, "v", hkv, d)
    _i32(slot_mapping, "slot_mapping")
    _need(slot_mapping.numel() == k.shape[0] == v.shape[0], "row counts differ")
    _check(load_library().pkv_store_kvcache_int8(
        _ptr(k), _ptr(v), ks, vs, _ptr(slot_mapping), k.shape[0], _ptr(k_codes), _ptr(v_codes),
        _ptr(k_scales), _ptr(v_scales), nb, hkv, d, _stream(stream)), "pkv_store_kvcache_int8")


def pkv_decode_attention_int8(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens,
                              scale: float, out, stream=None) -> None:
    """Decode over the INT8 cache; out bf16 [B, Hq, D] is written."""
    import torch
    nb, hkv, d = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    _need(q.dim() == 3, "q: [B, Hq, D]")
    b, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    _i32(block_tables, "block_tables")
    _i32(context_lens, "context_lens")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b and context_lens.numel() == b,
          "block_tables [B, max_blocks], context_lens [B]")
    _need(out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous()
          and tuple(out.shape) == (b, hq, d), "out: contiguous bf16 CUDA [B, Hq, D]")
    _check(load_library().pkv_decode_attention_int8(
        _ptr(q), qs, _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), nb,
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), b, hq, hkv, d,
        float(scale), _ptr(out), _stream(stream)), "pkv_decode_attention_int8")


def pkv_prefill_attention_int8(q, k_codes, v_codes, k_scales, v_scales, block_tables,
                               cu_seqlens_q, context_lens, scale: float, out, stream=None) -> None:
    """Chunked causal prefill over the INT8 cache: q [T, Hq, D] -> out [T, Hq, D]."""
    import torch
    nb, hkv, d = _int8_cache(k_codes, v_codes, k_scales, v_scales)
    _need(q.dim() == 3, "q: [T, Hq, D]")
    t, hq = int(q.shape[0]), int(q.shape[1])
    qs = _rows(q, "q", hq, d)
    for x, n in ((block_tables, "block_tables"), (cu_seqlens_q, "cu_seqlens_q"),
                 (context_lens, "context_lens")):
        _i32(x, n)
    b = int(context_lens.numel())
    _need(block_tables.dim() == 2 and block_tables.shape[0] == b, "block_tables: [B, max_blocks]")
    _need(cu_seqlens_q.numel() == b + 1, "cu_seqlens_q: [B + 1]")
    _need(out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous()
          and tuple(out.shape) == (t, hq, d), "out: contiguous bf16 CUDA [T, Hq, D]")
    _check(load_library().pkv_prefill_attention_int8(
        _ptr(q), qs, _ptr(k_codes), _ptr(v_codes), _ptr(k_scales), _ptr(v_scales), nb,
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(cu_seqlens_q), _ptr(context_lens),
        b, t, hq, hkv, d, float(scale), _ptr(out), _stream(stream)), "pkv_prefill_attention_int8")


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


def _host_i32(values):
    """(pointer, count) of int32 host data: a contiguous CPU int32 torch tensor
    or numpy array is passed in place; any other sequence of ints is copied."""
    if hasattr(values, "data_ptr") and not getattr(values, "is_cuda", True):
        import torch
        _need(values.dtype == torch.int32 and values.is_contiguous(),
              "tokens: contiguous CPU int32 tensor")
        return ctypes.c_void_p(values.data_ptr()), int(values.numel())
    if hasattr(values, "__array_interface__"):
        import numpy as np
        _need(values.dtype == np.int32 and values.flags["C_CONTIGUOUS"],
              "tokens: contiguous int32 array")
        return ctypes.c_void_p(values.ctypes.data), int(values.size)
    values = list(values)
    return (ctypes.c_int32 * max(len(values), 1))(*values), len(values)


class BlockManager:
    """Host block manager (``pkv_bm_*``): 256-token blocks with reference
    counts and a prefix cache; produces block tables, context lengths and slot
    mappings.  Pure host code: works without a GPU."""

    def __init__(self, num_blocks: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.pkv_bm_create(int(num_blocks), ctypes.byref(h)), "pkv_bm_create")
        self._h = h
        self.num_blocks = int(num_blocks)

    def close(self) -> None:
        if self._h:
            self._lib.pkv_bm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free_blocks(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pkv_bm_ref_count(self._h, int(block)))

    def allocate(self, seq_id: int, tokens) -> int:
        """Add a sequence with its prompt; returns the number of leading tokens
        whose K/V is already cached (a multiple of 256)."""
        buf, n = _host_i32(tokens)
        cached = ctypes.c_int32(0)
        _check(self._lib.pkv_bm_allocate(self._h, int(seq_id), buf, n, ctypes.byref(cached)),
               "pkv_bm_allocate")
        return int(cached.value)

    def append(self, seq_id: int, tokens) -> list:
        """Append tokens to a sequence; returns their cache slots."""
        buf, n = _host_i32(tokens)
        slots = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pkv_bm_append(self._h, int(seq_id), buf, n, slots), "pkv_bm_append")
        return list(slots[:n])

    def append_decode(self, seq_ids, tokens) -> list:
        """One decode step: one token per sequence; returns the slot mapping."""
        seq_ids = [int(x) for x in seq_ids]
        buf, n = _host_i32(tokens)
        _need(n == len(seq_ids), "append_decode: one token per sequence")
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        slots = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pkv_bm_append_decode(self._h, ids, n, buf, slots), "pkv_bm_append_decode")
        return list(slots[:n])

    def append_decode_into(self, seq_ids, tokens, slot_mapping) -> None:
        """append_decode on CPU tensors: seq_ids int64 [B], tokens int32 [B];
        fills the CPU int32 tensor slot_mapping [B] in place."""
        import torch
        for t, dt, name in ((seq_ids, torch.int64, "seq_ids"), (tokens, torch.int32, "tokens"),
                            (slot_mapping, torch.int32, "slot_mapping")):
            _need(t.device.type == "cpu" and t.dtype == dt and t.is_contiguous()
                  and t.numel() == seq_ids.numel(), f"{name}: contiguous CPU {dt} [B]")
        _check(self._lib.pkv_bm_append_decode(self._h, _ptr(seq_ids), seq_ids.numel(),
                                              _ptr(tokens), _ptr(slot_mapping)),
               "pkv_bm_append_decode")

    def decode_step(self, seq_ids, tokens, max_blocks: int):
        """One decode step: (slot_mapping, block_tables rows, context_lens) as lists."""
        seq_ids = [int(x) for x in seq_ids]
        buf, n = _host_i32(tokens)
        _need(n == len(seq_ids), "decode_step: one token per sequence")
        mb = int(max_blocks)
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        slots = (ctypes.c_int32 * max(n, 1))()
        tables = (ctypes.c_int32 * max(n * mb, 1))()
        lens = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pkv_bm_decode_step(self._h, ids, n, buf, mb, slots, tables, lens),
               "pkv_bm_decode_step")
        return list(slots[:n]), [list(tables[i * mb:(i + 1) * mb]) for i in range(n)], list(lens[:n])

    def decode_step_into(self, seq_ids, tokens, slot_mapping, block_tables, context_lens) -> None:
        """decode_step on CPU tensors (pinned ones can be copied to the device
        asynchronously): seq_ids int64 [B], tokens int32 [B]; fills int32
        slot_mapping [B], block_tables [B, max_blocks] and context_lens [B]."""
        import torch
        b = seq_ids.numel()
        for t, dt, name in ((seq_ids, torch.int64, "seq_ids"), (tokens, torch.int32, "tokens"),
                            (slot_mapping, torch.int32, "slot_mapping"),
                            (context_lens, torch.int32, "context_lens")):
            _need(t.device.type == "cpu" and t.dtype == dt and t.is_contiguous() and t.numel() == b,
                  f"{name}: contiguous CPU {dt} [B]")
        _need(block_tables.device.type == "cpu" and block_tables.dtype == torch.int32
              and block_tables.is_contiguous() and block_tables.dim() == 2
              and block_tables.shape[0] == b, "block_tables: CPU int32 [B, max_blocks]")
        _check(self._lib.pkv_bm_decode_step(self._h, _ptr(seq_ids), b, _ptr(tokens),
                                            block_tables.shape[1], _ptr(slot_mapping),
                                            _ptr(block_tables), _ptr(context_lens)),
               "pkv_bm_decode_step")

    def free(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free(self._h, int(seq_id)), "pkv_bm_free")

    def slots(self, seq_id: int, begin: int, end: int) -> list:
        n = max(int(end) - int(begin), 0)
        out = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pkv_bm_slots(self._h, int(seq_id), int(begin), int(end), out),
               "pkv_bm_slots")
        return list(out[:n])

    def block_tables(self, seq_ids, max_blocks: int):
        """(block_tables rows as lists, context_lens list) for the sequences."""
        seq_ids = [int(x) for x in seq_ids]
        b, mb = len(seq_ids), int(max_blocks)
        ids = (ctypes.c_int64 * max(b, 1))(*seq_ids)
        tables = (ctypes.c_int32 * max(b * mb, 1))()
        lens = (ctypes.c_int32 * max(b, 1))()
        _check(self._lib.pkv_bm_block_tables(self._h, ids, b, mb, tables, lens),
               "pkv_bm_block_tables")
        return [list(tables[i * mb:(i + 1) * mb]) for i in range(b)], list(lens[:b])

    def block_tables_into(self, seq_ids, block_tables, context_lens) -> None:
        """Fill pinned or plain CPU int32 tensors block_tables [B, max_blocks]
        and context_lens [B] in place; seq_ids is best a CPU int64 tensor
        (then nothing is copied)."""
        import torch
        seq = seq_ids
        if not (isinstance(seq, torch.Tensor) and seq.device.type == "cpu"
                and seq.dtype == torch.int64 and seq.is_contiguous()):
            seq = torch.as_tensor([int(x) for x in seq_ids], dtype=torch.int64)
        _need(block_tables.device.type == "cpu" and block_tables.dtype == torch.int32
              and block_tables.is_contiguous() and block_tables.dim() == 2
              and block_tables.shape[0] == seq.numel(), "block_tables: CPU int32 [B, max_blocks]")
        _need(context_lens.device.type == "cpu" and context_lens.dtype == torch.int32
              and context_lens.is_contiguous() and context_lens.numel() == seq.numel(),
              "context_lens: CPU int32 [B]")
        _check(self._lib.pkv_bm_block_tables(self._h, _ptr(seq), seq.numel(),
                                             block_tables.shape[1], _ptr(block_tables),
                                             _ptr(context_lens)), "pkv_bm_block_tables")
