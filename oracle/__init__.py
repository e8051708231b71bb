"""ctypes front end of the fp64 CPU oracle (``pkv_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  Inputs are CPU torch
tensors (bf16 viewed as raw uint16 bits, int32 metadata); outputs are fp64
numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")

ERRORS = {0: "ok", 1: "bad argument", 2: "block id out of range",
          3: "context length out of range", 4: "chunk longer than context",
          5: "slot out of range", 6: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (plain -O2, no fast-math, no vectorising flags)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        _lib.oracle_store_kvcache.argtypes = [P, P, I64, I64, P, I64, P, P, I64, I32, I32]
        _lib.oracle_gather.argtypes = [P, P, I64, I32, I32, P, I32, I32, P, P]
        _lib.oracle_attend.argtypes = [P, P, P, I32, I32, I32, I32, D, P, P]
        _lib.oracle_attend.restype = None
        _lib.oracle_decode.argtypes = [P, P, P, I64, P, I32, P, I32, I32, I32, I32, D, P, I32, P]
        _lib.oracle_prefill.argtypes = [P, P, P, I64, P, I32, P, P, I32, I32, I32, I32, D, P, I32, P]
        _lib.oracle_bf16_to_f64.argtypes = [P, I64, P]
        _lib.oracle_bf16_to_f64.restype = None
        _lib.oracle_quantize_row.argtypes = [P, I32, P, P]
        _lib.oracle_quantize_row.restype = None
        _lib.oracle_quantize_rows.argtypes = [P, I64, I32, P, P]
        _lib.oracle_quantize_rows.restype = None
        _lib.oracle_store_kvcache_int8.argtypes = [P, P, I64, I64, P, I64, P, P, P, P, I64, I32, I32]
        _lib.oracle_gather_int8.argtypes = [P, P, P, P, I64, I32, I32, P, I32, I32, P, P]
        _lib.oracle_decode_int8.argtypes = [P, P, P, P, P, I64, P, I32, P, I32, I32, I32, I32, D,
                                            P, I32, P]
        _lib.oracle_prefill_int8.argtypes = [P, P, P, P, P, I64, P, I32, P, P, I32, I32, I32,
                                             I32, D, P, I32, P]
    return _lib


def _bits(t: torch.Tensor) -> torch.Tensor:
    assert t.device.type == "cpu" and t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)


def _i32(t) -> torch.Tensor:
    t = torch.as_tensor(t, dtype=torch.int32)
    assert t.device.type == "cpu"
    return t.contiguous()


def _ptr(t) -> ctypes.c_void_p:
    if isinstance(t, np.ndarray):
        return ctypes.c_void_p(t.ctypes.data)
    return ctypes.c_void_p(t.data_ptr())


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"error {rc}"))


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    b = _bits(t)
    out = np.empty(b.numel(), dtype=np.float64)
    lib().oracle_bf16_to_f64(_ptr(b), b.numel(), _ptr(out))
    return out.reshape(tuple(t.shape))


def store_kvcache(k: torch.Tensor, v: torch.Tensor, slot_mapping, k_cache: torch.Tensor,
                  v_cache: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """Returns new (k_cache, v_cache) bf16 tensors; the inputs are not modified."""
    nb, bs, hkv, d = k_cache.shape
    kc = k_cache.clone().contiguous()
    vc = v_cache.clone().contiguous()
    kb, vb, sm = _bits(k), _bits(v), _i32(slot_mapping)
    n = int(sm.numel())
    _check(lib().oracle_store_kvcache(_ptr(kb), _ptr(vb), hkv * d, hkv * d, _ptr(sm), n,
                                      _ptr(kc.view(torch.int16)), _ptr(vc.view(torch.int16)),
                                      nb, hkv, d))
    return kc, vc


def gather(k_cache, v_cache, block_table_row, context_len: int) -> Tuple[np.ndarray, np.ndarray]:
    nb, bs, hkv, d = k_cache.shape
    row = _i32(block_table_row)
    n = max(int(context_len), 1)
    K = np.zeros((n, hkv, d), dtype=np.float64)
    V = np.zeros((n, hkv, d), dtype=np.float64)
    kb, vb = _bits(k_cache), _bits(v_cache)
    _check(lib().oracle_gather(_ptr(kb), _ptr(vb), nb, hkv, d, _ptr(row),
                               int(row.numel()), int(context_len), _ptr(K), _ptr(V)))
    return K[:context_len], V[:context_len]


def attend(q_row: np.ndarray, K: np.ndarray, V: np.ndarray, kv_head: int, n_keys: int,
           scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """One query row against gathered K/V; returns (out[D], probs[n_keys])."""
    q_row = np.ascontiguousarray(q_row, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    hkv, d = K.shape[1], K.shape[2]
    out = np.zeros(d, dtype=np.float64)
    probs = np.zeros(max(n_keys, 1), dtype=np.float64)
    lib().oracle_attend(_ptr(q_row), _ptr(K), _ptr(V), hkv, d, int(kv_head), int(n_keys),
                        float(scale), _ptr(out), _ptr(probs))
    return out, probs[:n_keys]


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables,
           context_lens, scale: float,
           rows: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Full [B, Hq, D] output, or [len(rows), D] for (seq, q head) pairs."""
    b, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d == d2
    bt, cl = _i32(block_tables), _i32(context_lens)
    if rows is None:
        out = np.zeros((b, hq, d), dtype=np.float64)
        rptr, nr = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((r.shape[0], d), dtype=np.float64)
        rptr, nr = _ptr(r), r.shape[0]
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    _check(lib().oracle_decode(_ptr(qb), _ptr(kb), _ptr(vb), nb,
                               _ptr(bt), int(bt.shape[1]), _ptr(cl), b, hq, hkv, d, float(scale),
                               rptr, nr, _ptr(out)))
    return out


def prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables,
            cu_seqlens_q, context_lens, scale: float,
            rows: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Full [T, Hq, D] output, or [len(rows), D] for (token row, q head) pairs."""
    t, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d == d2
    bt, cu, cl = _i32(block_tables), _i32(cu_seqlens_q), _i32(context_lens)
    if rows is None:
        out = np.zeros((t, hq, d), dtype=np.float64)
        rptr, nr = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((r.shape[0], d), dtype=np.float64)
        rptr, nr = _ptr(r), r.shape[0]
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    _check(lib().oracle_prefill(_ptr(qb), _ptr(kb), _ptr(vb), nb,
                                _ptr(bt), int(bt.shape[1]), _ptr(cu), _ptr(cl), int(cu.numel() - 1),
                                hq, hkv, d, float(scale), rptr, nr, _ptr(out)))
    return out


# ---------------------------------------------------------------------------
# INT8 KV cache: codes int8 [num_blocks, Hkv, 256, D], scales float32
# [num_blocks, Hkv, 256] (each block holds its KV heads one after another);
# a value is code * scale.
# ---------------------------------------------------------------------------

def quantize_rows(x: torch.Tensor) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 [..., D] -> (int8 codes [..., D], float32 scales [...]), one scale per row."""
    xb = _bits(x).reshape(-1, x.shape[-1])
    n, d = xb.shape
    codes = np.zeros((n, d), dtype=np.int8)
    scales = np.zeros(n, dtype=np.float32)
    lib().oracle_quantize_rows(_ptr(xb), n, d, _ptr(codes), _ptr(scales))
    return codes.reshape(tuple(x.shape)), scales.reshape(tuple(x.shape[:-1]))


def quantize_pool(cache: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """A bf16 pool [NB, 256, Hkv, D] as an INT8 pool holding the same tokens:
    (codes int8 [NB, Hkv, 256, D], scales float32 [NB, Hkv, 256]) -- every
    row quantised, then laid out head-major within each block."""
    codes, scales = quantize_rows(cache)
    return (torch.from_numpy(codes).transpose(1, 2).contiguous(),
            torch.from_numpy(scales).transpose(1, 2).contiguous())


def store_kvcache_int8(k: torch.Tensor, v: torch.Tensor, slot_mapping, k_codes, v_codes,
                       k_scales, v_scales):
    """Returns new (k_codes, v_codes, k_scales, v_scales) CPU tensors; inputs unchanged."""
    nb, hkv, bs, d = k_codes.shape
    kc, vc = k_codes.clone().contiguous(), v_codes.clone().contiguous()
    ks, vs = k_scales.clone().contiguous(), v_scales.clone().contiguous()
    kb, vb, sm = _bits(k), _bits(v), _i32(slot_mapping)
    _check(lib().oracle_store_kvcache_int8(_ptr(kb), _ptr(vb), hkv * d, hkv * d, _ptr(sm),
                                           int(sm.numel()), _ptr(kc), _ptr(vc), _ptr(ks),
                                           _ptr(vs), nb, hkv, d))
    return kc, vc, ks, vs


def gather_int8(k_codes, v_codes, k_scales, v_scales, block_table_row,
                context_len: int) -> Tuple[np.ndarray, np.ndarray]:
    nb, hkv, bs, d = k_codes.shape
    row = _i32(block_table_row)
    n = max(int(context_len), 1)
    K = np.zeros((n, hkv, d), dtype=np.float64)
    V = np.zeros((n, hkv, d), dtype=np.float64)
    kc, vc = k_codes.contiguous(), v_codes.contiguous()
    ks, vs = k_scales.contiguous(), v_scales.contiguous()
    _check(lib().oracle_gather_int8(_ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, hkv, d,
                                    _ptr(row), int(row.numel()), int(context_len), _ptr(K),
                                    _ptr(V)))
    return K[:context_len], V[:context_len]


def decode_int8(q: torch.Tensor, k_codes, v_codes, k_scales, v_scales, block_tables,
                context_lens, scale: float,
                rows: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Decode over an INT8 cache: full [B, Hq, D] output, or [len(rows), D]."""
    b, hq, d = q.shape
    nb, hkv, bs, d2 = k_codes.shape
    assert d == d2 and k_codes.dtype == torch.int8 and k_scales.dtype == torch.float32
    bt, cl = _i32(block_tables), _i32(context_lens)
    if rows is None:
        out = np.zeros((b, hq, d), dtype=np.float64)
        rptr, nr = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((r.shape[0], d), dtype=np.float64)
        rptr, nr = _ptr(r), r.shape[0]
    kc, vc = k_codes.contiguous(), v_codes.contiguous()
    ks, vs = k_scales.contiguous(), v_scales.contiguous()
    qb = _bits(q)
    _check(lib().oracle_decode_int8(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb,
                                    _ptr(bt), int(bt.shape[1]), _ptr(cl), b, hq, hkv, d,
                                    float(scale), rptr, nr, _ptr(out)))
    return out


def prefill_int8(q: torch.Tensor, k_codes, v_codes, k_scales, v_scales, block_tables,
                 cu_seqlens_q, context_lens, scale: float,
                 rows: Optional[Sequence[Tuple[int, int]]] = None) -> np.ndarray:
    """Chunked prefill over an INT8 cache: full [T, Hq, D] output, or
    [len(rows), D] for (token row, q head) pairs."""
    t, hq, d = q.shape
    nb, hkv, bs, d2 = k_codes.shape
    assert d == d2 and k_codes.dtype == torch.int8 and k_scales.dtype == torch.float32
    bt, cu, cl = _i32(block_tables), _i32(cu_seqlens_q), _i32(context_lens)
    if rows is None:
        out = np.zeros((t, hq, d), dtype=np.float64)
        rptr, nr = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        out = np.zeros((r.shape[0], d), dtype=np.float64)
        rptr, nr = _ptr(r), r.shape[0]
    kc, vc = k_codes.contiguous(), v_codes.contiguous()
    ks, vs = k_scales.contiguous(), v_scales.contiguous()
    qb = _bits(q)
    _check(lib().oracle_prefill_int8(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb,
                                     _ptr(bt), int(bt.shape[1]), _ptr(cu), _ptr(cl),
                                     int(cu.numel() - 1), hq, hkv, d, float(scale), rptr, nr,
                                     _ptr(out)))
    return out
