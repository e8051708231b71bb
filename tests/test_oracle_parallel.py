"""The multi-core driver of the oracle returns exactly what the
single-threaded oracle returns: it only cuts the work into per-sequence (and
per-head-group) calls of the same C functions and puts the rows back."""
import numpy as np
import torch

import oracle
from oracle import parallel
from paged_kv_cache_493_b300 import workloads as W


def test_parallel_decode_equals_serial():
    case = W.make_decode_case("p", [1, 37, 256, 300, 700, 0, 513], 8, 2, 64, 24, seed=31)
    c = case.cache
    ref = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    got = parallel.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens,
                          case.scale, workers=4)
    assert np.array_equal(got, ref)


def test_parallel_prefill_equals_serial():
    case = W.make_prefill_case("p", [300, 0, 17], [40, 33, 0], 8, 2, 64, 16, seed=32)
    c = case.cache
    ref = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, case.cu_seqlens_q,
                         c.context_lens, case.scale)
    for groups in (1, 2, 8):
        got = parallel.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, case.cu_seqlens_q,
                               c.context_lens, case.scale, workers=4, head_groups=groups)
        assert np.array_equal(got, ref), groups


def test_parallel_decode_int8_equals_serial():
    case = W.make_decode_case("p", [5, 260, 90], 4, 2, 64, 8, seed=33)
    c = case.cache
    kc, ks = oracle.quantize_pool(c.k_cache)
    vc, vs = oracle.quantize_pool(c.v_cache)
    ref = oracle.decode_int8(case.q, kc, vc, ks, vs, c.block_tables, c.context_lens, case.scale)
    got = parallel.decode_int8(case.q, kc, vc, ks, vs, c.block_tables, c.context_lens,
                               case.scale, workers=3)
    assert np.array_equal(got, ref)


def test_parallel_prefill_int8_equals_serial():
    case = W.make_prefill_case("p", [300, 0, 17], [40, 33, 0], 8, 2, 64, 16, seed=34)
    c = case.cache
    kc, ks = oracle.quantize_pool(c.k_cache)
    vc, vs = oracle.quantize_pool(c.v_cache)
    ref = oracle.prefill_int8(case.q, kc, vc, ks, vs, c.block_tables, case.cu_seqlens_q,
                              c.context_lens, case.scale)
    for groups in (1, 4):
        got = parallel.prefill_int8(case.q, kc, vc, ks, vs, c.block_tables, case.cu_seqlens_q,
                                    c.context_lens, case.scale, workers=3, head_groups=groups)
        assert np.array_equal(got, ref), groups


def test_worker_count_respects_memory():
    assert parallel.pick_workers(0, workers=5) == 5
    assert parallel.pick_workers(1 << 62) == 1   # one task's buffers exceed the memory
