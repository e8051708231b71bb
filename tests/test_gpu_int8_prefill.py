"""Chunked prefill over the INT8 cache on the GPU against the oracle.

The kernel dequantises each tile to bf16 (code * scale, rounded to nearest
even) in shared memory and then runs the bf16 prefill pipeline, so:
  - against the oracle's exact values code * scale it stays within the
    bf16-attention tolerance of the other prefill tests;
  - with integer rows (every scale 1, dequantisation exact) it returns the
    bf16 prefill's output bit for bit;
  - a query that sees one overwhelming key returns that key's dequantised
    V row, bf16(code * scale), exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.parallel as oracle_parallel
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import assert_close, cache_to_device, dev, no_device_error, run_prefill_step

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs():
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()


def int8_pool(cache):
    """CPU INT8 pool (k_codes, v_codes, k_scales, v_scales) holding the same
    tokens as a bf16 pool."""
    kc, ks = oracle.quantize_pool(cache.k_cache)
    vc, vs = oracle.quantize_pool(cache.v_cache)
    return [kc, vc, ks, vs]


def run_int8_prefill_step(case, pool=None):
    """INT8 pool on the device, the chunk's rows stored by the quantising
    store, then the INT8 prefill; returns (out, pool, device pool)."""
    c = case.cache
    pool = int8_pool(c) if pool is None else pool
    kc, vc, ks, vs = [dev(t) for t in pool]
    pkv.pkv_store_kvcache_int8(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc,
                               ks, vs)
    q = dev(case.q)
    out = torch.full_like(q, float("nan"))
    pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, dev(c.block_tables), dev(case.cu_seqlens_q),
                                   dev(c.context_lens), case.scale, out)
    torch.cuda.synchronize()
    return out, pool, (kc, vc, ks, vs)


def oracle_int8_prefill_after_store(case, pool, rows=None):
    c = case.cache
    after = oracle.store_kvcache_int8(case.k_new, case.v_new, case.slot_mapping, *pool)
    if rows is None:
        return oracle_parallel.prefill_int8(case.q, *after, c.block_tables, case.cu_seqlens_q,
                                            c.context_lens, case.scale)
    return oracle.prefill_int8(case.q, *after, c.block_tables, case.cu_seqlens_q, c.context_lens,
                               case.scale, rows=rows)


def check_case(case, rows=None):
    out, pool, _ = run_int8_prefill_step(case)
    ref = oracle_int8_prefill_after_store(case, pool, rows)
    if rows is None:
        assert_close(out, ref, case.name)
    else:
        assert_close(torch.stack([out[t, h] for t, h in rows]), ref, case.name)
    no_device_error()


@pytest.mark.parametrize("cached,chunk", [(0, 1), (0, 130), (5, 1), (255, 2), (256, 100),
                                          (300, 129), (1000, 300)])
def test_int8_prefill_shapes_full(cuda_device, cached, chunk):
    case = W.make_prefill_case("p8", [cached, cached + 17], [chunk, chunk + 3], 16, 8, 128, 48,
                               seed=cached + chunk + 500, skip_prob=0.05)
    check_case(case)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 2), (16, 1)])
def test_int8_prefill_geometries(cuda_device, d, hq, hkv):
    case = W.make_prefill_case("g8", [0, 300, 77], [200, 70, 1], hq, hkv, d, 24,
                               seed=hq * 3 + hkv + d)
    check_case(case)


def test_int8_prefill_ragged_batch_with_empty_chunks(cuda_device):
    case = W.make_prefill_case("r8", [10, 0, 700, 256, 3], [0, 33, 0, 257, 64], 16, 8, 128, 32,
                               seed=509)
    check_case(case)


def test_int8_chunked_prefill_8x512_full(cuda_device):
    """Full size (8 x 512 queries over 4608 keys, ~5% of slots -1): every
    (query, head) output against the oracle (run over the host cores)."""
    check_case(W.chunked_prefill())


def test_int8_prefill_is_bf16_prefill_when_quantisation_is_exact(cuda_device):
    """Integer K/V rows with a +-127 in each (every scale 1): the dequantised
    tiles equal the bf16 tiles, so both kernels give the same bits."""
    case = W.make_prefill_case("exact8", [0, 300, 1000], [130, 64, 200], 16, 8, 128, 24,
                               seed=511)
    g = torch.Generator().manual_seed(512)
    for t in (case.cache.k_cache, case.cache.v_cache, case.k_new, case.v_new):
        ints = torch.randint(-126, 127, t.shape, generator=g).float()
        ints[..., 0] = torch.where(torch.rand(t.shape[:-1], generator=g) < 0.5, 127.0, -127.0)
        t.copy_(ints.to(torch.bfloat16))
    case.q.copy_((case.q.float() / 64).to(torch.bfloat16))
    out8, pool, _ = run_int8_prefill_step(case)
    assert torch.all(pool[2] == 1) and torch.all(pool[3] == 1)
    out16, _, _ = run_prefill_step(case)
    assert torch.equal(out8.view(torch.int16), out16.view(torch.int16))
    no_device_error()


def test_int8_prefill_dominant_key_returns_dequantised_row(cuda_device):
    """Queries that see a planted key with an overwhelming logit return its
    V row as bf16(code * scale) exactly, for every head of its KV head."""
    case = W.make_prefill_case("dom8", [300], [200], 16, 8, 128, 8, seed=513)
    c = case.cache
    q = torch.zeros_like(case.q)
    q[..., 0] = 16.0
    kc = c.k_cache.clone()
    kc[..., 0] = 0.0
    k_new = case.k_new.clone()
    k_new[..., 0] = 0.0
    t_star = 123                                   # a cached position every query sees
    blk = int(c.block_tables[0, t_star // 256])
    kc[blk, t_star % 256, :, 0] = 64.0             # codes: +127 at d = 0, 0 elsewhere
    case.q, case.k_new = q, k_new
    case.cache.k_cache = kc
    out, pool, _ = run_int8_prefill_step(case)
    vcodes, vscales = pool[1], pool[3]
    for h in range(8):
        want = (vcodes[blk, h, t_star % 256].float() * vscales[blk, h, t_star % 256]).to(torch.bfloat16)
        got = out[:, 2 * h:2 * h + 2].cpu()
        assert torch.equal(got.view(torch.int16), want.expand_as(got).view(torch.int16)), h
    no_device_error()


def test_int8_prefill_of_one_query_matches_int8_decode_oracle(cuda_device):
    case = W.make_decode_case("x8", [1, 256, 257, 513, 2000], 16, 8, 128, 24, seed=514)
    c = case.cache
    pool = int8_pool(c)
    kc, vc, ks, vs = [dev(t) for t in pool]
    pkv.pkv_store_kvcache_int8(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc,
                               ks, vs)
    q = dev(case.q)
    out = torch.empty_like(q)
    cu = torch.arange(0, 6, dtype=torch.int32)
    pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, dev(c.block_tables), dev(cu),
                                   dev(c.context_lens), case.scale, out)
    torch.cuda.synchronize()
    after = oracle.store_kvcache_int8(case.k_new, case.v_new, case.slot_mapping, *pool)
    ref = oracle.decode_int8(case.q, *after, c.block_tables, c.context_lens, case.scale)
    assert_close(out, ref, "INT8 prefill Lq=1")
    no_device_error()


def test_int8_prefill_long_context_sampled(cuda_device):
    """One 256-token chunk over 8192 cached keys: long per-tile key loops."""
    case = W.make_prefill_case("long8", [8192], [256], 16, 8, 128, 40, seed=515, skip_prob=0.05)
    rows = [(t, (t * 7) % 16) for t in range(0, 256, 9)] + [(255, h) for h in range(16)]
    check_case(case, rows=rows)


def test_int8_prefill_bad_block_and_chunk_give_zeros(cuda_device):
    case = W.make_prefill_case("bad8", [300, 100], [100, 50], 16, 8, 128, 8, seed=516)
    pool = int8_pool(case.cache)
    kc, vc, ks, vs = [dev(t) for t in pool]
    bt, cl = dev(case.cache.block_tables), dev(case.cache.context_lens)
    bt[0, 0] = -3                                  # sequence 0: bad block id
    cl[1] = 20                                     # sequence 1: Lq = 50 > C = 20
    q = dev(case.q)
    out = torch.full_like(q, 7.0)
    pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, bt, dev(case.cu_seqlens_q), cl, case.scale,
                                   out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out == 0)


def test_int8_prefill_expired_waits_report_timeout_and_recover(cuda_device):
    case = W.make_prefill_case("t8", [2000], [300], 16, 8, 128, 16, seed=517)
    pool = int8_pool(case.cache)
    pkv.pkv_set_wait_limit_ns(0)
    run_int8_prefill_step(case, pool)
    code, site = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_TIMEOUT, (code, site)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    out, _, _ = run_int8_prefill_step(case, pool)
    assert_close(out, oracle_int8_prefill_after_store(case, pool), "after timeouts")
    no_device_error()


def test_int8_prefill_graph_replays_follow_new_inputs(cuda_device):
    case = W.make_prefill_case("g8r", [3000, 100, 700], [300, 200, 64], 16, 8, 128, 64, seed=518)
    c = case.cache
    pool = int8_pool(c)
    kc, vc, ks, vs = [dev(t) for t in pool]
    q = dev(case.q)
    kn, vn, sm = dev(case.k_new), dev(case.v_new), dev(case.slot_mapping)
    bt, cu, cl = dev(c.block_tables), dev(case.cu_seqlens_q), dev(c.context_lens)
    out = torch.empty_like(q)

    def step():
        pkv.pkv_store_kvcache_int8(kn, vn, sm, kc, vc, ks, vs)
        pkv.pkv_prefill_attention_int8(q, kc, vc, ks, vs, bt, cu, cl, case.scale, out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    after = oracle.store_kvcache_int8(case.k_new, case.v_new, case.slot_mapping, *pool)
    rows = [(t, (t * 5) % 16) for t in range(0, 564, 7)]
    gen = torch.Generator().manual_seed(519)
    for i in range(2):
        q_host = torch.randn(case.q.shape, generator=gen).to(torch.bfloat16)
        q.copy_(q_host)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.prefill_int8(q_host, *after, c.block_tables, case.cu_seqlens_q,
                                  c.context_lens, case.scale, rows=rows)
        assert_close(torch.stack([out[t, h] for t, h in rows]), ref, f"replay {i}")
    no_device_error()
