"""INT8 KV cache on the GPU against the oracle: the quantising store must give
exactly the oracle's codes and scales, and decode over the INT8 cache must
match the oracle's decode of the values the codes stand for."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import assert_close, dev, no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs():
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_get_device_error()


def int8_pool(cache):
    """The INT8 cache holding the same tokens as a bf16 pool (CPU tensors:
    codes [NB, Hkv, 256, D], scales [NB, Hkv, 256])."""
    kc, ks = oracle.quantize_pool(cache.k_cache)
    vc, vs = oracle.quantize_pool(cache.v_cache)
    return [kc, vc, ks, vs]


def tie_rows(n, hkv, d):
    """Rows whose codes include exact ties (scale 1): 127, 2.5, 3.5, -2.5, ..."""
    base = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, -0.5, 1.5, -126.5])
    x = base.repeat(d // 8)
    return x.expand(n, hkv, d).clone().to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_store_int8_codes_and_scales_are_exact(cuda_device, d):
    nb, hkv, n = 6, 4, 300
    g = torch.Generator().manual_seed(d)
    mag = torch.exp(torch.randn(n, hkv, 1, generator=g) * 3)
    k = (torch.randn(n, hkv, d, generator=g) * mag).to(torch.bfloat16)
    v = (torch.randn(n, hkv, d, generator=g) * mag).to(torch.bfloat16)
    k[:20] = tie_rows(20, hkv, d)
    v[20:30] = 0                                   # zero rows: scale 0, codes 0
    slots = torch.randperm(nb * 256, generator=g)[:n].to(torch.int32)
    slots[::7] = -1
    kc = torch.randint(-127, 128, (nb, hkv, 256, d), generator=g, dtype=torch.int8)
    vc = kc.clone()
    ks = torch.rand(nb, hkv, 256, generator=g)
    vs = ks.clone()
    want = oracle.store_kvcache_int8(k, v, slots, kc, vc, ks, vs)
    got = [dev(t) for t in (kc, vc, ks, vs)]
    pkv.pkv_store_kvcache_int8(dev(k), dev(v), dev(slots), *got)
    torch.cuda.synchronize()
    for w, gt, name in zip(want, got, ("k_codes", "v_codes", "k_scales", "v_scales")):
        assert torch.equal(gt.cpu().view(torch.int8) if gt.dtype == torch.int8 else gt.cpu().view(torch.int32),
                           w.view(torch.int8) if w.dtype == torch.int8 else w.view(torch.int32)), name
    no_device_error()


def run_int8_decode_step(case):
    """INT8 pool on the device, the new rows stored by the quantising store,
    then decode; returns the output and the device caches."""
    c = case.cache
    pool = int8_pool(c)
    kc, vc, ks, vs = [dev(t) for t in pool]
    bt, cl = dev(c.block_tables), dev(c.context_lens)
    pkv.pkv_store_kvcache_int8(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc,
                               ks, vs)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    return out, pool, (kc, vc, ks, vs)


def oracle_int8_after_store(case, pool, rows=None):
    c = case.cache
    after = oracle.store_kvcache_int8(case.k_new, case.v_new, case.slot_mapping, *pool)
    return after, oracle.decode_int8(case.q, *after, c.block_tables, c.context_lens, case.scale,
                                     rows=rows)


def check_case(case, rows=None):
    out, pool, device_cache = run_int8_decode_step(case)
    after, ref = oracle_int8_after_store(case, pool, rows)
    for w, gt in zip(after, device_cache):  # the store, at the full pool size
        assert torch.equal(gt.cpu(), w)
    if rows is None:
        assert_close(out, ref, case.name)
    else:
        assert_close(torch.stack([out[s, h] for s, h in rows]), ref, case.name)
    no_device_error()


def test_int8_tiny_decode(cuda_device):
    check_case(W.tiny_decode())


def test_int8_qwen_decode_b128(cuda_device):
    check_case(W.qwen_decode())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (64, 8), (32, 2), (16, 1)])
def test_int8_geometries(cuda_device, d, hq, hkv):
    case = W.make_decode_case("g8", [0, 1, 300, 1100, 513], hq, hkv, d, 24, seed=hq * 7 + hkv + d)
    check_case(case)


@pytest.mark.parametrize("d", [64, 128])
def test_int8_chunk_and_block_edges(cuda_device, d):
    """Contexts on either side of the 32-token half-chunk, the 64-token INT8
    chunk and the 256-token block edges (the last chunk partly or wholly
    past the context, a half with no token)."""
    lens = [1, 31, 32, 33, 63, 64, 65, 96, 127, 128, 129, 255, 256, 257, 511, 513]
    case = W.make_decode_case("edge8", lens, 16, 8, d, 40, seed=80 + d)
    check_case(case)


def test_int8_long_contexts(cuda_device):
    case = W.make_decode_case("long8", [9000, 4097, 31], 16, 8, 128, 64, seed=77)
    check_case(case)


@pytest.mark.parametrize("cap", [1, 3])
def test_int8_split_cap_does_not_change_result(cuda_device, cap):
    case = W.make_decode_case("cap8", [1, 300, 1500, 4000], 16, 8, 128, 40, seed=78, k_scale=3.0)
    pkv.pkv_set_max_splits(cap)
    try:
        check_case(case)
    finally:
        pkv.pkv_set_max_splits(0)


def test_int8_many_kv_heads(cuda_device):
    """32 KV heads (one query head each), head_dim 64: each head's tiles and
    scales are its own contiguous runs of the block."""
    case = W.make_decode_case("h32", [5, 300, 700], 32, 32, 64, 12, seed=79)
    check_case(case)


def test_int8_graph_replays_follow_new_inputs(cuda_device):
    case = W.qwen_decode(seed=1047, num_seqs=24)
    c = case.cache
    pool = int8_pool(c)
    kc, vc, ks, vs = [dev(t) for t in pool]
    bt, cl = dev(c.block_tables), dev(c.context_lens)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_reserve_workspace(24, 16, 128, int(bt.shape[1]))
    pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)
    for seed in (1, 2):
        newq = W.randn_bf16(tuple(case.q.shape), torch.Generator().manual_seed(seed))
        q.copy_(dev(newq))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.decode_int8(newq, *pool, c.block_tables, c.context_lens, case.scale)
        assert_close(out, ref, f"replay {seed}")
    no_device_error()


def test_int8_bad_block_and_context_give_zeros(cuda_device):
    case = W.make_decode_case("bad8", [300, 600, 40], 16, 8, 128, 16, seed=1)
    pool = int8_pool(case.cache)
    kc, vc, ks, vs = [dev(t) for t in pool]
    bt, cl = dev(case.cache.block_tables), dev(case.cache.context_lens)
    bt[1, 1] = 16                         # == num_blocks: out of range
    cl[2] = 16 * 256 + 1                  # beyond the table width
    q = dev(case.q)
    out = torch.full_like(q, 7.0)
    pkv.pkv_decode_attention_int8(q, kc, vc, ks, vs, bt, cl, case.scale, out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    ref = oracle.decode_int8(case.q, *pool, case.cache.block_tables, case.cache.context_lens,
                             case.scale, rows=[(0, h) for h in range(16)])
    assert_close(out[0], ref, "unaffected sequence")
