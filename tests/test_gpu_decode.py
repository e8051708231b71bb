"""Paged decode attention on the GPU against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import (assert_close, cache_to_device, dev, no_device_error,
                     oracle_decode_after_store, run_decode_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs():
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    yield
    pkv.pkv_set_max_splits(0)


def test_tiny_decode_full(cuda_device):
    case = W.tiny_decode()
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), "tiny_decode")
    no_device_error()


def test_qwen_decode_b128_full(cuda_device):
    case = W.qwen_decode()
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), "qwen_decode_b128")
    no_device_error()


def test_prefix_decode_b64_full(cuda_device):
    case = W.prefix_decode()
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), "prefix_decode_b64")
    no_device_error()


def test_long_decode_32k_full(cuda_device):
    """Full size (16 x 32768, 2048-block pool, K x3), every (sequence, head)
    output against the oracle (run over the host cores)."""
    case = W.long_decode()
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), "long_decode_32k")
    no_device_error()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2), (32, 2)])
def test_decode_geometries(cuda_device, d, hq, hkv):
    lens = [0, 1, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000]
    case = W.make_decode_case("g", lens, hq, hkv, d, 40, seed=hq * 100 + hkv + d)
    out, _, _ = run_decode_step(case)
    ref = oracle_decode_after_store(case)
    assert_close(out, ref, f"d={d} hq={hq} hkv={hkv}")
    assert torch.all(out[0] == 0)  # empty context -> zeros
    no_device_error()


@pytest.mark.parametrize("cap", [1, 2, 3, 7, 64])
def test_split_cap_does_not_change_result(cuda_device, cap):
    case = W.make_decode_case("s", [1, 300, 1500, 4000], 16, 8, 128, 40, seed=77, k_scale=3.0)
    pkv.pkv_set_max_splits(cap)
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), f"cap={cap}")
    no_device_error()


def test_single_key_returns_value_bit_exact(cuda_device):
    case = W.tiny_decode()
    out, kc, vc = run_decode_step(case)
    blk = int(case.cache.block_tables[0, 0])
    # context 1: the stored new row is the only key, so out = its V row exactly.
    for h in range(4):
        assert torch.equal(out[0, h].cpu(), case.v_new[0, h // 2])


def test_dominant_key_selects_value_bit_exact(cuda_device):
    """A planted key whose logit exceeds all others by > 127 (log2 units) makes
    every other weight underflow to 0, so the output is that V row exactly:
    this pins the block-table addressing through the kernel."""
    lens = [300, 1000, 4000, 2]
    case = W.make_decode_case("p", lens, 16, 8, 128, 40, seed=5)
    c = case.cache
    q = torch.zeros_like(case.q)
    q[:, :, 0] = 16.0
    kc = c.k_cache.clone()
    kc[..., 0] = 0.0
    k_new = case.k_new.clone()
    k_new[..., 0] = 0.0
    planted = [(0, 298), (1, 517), (2, 3333), (3, 0)]  # never the newly stored position
    for s, t in planted:
        blk = int(c.block_tables[s, t // 256])
        kc[blk, t % 256, :, 0] = 64.0   # logit 1024 / sqrt(128) = 90.5 -> 130.6 in log2 units
    case.q, case.k_new = q, k_new
    case.cache.k_cache = kc
    out, kcd, vcd = run_decode_step(case)
    vpost = vcd.cpu()
    for s, t in planted:
        blk = int(c.block_tables[s, t // 256])
        for h in range(16):
            assert torch.equal(out[s, h].cpu(), vpost[blk, t % 256, h // 2]), (s, t, h)


def test_block_relabelling_and_prefix_copies(cuda_device):
    case = W.make_decode_case("r", [2 * 256 + 10, 2 * 256 + 300, 2 * 256 + 1], 16, 8, 128, 24,
                              seed=21, shared_prefix_blocks=2)
    out, kc, vc = run_decode_step(case)
    c = case.cache
    # (a) relabel every physical block
    perm = torch.randperm(c.num_blocks, generator=torch.Generator().manual_seed(2))
    nk, nv = torch.empty_like(kc), torch.empty_like(vc)
    nk[dev(perm)] = kc
    nv[dev(perm)] = vc
    nt = c.block_tables.clone()
    m = nt >= 0
    nt[m] = perm.to(torch.int32)[nt[m].long()]
    q = dev(case.q)
    o2 = torch.empty_like(q)
    pkv.pkv_decode_attention(q, nk, nv, dev(nt), dev(c.context_lens), case.scale, o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, out)
    # (b) private copies of the shared prefix blocks
    tb = c.block_tables
    used = set(int(x) for x in tb.flatten().tolist() if x >= 0)
    free = [b for b in range(c.num_blocks) if b not in used]
    pk, pv_, pt = kc.clone(), vc.clone(), tb.clone()
    for s in (1, 2):
        for j in range(2):
            dst = free.pop()
            pk[dst] = kc[int(tb[s, j])]
            pv_[dst] = vc[int(tb[s, j])]
            pt[s, j] = dst
    o3 = torch.empty_like(q)
    pkv.pkv_decode_attention(q, pk, pv_, dev(pt), dev(c.context_lens), case.scale, o3)
    torch.cuda.synchronize()
    assert torch.equal(o3, out)
    no_device_error()


def test_strided_query_and_non_default_stream(cuda_device):
    case = W.make_decode_case("q", [5, 700, 2049], 16, 8, 128, 24, seed=8)
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    g = torch.Generator().manual_seed(1)
    qkv = dev(W.randn_bf16((3, 32, 128), g))
    qkv[:, :16] = dev(case.q)
    q = qkv[:, :16]
    out = torch.empty(3, 16, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out, stream=s)
    s.synchronize()
    assert_close(out, oracle_decode_after_store(case), "strided q")


def test_decode_call_finishes_promptly(cuda_device):
    """A launch that only ends when a bounded wait expires still gives right
    answers; this catches it by time (the 128-sequence batch takes well under a
    millisecond on a B300, a drain or wait expiry takes a second or more)."""
    import time
    case = W.qwen_decode()
    kc, vc, bt, cl = cache_to_device(case.cache)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    assert (time.perf_counter() - t0) / 5 < 0.05
    no_device_error()


def test_graph_replays_follow_new_inputs(cuda_device):
    """Store + decode captured once in a CUDA graph (as a serving engine
    replays its decode step), then replayed over three different query
    batches written into the captured buffers: every replay must give that
    batch's attention.  Long contexts over a few pairs make the decode cut
    every (sequence, KV head) context into several pieces, so each replay
    goes through the cross-block merge and its arrival counters."""
    case = W.make_decode_case("graph", [3000, 9000, 17, 5000], 16, 8, 128, 96, seed=511)
    q, kc, vc, bt, cl = (dev(case.q), *cache_to_device(case.cache))
    kn, vn, sm = dev(case.k_new), dev(case.v_new), dev(case.slot_mapping)
    out = torch.empty_like(q)
    pkv.pkv_reserve_workspace(case.num_seqs, 16, 128, bt.shape[1])

    def step():
        pkv.pkv_store_kvcache(kn, vn, sm, kc, vc)
        pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out)

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
    gen = torch.Generator().manual_seed(77)
    for i in range(3):
        q_host = torch.randn(case.q.shape, generator=gen).to(torch.bfloat16)
        q.copy_(q_host)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        replayed = W.DecodeCase(**{**case.__dict__, "q": q_host})
        assert_close(out, oracle_decode_after_store(replayed), f"replay {i}")
    no_device_error()


def test_decode_negative_scale(cuda_device):
    case = W.make_decode_case("neg", [1, 40, 256, 700, 3000], 16, 8, 128, 32, seed=92,
                              scale=-0.08)
    out, _, _ = run_decode_step(case)
    assert_close(out, oracle_decode_after_store(case), "negative scale")
    no_device_error()
