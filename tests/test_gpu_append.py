"""Fused store + decode (pkv_decode_attention_append) on the GPU.

One kernel does what pkv_store_kvcache followed by pkv_decode_attention does:
the new rows land in the cache bit for bit (checked over the whole pool
against the oracle's store) and the attention output matches the oracle's
store-then-decode within the attention tolerance.
"""
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import assert_close, cache_to_device, dev, no_device_error, oracle_decode_after_store

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs(cuda_device):
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_set_max_splits(0)
    pkv.pkv_get_device_error()


def run_append(case, slot_mapping=None):
    kc, vc, bt, cl = cache_to_device(case.cache)
    q = dev(case.q)
    out = torch.full_like(q, float("nan"))
    sm = case.slot_mapping if slot_mapping is None else slot_mapping
    pkv.pkv_decode_attention_append(q, dev(case.k_new), dev(case.v_new), dev(sm), kc, vc, bt, cl,
                                    case.scale, out)
    torch.cuda.synchronize()
    return out, kc, vc


def check_pool(case, kc, vc, slot_mapping):
    c = case.cache
    rk, rv = oracle.store_kvcache(case.k_new, case.v_new, slot_mapping, c.k_cache, c.v_cache)
    assert torch.equal(kc.cpu().view(torch.int16), rk.view(torch.int16)), "k_cache"
    assert torch.equal(vc.cpu().view(torch.int16), rv.view(torch.int16)), "v_cache"


@pytest.mark.parametrize("name", ["tiny_decode", "qwen_decode_b128"])
def test_append_workloads(cuda_device, name):
    case = W.WORKLOADS[name]()
    out, kc, vc = run_append(case)
    check_pool(case, kc, vc, case.slot_mapping)
    assert_close(out, oracle_decode_after_store(case), name)
    no_device_error()


def test_append_long_contexts_cut_across_blocks(cuda_device):
    case = W.make_decode_case("l", [1, 31, 32, 33, 5000, 9000, 257], 16, 8, 128, 80, seed=701,
                              k_scale=3.0)
    for cap in (0, 2):
        pkv.pkv_set_max_splits(cap)
        out, kc, vc = run_append(case)
        check_pool(case, kc, vc, case.slot_mapping)
        assert_close(out, oracle_decode_after_store(case), f"cap={cap}")
    no_device_error()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 4), (32, 2)])
def test_append_geometries(cuda_device, d, hq, hkv):
    lens = [1, 31, 32, 33, 255, 256, 257, 511, 512, 513, 1000]
    case = W.make_decode_case("g", lens, hq, hkv, d, 40, seed=702 + hq + hkv + d)
    out, kc, vc = run_append(case)
    check_pool(case, kc, vc, case.slot_mapping)
    assert_close(out, oracle_decode_after_store(case), f"d={d} hq={hq} hkv={hkv}")
    no_device_error()


def test_append_skips_minus_one_and_rejects_other_slots(cuda_device):
    """Slot -1: nothing stored, the pool row is attended as it stands.  A slot
    that is not the new token's position: not stored, reported, and attended
    like -1."""
    case = W.make_decode_case("s", [40, 300, 700, 5], 16, 8, 128, 16, seed=703)
    sm = case.slot_mapping.clone()
    sm[1] = -1
    sm[2] = sm[2] + 1 if int(sm[2]) % 256 != 255 else sm[2] - 1  # another slot of its block
    out, kc, vc = run_append(case, sm)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    stored = sm.clone()
    stored[2] = -1
    check_pool(case, kc, vc, stored)
    case.slot_mapping = stored
    assert_close(out, oracle_decode_after_store(case), "after -1 and a rejected slot")


def test_append_graph_replays(cuda_device):
    case = W.qwen_decode(seed=1046, num_seqs=32)
    kc, vc, bt, cl = cache_to_device(case.cache)
    q, kn, vn, sm = dev(case.q), dev(case.k_new), dev(case.v_new), dev(case.slot_mapping)
    out = torch.empty_like(q)
    pkv.pkv_reserve_workspace(32, 16, 128, int(bt.shape[1]))
    pkv.pkv_decode_attention_append(q, kn, vn, sm, kc, vc, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkv.pkv_decode_attention_append(q, kn, vn, sm, kc, vc, bt, cl, case.scale, out)
    for seed in (1, 2):
        g = torch.Generator().manual_seed(seed)
        newk = W.randn_bf16(tuple(case.k_new.shape), g)
        newq = W.randn_bf16(tuple(case.q.shape), g)
        kn.copy_(dev(newk))
        q.copy_(dev(newq))
        graph.replay()
        torch.cuda.synchronize()
        case.k_new, case.q = newk, newq
        check_pool(case, kc, vc, case.slot_mapping)
        assert_close(out, oracle_decode_after_store(case), f"replay {seed}")
    no_device_error()
