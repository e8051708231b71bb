"""Shared-prefix ("cascade") decode on the GPU against the fp64 oracle.

pkv_decode_attention_shared_prefix reads the blocks every sequence shares
once for the whole batch (a tcgen05 kernel over all sequences' queries),
streams each sequence's private tokens, and merges the two by log-sum-exp.
Paging is addressing only, so the oracle's output for the same inputs -- a
plain softmax over each sequence's gathered keys -- is the reference; the
oracle's own prefix-sharing invariance (shared blocks vs private copies) is
pinned in tests/test_oracle.py.
"""
import pytest
import torch

import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import (assert_close, cache_to_device, dev, no_device_error,
                     oracle_decode_after_store)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs(cuda_device):
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_shared_prefix_units(0)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_shared_prefix_units(0)
    pkv.pkv_get_device_error()


def run_cascade(case, shared_blocks, bt_override=None, cl_override=None):
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    if bt_override is not None:
        bt = dev(bt_override)
    if cl_override is not None:
        cl = dev(cl_override)
    q = dev(case.q)
    out = torch.full_like(q, float("nan"))
    pkv.pkv_decode_attention_shared_prefix(q, kc, vc, bt, cl, case.scale, shared_blocks, out)
    torch.cuda.synchronize()
    return out


def test_prefix_decode_b64_full(cuda_device):
    """The 64-sequence workload (8 shared blocks, private U[0,512] + 1)."""
    case = W.prefix_decode()
    out = run_cascade(case, 8)
    assert_close(out, oracle_decode_after_store(case), "prefix_decode_b64 cascade")
    no_device_error()


@pytest.mark.parametrize("units", [1, 2, 4, 8, 16])
def test_unit_count_does_not_change_result(cuda_device, units):
    case = W.make_decode_case("u", [1024 + 1, 1024 + 300, 1024 + 33, 1024 + 700], 16, 8, 128, 40,
                              seed=500 + units, shared_prefix_blocks=4, k_scale=3.0)
    pkv.pkv_set_shared_prefix_units(units)
    out = run_cascade(case, 4)
    assert_close(out, oracle_decode_after_store(case), f"units={units}")
    no_device_error()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2), (32, 2)])
def test_cascade_geometries(cuda_device, d, hq, hkv):
    lens = [512 + x for x in (1, 31, 32, 33, 255, 256, 257, 600, 1)]
    case = W.make_decode_case("g", lens, hq, hkv, d, 40, seed=600 + hq * 10 + hkv + d,
                              shared_prefix_blocks=2)
    out = run_cascade(case, 2)
    assert_close(out, oracle_decode_after_store(case), f"d={d} hq={hq} hkv={hkv}")
    no_device_error()


def test_more_rows_than_one_tile(cuda_device):
    """200 sequences x G = 2 = 400 query rows per KV head: four row tiles."""
    g = torch.Generator().manual_seed(7)
    lens = (256 * 3 + torch.randint(1, 300, (200,), generator=g)).tolist()
    case = W.make_decode_case("r", lens, 16, 8, 128, 1024, seed=601, shared_prefix_blocks=3)
    out = run_cascade(case, 3)
    assert_close(out, oracle_decode_after_store(case), "200 sequences")
    no_device_error()


def test_empty_private_parts_and_split_caps(cuda_device):
    """Contexts that end exactly at the shared prefix (no private token: the
    output comes from the shared partials alone), long private parts cut into
    pieces across blocks, and a cap on the split count."""
    lens = [768, 768 + 1, 768 + 9000, 768, 768 + 4000]
    case = W.make_decode_case("e", lens, 16, 8, 128, 80, seed=602, shared_prefix_blocks=3)
    # A context that ends at the prefix has its last token in a shared block:
    # no new row is stored for it (two such rows would hit the same slot).
    case.slot_mapping[torch.tensor(lens) == 768] = -1
    for cap in (0, 1, 3):
        pkv.pkv_set_max_splits(cap)
        out = run_cascade(case, 3)
        assert_close(out, oracle_decode_after_store(case), f"cap={cap}")
    no_device_error()


def test_zero_shared_blocks_is_plain_decode(cuda_device):
    case = W.make_decode_case("z", [1, 37, 256, 300], 16, 8, 128, 8, seed=603)
    out = run_cascade(case, 0)
    assert_close(out, oracle_decode_after_store(case), "shared_blocks=0")
    no_device_error()


def test_cascade_matches_plain_decode(cuda_device):
    """The same step with and without the cascade: both within the oracle's
    tolerance, and close to each other."""
    case = W.prefix_decode(seed=1044)
    casc = run_cascade(case, 8)
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    q = dev(case.q)
    plain = torch.empty_like(q)
    pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, plain)
    torch.cuda.synchronize()
    ref = oracle_decode_after_store(case)
    assert_close(casc, ref, "cascade")
    assert_close(plain, ref, "plain")
    assert (casc.float() - plain.float()).abs().max().item() <= 2e-2


def test_dominant_shared_key_is_exact(cuda_device):
    """A key in the shared prefix with a logit gap of ~64 nats over all others:
    every sequence's output is that key's V row, bit for bit (block
    addressing through the shared kernel and the merge)."""
    case = W.make_decode_case("d", [1024 + 5, 1024 + 77, 1024 + 300], 16, 8, 128, 16, seed=604,
                              shared_prefix_blocks=4)
    c = case.cache
    t = 600                                          # a shared position (block 2)
    blk = int(c.block_tables[0, t // 256])
    q = case.q.float()
    for s in range(3):
        for h in range(16):
            q[s, h] = 0.0
    q[:, :, 0] = 1.0
    case.q = q.to(torch.bfloat16)
    c.k_cache[blk, t % 256, :, 0] = 64.0 * (128 ** 0.5)
    out = run_cascade(case, 4)
    want = c.v_cache[blk, t % 256]                   # [Hkv, D]
    for s in range(3):
        for h in range(16):
            assert torch.equal(out[s, h].cpu(), want[h // 2]), (s, h)
    no_device_error()


@pytest.mark.parametrize("long_private", [20, 6000])
def test_mismatched_table_and_short_context_are_rejected(cuda_device, long_private):
    """A sequence that does not share the prefix blocks (its private part
    whole in one decode block, or cut into pieces across blocks) and one whose
    context is shorter than the prefix: zero outputs and PKV_ERR_DEVICE_CHECK;
    the others are right."""
    case = W.make_decode_case("m", [512 + 10, 512 + long_private, 512 + 30, 512 + 40], 16, 8,
                              128, 48, seed=605, shared_prefix_blocks=2)
    good = oracle_decode_after_store(case)
    bt = case.cache.block_tables.clone()
    bt[1, 1] = bt[1, 2]                              # sequence 1 does not share block 1
    cl = case.cache.context_lens.clone()
    cl[3] = 300                                      # shorter than the 512-token prefix
    out = run_cascade(case, 2, bt_override=bt, cl_override=cl)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[1] == 0) and torch.all(out[3] == 0)
    assert_close(out[[0, 2]], good[[0, 2]], "sharing sequences")


def test_graph_replays_follow_new_inputs(cuda_device):
    case = W.prefix_decode(seed=1045, num_seqs=16)
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_reserve_workspace(16, 16, 128, int(bt.shape[1]))
    pkv.pkv_decode_attention_shared_prefix(q, kc, vc, bt, cl, case.scale, 8, out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkv.pkv_decode_attention_shared_prefix(q, kc, vc, bt, cl, case.scale, 8, out)
    for seed in (1, 2):
        newq = W.randn_bf16(tuple(case.q.shape), torch.Generator().manual_seed(seed))
        q.copy_(dev(newq))
        graph.replay()
        torch.cuda.synchronize()
        case.q = newq
        assert_close(out, oracle_decode_after_store(case), f"replay {seed}")
    no_device_error()


@pytest.mark.parametrize("hq,hkv,seqs", [(32, 2, 700), (16, 2, 1400)])
def test_many_whole_pairs_per_block(cuda_device, hq, hkv, seqs):
    """Many short private parts: each decode block streams more whole pairs
    than it sets aside for the fold after its stream (64 / G of them), so the
    rest are folded as they come; both kinds match the oracle."""
    g = torch.Generator().manual_seed(hq + seqs)
    lens = (256 + torch.randint(1, 41, (seqs,), generator=g)).tolist()
    case = W.make_decode_case("w", lens, hq, hkv, 64, seqs + 20, seed=606 + hq,
                              shared_prefix_blocks=1)
    out = run_cascade(case, 1)
    assert_close(out, oracle_decode_after_store(case), f"hq={hq} hkv={hkv}")
    no_device_error()
