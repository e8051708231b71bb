"""Chunked causal prefill (tcgen05) on the GPU against the fp64 oracle."""
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import (assert_close, cache_to_device, dev, no_device_error,
                     oracle_decode_after_store, oracle_prefill_after_store, run_prefill_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def default_knobs():
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    yield


@pytest.mark.parametrize("cached,chunk", [(0, 1), (0, 64), (0, 130), (5, 1), (255, 2), (256, 100),
                                          (300, 129), (1000, 300), (4096 - 256, 512)])
def test_prefill_shapes_full(cuda_device, cached, chunk):
    case = W.make_prefill_case("p", [cached, cached + 17], [chunk, chunk + 3], 16, 8, 128, 48,
                               seed=cached + chunk, skip_prob=0.05)
    out, _, _ = run_prefill_step(case)
    assert_close(out, oracle_prefill_after_store(case), f"cached={cached} chunk={chunk}")
    no_device_error()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2), (32, 2)])
def test_prefill_geometries(cuda_device, d, hq, hkv):
    case = W.make_prefill_case("g", [0, 300, 77], [200, 70, 1], hq, hkv, d, 24, seed=hq + hkv + d)
    out, _, _ = run_prefill_step(case)
    assert_close(out, oracle_prefill_after_store(case), f"d={d} hq={hq} hkv={hkv}")
    no_device_error()


def test_prefill_ragged_batch_with_empty_chunks(cuda_device):
    case = W.make_prefill_case("r", [10, 0, 700, 256, 3], [0, 33, 0, 257, 64], 16, 8, 128, 32,
                               seed=9)
    out, _, _ = run_prefill_step(case)
    assert_close(out, oracle_prefill_after_store(case), "ragged")
    no_device_error()


def test_chunked_prefill_8x512_sampled(cuda_device):
    """Full size (8 x 512 queries over 4608 keys, ~5% of slots -1); the oracle
    computes the first and last query of every chunk for all heads, plus a
    spread of rows across the chunks."""
    case = W.chunked_prefill()
    out, _, _ = run_prefill_step(case)
    rows = []
    for s in range(8):
        for i in (0, 511):
            rows += [(s * 512 + i, h) for h in range(16)]
        rows += [(s * 512 + (37 * k + 11 * s) % 512, (3 * k + s) % 16) for k in range(12)]
    ref = oracle_prefill_after_store(case, rows=rows)
    got = torch.stack([out[t, h] for t, h in rows])
    assert_close(got, ref, "chunked_prefill_8x512")
    no_device_error()


def test_prefill_of_one_query_matches_decode_oracle(cuda_device):
    case = W.make_decode_case("x", [1, 256, 257, 513, 2000], 16, 8, 128, 24, seed=31)
    c = case.cache
    kc, vc, bt, cl = cache_to_device(c)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    q = dev(case.q)
    out = torch.empty_like(q)
    cu = torch.arange(0, 6, dtype=torch.int32)
    pkv.pkv_prefill_attention(q, kc, vc, bt, dev(cu), cl, case.scale, out)
    torch.cuda.synchronize()
    assert_close(out, oracle_decode_after_store(case), "prefill Lq=1")


def test_dominant_key_selects_value_bit_exact(cuda_device):
    """Rows that can see a planted key with a logit gap > 127 (log2 units)
    return its V row exactly; rows before it stay within tolerance."""
    case = W.make_prefill_case("d", [300], [200], 16, 8, 128, 8, seed=4)
    c = case.cache
    q = torch.zeros_like(case.q)
    q[..., 0] = 16.0
    kc = c.k_cache.clone()
    kc[..., 0] = 0.0
    k_new = case.k_new.clone()
    k_new[..., 0] = 0.0
    t_star = 123                                       # a cached (not newly stored) position
    blk = int(c.block_tables[0, t_star // 256])
    kc[blk, t_star % 256, :, 0] = 64.0
    case.q, case.k_new = q, k_new
    case.cache.k_cache = kc
    out, kcd, vcd = run_prefill_step(case)
    vrow = vcd.cpu()[blk, t_star % 256]
    for i in range(200):                               # every query sits at position >= 300
        for h in range(16):
            assert torch.equal(out[i, h].cpu(), vrow[h // 2]), (i, h)
    no_device_error()


def test_prefill_block_relabelling_is_invisible(cuda_device):
    case = W.make_prefill_case("r", [700, 40], [300, 260], 16, 8, 128, 24, seed=12)
    out, kc, vc = run_prefill_step(case)
    c = case.cache
    perm = torch.randperm(c.num_blocks, generator=torch.Generator().manual_seed(3))
    nk, nv = torch.empty_like(kc), torch.empty_like(vc)
    nk[dev(perm)] = kc
    nv[dev(perm)] = vc
    nt = c.block_tables.clone()
    m = nt >= 0
    nt[m] = perm.to(torch.int32)[nt[m].long()]
    q = dev(case.q)
    o2 = torch.empty_like(q)
    pkv.pkv_prefill_attention(q, nk, nv, dev(nt), dev(case.cu_seqlens_q), dev(c.context_lens),
                              case.scale, o2)
    torch.cuda.synchronize()
    assert torch.equal(o2, out)


def test_prefill_negative_scale(cuda_device):
    """A negative softmax scale flips which raw score is the row maximum; the
    kernel then tracks the raw minimum.  Ragged chunks over cached prefixes."""
    case = W.make_prefill_case("neg", [0, 300, 77], [200, 70, 1], 16, 8, 128, 24, seed=91,
                               scale=-0.08)
    out, _, _ = run_prefill_step(case)
    assert_close(out, oracle_prefill_after_store(case), "negative scale")
    no_device_error()
