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


def test_chunked_prefill_8x512_full(cuda_device):
    """Full size (8 x 512 queries over 4608 keys, ~5% of slots -1): every
    (query, head) output against the oracle (run over the host cores)."""
    case = W.chunked_prefill()
    out, _, _ = run_prefill_step(case)
    assert_close(out, oracle_prefill_after_store(case), "chunked_prefill_8x512")
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


def _sample_rows(cu, num_heads, per_seq=24):
    rows = []
    for s in range(len(cu) - 1):
        c0, c1 = int(cu[s]), int(cu[s + 1])
        if c1 <= c0:
            continue
        picks = {c0, c1 - 1} | {c0 + (37 * k + 5 * s) % (c1 - c0) for k in range(per_seq)}
        rows += [(t, (t * 7 + s) % num_heads) for t in sorted(picks)]
        rows += [(c1 - 1, h) for h in range(num_heads)]
    return rows


def test_prefill_long_context_single_sequence(cuda_device):
    """One 256-token chunk over 8192 cached keys (about 5% of its rows not
    stored): few tiles, each with a long loop over 130 key tiles, and a
    softmax whose running max moves across many tiles."""
    case = W.make_prefill_case("long", [8192], [256], 16, 8, 128, 40, seed=21, skip_prob=0.05)
    out, _, _ = run_prefill_step(case)
    rows = _sample_rows(case.cu_seqlens_q, 16, per_seq=40)
    ref = oracle_prefill_after_store(case, rows=rows)
    assert_close(torch.stack([out[t, h] for t, h in rows]), ref, "long sequence")
    no_device_error()


def test_prefill_graph_replays_follow_new_inputs(cuda_device):
    """Store + prefill captured once in a CUDA graph (as an engine replays a
    captured step), replayed over three query batches written into the
    captured buffers: every replay must give that batch's attention."""
    case = W.make_prefill_case("pgraph", [3000, 100, 700], [300, 200, 64], 16, 8, 128, 64, seed=31)
    q, kc, vc, bt, cl = (dev(case.q), *cache_to_device(case.cache))
    kn, vn, sm, cu = dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), dev(case.cu_seqlens_q)
    out = torch.empty_like(q)
    pkv.pkv_reserve_workspace(case.num_seqs, 16, 128, bt.shape[1])

    def step():
        pkv.pkv_store_kvcache(kn, vn, sm, kc, vc)
        pkv.pkv_prefill_attention(q, kc, vc, bt, cu, cl, case.scale, out)

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
    gen = torch.Generator().manual_seed(78)
    rows = _sample_rows(case.cu_seqlens_q, 16)
    for i in range(3):
        q_host = torch.randn(case.q.shape, generator=gen).to(torch.bfloat16)
        q.copy_(q_host)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        replayed = W.PrefillCase(**{**case.__dict__, "q": q_host})
        ref = oracle_prefill_after_store(replayed, rows=rows)
        assert_close(torch.stack([out[t, h] for t, h in rows]), ref, f"replay {i}")
    no_device_error()


def test_prefill_batch_of_many_tiles(cuda_device):
    """16 chunks of 512 over 1024 cached keys: 1024 tiles (128-row tile x KV
    head), more than three waves of two blocks per SM."""
    case = W.make_prefill_case("waves", [1024] * 16, [512] * 16, 16, 8, 128, 112, seed=41,
                               skip_prob=0.05)
    out, _, _ = run_prefill_step(case)
    rows = _sample_rows(case.cu_seqlens_q, 16, per_seq=10)
    ref = oracle_prefill_after_store(case, rows=rows)
    assert_close(torch.stack([out[t, h] for t, h in rows]), ref, "waves then tail")
    no_device_error()
