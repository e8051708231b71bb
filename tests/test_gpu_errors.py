"""Device-side value checks and bounded waits.

Bad block ids, slots and lengths are never dereferenced: the kernels skip
them, write zeros for the affected output rows and record
PKV_ERR_DEVICE_CHECK.  A wait limit of 0 makes the first wait of every
block expire: the kernels record PKV_ERR_TIMEOUT, let their copies in flight
land, release tensor memory and return, and the next call on the same
context is correct again.
"""
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import (assert_close, cache_to_device, dev, oracle_decode_after_store,
                     oracle_prefill_after_store, run_decode_step, run_prefill_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_state(cuda_device):
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()


def test_bad_block_id_in_decode(cuda_device):
    case = W.make_decode_case("b", [300, 600, 40], 16, 8, 128, 16, seed=1)
    good = oracle_decode_after_store(case)
    case.cache.block_tables[1, 1] = 16          # == num_blocks: out of range
    out, _, _ = run_decode_step(case)
    code, site = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[1] == 0)
    assert_close(out[[0, 2]], good[[0, 2]], "unaffected sequences")


def test_bad_context_len_in_decode(cuda_device):
    case = W.make_decode_case("c", [300, 40], 16, 8, 128, 16, seed=2)
    kc, vc, bt, cl = cache_to_device(case.cache)
    cl[0] = 2 * 256 + 1                          # beyond the table width (2 blocks)
    q = dev(case.q)
    out = torch.full_like(q, 7.0)
    pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[0] == 0)


def test_bad_slot_in_store(cuda_device):
    case = W.tiny_decode()
    c = case.cache
    kc, vc = dev(c.k_cache), dev(c.v_cache)
    slots = case.slot_mapping.clone()
    slots[2] = 8 * 256                            # one past the pool
    slots[3] = -7
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(slots), kc, vc)
    code, site = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    keep = slots.clone()
    keep[2:] = -1
    rk, rv = oracle.store_kvcache(case.k_new, case.v_new, keep, c.k_cache, c.v_cache)
    assert torch.equal(kc.cpu().view(torch.int16), rk.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), rv.view(torch.int16))


def test_chunk_longer_than_context_in_prefill(cuda_device):
    case = W.make_prefill_case("l", [100, 0], [50, 40], 16, 8, 128, 16, seed=3)
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    cl[1] = 20                                    # Lq = 40 > C = 20
    q = dev(case.q)
    out = torch.full_like(q, 7.0)
    pkv.pkv_prefill_attention(q, kc, vc, bt, dev(case.cu_seqlens_q), cl, case.scale, out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[50:] == 0)
    ref = oracle_prefill_after_store(case, rows=[(t, h) for t in range(50) for h in range(16)])
    assert_close(out[:50].reshape(-1, 128), ref, "valid sequence")


def test_bad_block_id_in_prefill(cuda_device):
    case = W.make_prefill_case("k", [300], [100], 16, 8, 128, 8, seed=4)
    kc, vc, bt, cl = cache_to_device(case.cache)
    bt[0, 0] = -3
    q = dev(case.q)
    out = torch.full_like(q, 7.0)
    pkv.pkv_prefill_attention(q, kc, vc, bt, dev(case.cu_seqlens_q), cl, case.scale, out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out == 0)


def test_expired_waits_report_timeout_and_recover(cuda_device):
    dcase = W.make_decode_case("t", [3000, 5000], 16, 8, 128, 40, seed=5)
    pcase = W.make_prefill_case("t", [2000], [300], 16, 8, 128, 16, seed=6)
    pkv.pkv_set_wait_limit_ns(0)
    run_decode_step(dcase)
    code, site = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_TIMEOUT, (code, site)
    run_prefill_step(pcase)
    code, site = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_TIMEOUT, (code, site)
    # The context is still usable and results are right again.
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    out, _, _ = run_decode_step(dcase)
    assert_close(out, oracle_decode_after_store(dcase), "decode after timeouts")
    out, _, _ = run_prefill_step(pcase)
    assert_close(out, oracle_prefill_after_store(pcase), "prefill after timeouts")
    assert pkv.pkv_get_device_error()[0] == 0
